"""pkv_stage_from_host on the GPU: pinned host bytes copied into device
memory bit for bit at several sizes, memory the GPU cannot reach rejected
before any launch, and a decode step whose inputs are staged this way (in a
captured graph, as a serving loop replays it) giving the same bits as one
whose inputs were copied by the copy engine."""

import pytest
import torch

from paged_kv_gqa_pkv_gb300 import binding
from paged_kv_gqa_pkv_gb300 import workloads as W
from tests.parity import gpu, new_dev_err

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("nbytes", [16, 4112, 789248, 3 << 20])
def test_pinned_bytes_arrive_exactly(nbytes):
    gen = torch.Generator().manual_seed(nbytes)
    src = torch.randint(0, 256, (nbytes,), dtype=torch.uint8, generator=gen).pin_memory()
    dst = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    binding.pkv_stage_from_host(dst, src)
    torch.cuda.synchronize()
    assert torch.equal(dst.cpu(), src)


def test_unreachable_or_misaligned_memory_is_rejected():
    pageable = torch.ones(4096, dtype=torch.uint8)          # not pinned
    dst = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    with pytest.raises(binding.PkvError) as e:
        binding.pkv_stage_from_host(dst, pageable)
    assert e.value.status == 1
    pinned = torch.ones(4096 + 16, dtype=torch.uint8).pin_memory()
    with pytest.raises(binding.PkvError) as e:
        binding.pkv_stage_from_host(dst[8:8 + 4096 - 16], pinned[:4096 - 16])
    assert e.value.status == 2
    with pytest.raises(binding.PkvError) as e:
        binding.pkv_stage_from_host(dst[:24], pinned[:24])
    assert e.value.status == 1
    torch.cuda.synchronize()
    assert torch.all(dst == 0)


def test_staged_decode_step_in_a_graph_matches_copied_inputs():
    c = W.qwen3_b64_decode(3, permute=True)
    ins = [c.q, c.k_new, c.v_new, c.batch_idx, c.seq_lens, c.page_table]
    offs, n = [], 0
    for t in ins:
        offs.append(n)
        n += (t.numel() * t.element_size() + 255) // 256 * 256
    host = torch.zeros(n, dtype=torch.uint8).pin_memory()
    dev = torch.zeros(n, dtype=torch.uint8, device="cuda")
    hv, dv = [], []
    for t, o in zip(ins, offs):
        nb = t.numel() * t.element_size()
        hv.append(host[o:o + nb].view(t.dtype).view(t.shape))
        dv.append(dev[o:o + nb].view(t.dtype).view(t.shape))
    for h, t in zip(hv, ins):
        h.copy_(t)
    q, kn, vn, bi, sl, pt = dv
    ref_k, ref_v = gpu(c.k_pool), gpu(c.v_pool)
    ref_o, ref_l = binding.pkv_decode_append_attention(
        ref_k, ref_v, gpu(c.page_table), gpu(c.q), gpu(c.k_new), gpu(c.v_new),
        gpu(c.batch_idx), gpu(c.seq_lens), c.page_size, c.scale)
    kp, vp = gpu(c.k_pool), gpu(c.v_pool)
    out = torch.empty_like(ref_o)
    lse = torch.empty_like(ref_l)
    ws = torch.empty(binding.pkv_decode_workspace_size(kp, pt, c.page_size, c.batch,
                                                       c.num_q_heads), dtype=torch.uint8,
                     device="cuda")
    err = new_dev_err()

    def step():
        binding.pkv_stage_from_host(dev, host)
        binding.pkv_decode_append_attention(kp, vp, pt, q, kn, vn, bi, sl, c.page_size,
                                            c.scale, out=out, lse=lse, workspace=ws,
                                            dev_err=err)

    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        step()
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            step()
    for _ in range(2):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert torch.equal(out, ref_o) and torch.equal(lse, ref_l)
        assert torch.equal(kp, ref_k) and torch.equal(vp, ref_v)
