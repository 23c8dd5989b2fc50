"""The decode entry point for callers that cannot allocate device memory.

Callers such as allocator hooks, processes that reserve all device memory at
start-up, or plug-in hosts that forbid allocations while running cannot pass
``pkv_decode_attention`` a workspace. ``pkv_decode_attention_static_scratch``
serves them from a scratch array built into the library. Here it is called
through the C ABI twice in a row and must agree with the workspace entry
point on the same inputs, within the attention tolerance used throughout the
tests. This file is collected last so that a stop-at-first-failure run has
already run every other test.
"""

import pytest
import torch

from paged_kv_gqa_pkv_gb300 import binding
from paged_kv_gqa_pkv_gb300 import workloads as W
from tests.parity import OUT_MAX_ABS, OUT_MEAN_ABS, LSE_ABS, gpu, new_dev_err

pytestmark = pytest.mark.gpu


def _inputs(case):
    return dict(k_pool=gpu(case.k_pool), v_pool=gpu(case.v_pool),
                page_table=gpu(case.page_table), q=gpu(case.q),
                batch_idx=gpu(case.batch_idx), seq_lens=gpu(case.seq_lens))


def _close(a_out, a_lse, b_out, b_lse):
    d = (a_out.float() - b_out.float()).abs()
    assert d.max().item() <= OUT_MAX_ABS and d.mean().item() <= OUT_MEAN_ABS
    fin = torch.isfinite(b_lse)
    assert torch.equal(torch.isneginf(a_lse), torch.isneginf(b_lse))
    if fin.any():
        assert (a_lse[fin] - b_lse[fin]).abs().max().item() <= LSE_ABS


@pytest.mark.parametrize("maker", [W.qwen3_b64_decode, W.padded_bucket_decode])
def test_static_scratch_matches_workspace_entry_point_twice(maker):
    case = maker(0)
    x = _inputs(case)
    ref_out, ref_lse = binding.pkv_decode_attention(
        x["k_pool"], x["v_pool"], x["page_table"], x["q"], x["batch_idx"], x["seq_lens"],
        case.page_size, case.scale)
    for _ in range(2):
        err = new_dev_err()
        out, lse = binding.pkv_decode_attention_static_scratch(
            x["k_pool"], x["v_pool"], x["page_table"], x["q"], x["batch_idx"], x["seq_lens"],
            case.page_size, case.scale, dev_err=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        _close(out.cpu(), lse.cpu(), ref_out.cpu(), ref_lse.cpu())


def test_static_scratch_rejects_batches_past_its_limit():
    case = W.qwen3_b64_decode(0)
    x = _inputs(case)
    B = 500    # 8 KV heads x 500 rows needs about 11 MB, past the built-in 8 MiB
    q = torch.zeros((B, case.num_q_heads, 128), dtype=torch.bfloat16, device="cuda")
    z = torch.zeros(B, dtype=torch.int32, device="cuda")
    with pytest.raises(binding.PkvError) as e:
        binding.pkv_decode_attention_static_scratch(
            x["k_pool"], x["v_pool"], x["page_table"], q, z, z, case.page_size, case.scale)
    assert e.value.status == 4
