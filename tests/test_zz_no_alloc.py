"""The decode entry point for callers that cannot allocate device memory.

Callers such as allocator hooks, processes that reserve all device memory at
start-up, or plug-in hosts that forbid allocations while running cannot pass
``pkv_decode_attention`` a workspace. ``pkv_decode_attention_static_scratch``
serves them from a scratch array built into the library. Here it is called
through the C ABI twice in a row and must agree with the workspace entry
point on the same inputs, and with the oracle, within the attention
tolerance used throughout the tests; once its first call on the device has
run, further calls must leave the device's free memory unchanged. This file
is collected last so that a stop-at-first-failure run has already run every
other test.
"""

import gc

import pytest
import torch

from paged_kv_gqa_pkv_gb300 import binding
from paged_kv_gqa_pkv_gb300 import workloads as W
from tests.parity import (OUT_MAX_ABS, OUT_MEAN_ABS, LSE_ABS, assert_attention_close, gpu,
                          new_dev_err, oracle_decode_step)

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


def test_static_scratch_batches_above_512_rows_run_when_each_launch_fits():
    """Above 512 rows a call runs as equal launches, and the built-in scratch
    holds one launch's partials: 1030 rows (three launches of 344 on a 152-SM
    GB300) fit and give the workspace entry point's bits; 1100 rows (three of
    367) do not fit and are refused before any launch."""
    lens = torch.randint(1, 120, (1100,), generator=torch.Generator().manual_seed(21)).tolist()
    case = W.custom_decode(21, lens, hq=32, hkv=8, page_size=16, permute=True)
    x = _inputs(case)
    seen = set()
    for B in (1030, 1100):
        args = (x["k_pool"], x["v_pool"], x["page_table"], x["q"][:B].contiguous(),
                x["batch_idx"][:B].contiguous(), x["seq_lens"][:B].contiguous(),
                case.page_size, case.scale)
        need = binding.pkv_decode_workspace_size(x["k_pool"], x["page_table"], case.page_size,
                                                 B, case.num_q_heads)
        if need <= 8 << 20:
            ref_out, ref_lse = binding.pkv_decode_attention(*args)
            out, lse = binding.pkv_decode_attention_static_scratch(*args)
            torch.cuda.synchronize()
            assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)
            seen.add("fits")
        else:
            with pytest.raises(binding.PkvError) as e:
                binding.pkv_decode_attention_static_scratch(*args)
            assert e.value.status == 4
            seen.add("refused")
    if torch.cuda.get_device_properties(0).multi_processor_count == 152:
        assert seen == {"fits", "refused"}


def test_static_scratch_matches_oracle_and_allocates_nothing():
    case = W.tiny_decode(0)
    x = _inputs(case)
    # attend the pools as they stand (no append), against the oracle on the same pools
    _, _, ref_o, ref_l, _, bad_rows = oracle_decode_step(case, append=False)
    assert not bad_rows
    B, hq = case.q.shape[0], case.num_q_heads
    out = torch.empty((B, hq, 128), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, hq), dtype=torch.float32, device="cuda")
    err = new_dev_err()

    def call():
        binding.pkv_decode_attention_static_scratch(
            x["k_pool"], x["v_pool"], x["page_table"], x["q"], x["batch_idx"], x["seq_lens"],
            case.page_size, case.scale, out=out, lse=lse, dev_err=err)

    call()                      # the first call on a device may load the library's module
    torch.cuda.synchronize()
    gc.collect()                # earlier tests' garbage is not freed inside the window below
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    used0 = torch.cuda.memory_allocated()
    for _ in range(2):
        out.fill_(float("nan"))
        call()
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert_attention_close(out.cpu(), lse.cpu(), ref_o, ref_l, tag="static scratch")
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0 and torch.cuda.memory_allocated() == used0


def test_static_scratch_empty_batch_and_bad_arguments_match_workspace_entry_point():
    case = W.tiny_decode(0)
    x = _inputs(case)
    q0 = torch.zeros((0, case.num_q_heads, 128), dtype=torch.bfloat16, device="cuda")
    z0 = torch.zeros(0, dtype=torch.int32, device="cuda")
    out, lse = binding.pkv_decode_attention_static_scratch(
        x["k_pool"], x["v_pool"], x["page_table"], q0, z0, z0, case.page_size, case.scale)
    assert out.shape[0] == 0 and lse.shape[0] == 0
    # a GQA group the kernels do not serve (3 q heads per kv head): both entry points say ARG
    q3 = torch.zeros((2, 3 * case.num_kv_heads, 128), dtype=torch.bfloat16, device="cuda")
    z2 = torch.ones(2, dtype=torch.int32, device="cuda")
    for fn in (binding.pkv_decode_attention_static_scratch, binding.pkv_decode_attention):
        with pytest.raises(binding.PkvError) as e:
            kw = {} if fn is binding.pkv_decode_attention_static_scratch else {
                "workspace": torch.empty(1 << 20, dtype=torch.uint8, device="cuda")}
            fn(x["k_pool"], x["v_pool"], x["page_table"], q3, z2, z2, case.page_size,
               case.scale, **kw)
        assert e.value.status == 1
