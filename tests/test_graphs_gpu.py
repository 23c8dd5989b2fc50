"""Bucketed CUDA-graph decode: replaying the captured append + decode for a
bucket gives bit-identical pools and outputs to eager calls, for batch sizes
that need padding rows, and stays within tolerance of the oracle."""

import numpy as np
import pytest
import torch

from paged_kv_gqa_pkv_gb300 import binding
from paged_kv_gqa_pkv_gb300 import workloads as W
from paged_kv_gqa_pkv_gb300.graphs import DecodeGraphs
from paged_kv_gqa_pkv_gb300.workloads import bf16_bits
from tests.parity import assert_attention_close, gpu, oracle_decode_step

pytestmark = pytest.mark.gpu


def _rows(case, B):
    return (gpu(case.q[:B]), gpu(case.k_new[:B]), gpu(case.v_new[:B]),
            gpu(case.batch_idx[:B]), gpu(case.input_pos[:B]), gpu(case.seq_lens[:B]))


@pytest.mark.parametrize("fused", [True, False], ids=["fused", "two_calls"])
@pytest.mark.parametrize("B", [1, 3, 17, 64])
def test_graph_replay_matches_eager(B, fused):
    case = W.qwen3_b64_decode(0, permute=True)
    kp_g, vp_g, pt = gpu(case.k_pool), gpu(case.v_pool), gpu(case.page_table)
    graphs = DecodeGraphs(kp_g, vp_g, pt, case.page_size, case.num_q_heads, case.scale,
                          buckets=(1, 2, 4, 8, 16, 32, 64), fused=fused)
    q, kn, vn, bi, ip, sl = _rows(case, B)
    out_g, lse_g = graphs.step(q, kn, vn, bi, ip, sl)
    torch.cuda.synchronize()
    assert int(graphs.dev_err.item()) == 0

    kp_e, vp_e = gpu(case.k_pool), gpu(case.v_pool)
    binding.pkv_append(kp_e, vp_e, pt, kn, vn, bi, ip, case.page_size)
    out_e, lse_e = binding.pkv_decode_attention(kp_e, vp_e, pt, q, bi, sl, case.page_size,
                                                case.scale)
    torch.cuda.synchronize()
    assert torch.equal(kp_g, kp_e) and torch.equal(vp_g, vp_e)
    assert torch.equal(out_g, out_e) and torch.equal(lse_g, lse_e)


@pytest.mark.parametrize("fused", [True, False], ids=["fused", "two_calls"])
def test_graph_steps_follow_the_cache_and_match_the_oracle(fused):
    """Two steps through one captured graph: the second sees the first step's
    appended tokens (the pools are updated in place, by pointer)."""
    case = W.custom_decode(4, [40, 130, 7, 300, 77], hq=32, hkv=8, page_size=128,
                           permute=True, max_blocks=4)
    kp, vp, pt = gpu(case.k_pool), gpu(case.v_pool), gpu(case.page_table)
    graphs = DecodeGraphs(kp, vp, pt, case.page_size, case.num_q_heads, case.scale,
                          buckets=(4, 8), fused=fused)
    q, kn, vn, bi, ip, sl = _rows(case, case.batch)
    graphs.step(q, kn, vn, bi, ip, sl)
    # step 2: one more token per row
    gen = torch.Generator().manual_seed(11)
    case2 = case
    case2.k_pool, case2.v_pool = kp.cpu(), vp.cpu()
    case2.q = torch.randn(case.q.shape, generator=gen).to(torch.bfloat16)
    case2.k_new = torch.randn(case.k_new.shape, generator=gen).to(torch.bfloat16)
    case2.v_new = torch.randn(case.v_new.shape, generator=gen).to(torch.bfloat16)
    case2.input_pos = case.input_pos + 1
    case2.seq_lens = case.seq_lens + 1
    out, lse = graphs.step(*_rows(case2, case2.batch))
    torch.cuda.synchronize()
    assert int(graphs.dev_err.item()) == 0
    ek, ev, ref_o, ref_l, bad_tok, bad_rows = oracle_decode_step(case2)
    assert not bad_tok and not bad_rows
    assert np.array_equal(bf16_bits(kp.cpu()), ek) and np.array_equal(bf16_bits(vp.cpu()), ev)
    assert_attention_close(out.cpu(), lse.cpu(), ref_o, ref_l, tag="graph step 2")


def test_bucket_selection():
    case = W.tiny_decode(0)
    graphs = DecodeGraphs(gpu(case.k_pool), gpu(case.v_pool), gpu(case.page_table),
                          case.page_size, case.num_q_heads, case.scale, buckets=(2, 8, 4))
    assert graphs.buckets == (2, 4, 8)
    assert [graphs.bucket_for(b) for b in (1, 2, 3, 5, 8)] == [2, 2, 4, 8, 8]
    with pytest.raises(ValueError):
        graphs.bucket_for(9)
