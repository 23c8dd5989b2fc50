"""Fused append + decode (``pkv_decode_append_attention``) on the GPU: the
pools bit-exact against the oracle's append, the attention against the
oracle's decode over the appended cache, and bit-identical to the two-call
path (``pkv_append`` then ``pkv_decode_attention``)."""

import numpy as np
import pytest
import torch

import oracle.paged_attention as orc
from paged_kv_gqa_pkv_gb300 import binding
from paged_kv_gqa_pkv_gb300 import workloads as W
from paged_kv_gqa_pkv_gb300.workloads import bf16_bits
from tests.parity import (assert_attention_close, gpu, new_dev_err, oracle_decode_step,
                          run_decode_step)

pytestmark = pytest.mark.gpu


def run_fused(case, dev_err=None):
    kp, vp = gpu(case.k_pool), gpu(case.v_pool)
    err = new_dev_err() if dev_err is None else dev_err
    out, lse = binding.pkv_decode_append_attention(
        kp, vp, gpu(case.page_table), gpu(case.q), gpu(case.k_new), gpu(case.v_new),
        gpu(case.batch_idx), gpu(case.seq_lens), case.page_size, case.scale, dev_err=err)
    torch.cuda.synchronize()
    return kp.cpu(), vp.cpu(), out.cpu(), lse.cpu(), int(err.item())


def _live_rows_decode_convention(case):
    live = case.batch_idx.numpy() != 0
    assert np.array_equal(case.input_pos.numpy()[live] + 1, case.seq_lens.numpy()[live])


@pytest.mark.parametrize("maker", [W.tiny_decode, lambda s: W.qwen3_b64_decode(s, permute=False),
                                   lambda s: W.qwen3_b64_decode(s, permute=True),
                                   W.padded_bucket_decode, W.long_context_decode],
                         ids=["tiny", "qwen3_b64_seq", "qwen3_b64_perm", "padded_bucket",
                              "long_context_b256"])
def test_fused_matches_oracle(maker):
    c = maker(0)
    _live_rows_decode_convention(c)
    kp, vp, out, lse, err = run_fused(c)
    ek, ev, ref_o, ref_l, bad_tok, bad_rows = oracle_decode_step(c)
    assert err == 0 and not bad_tok and not bad_rows
    assert np.array_equal(bf16_bits(kp), ek) and np.array_equal(bf16_bits(vp), ev)
    assert_attention_close(out, lse, ref_o, ref_l, tag=c.name)


@pytest.mark.parametrize("maker", [lambda s: W.qwen3_b64_decode(s, permute=True),
                                   W.padded_bucket_decode])
def test_fused_is_bit_identical_to_two_calls(maker):
    c = maker(1)
    k1, v1, o1, l1, e1 = run_fused(c)
    k2, v2, o2, l2, e2 = run_decode_step(c)
    assert e1 == 0 and e2 == 0
    assert torch.equal(k1, k2) and torch.equal(v1, v2)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_new_token_slot_holding_nan_is_overwritten_before_it_is_read():
    """The new token's slot holds NaN before the call: the tile that holds it
    must be read after the fused write lands, or NaN reaches the result."""
    lens = [1, 16, 17, 33, 128, 129, 700, 2048]
    c = W.custom_decode(31, lens, hq=32, hkv=8, page_size=16, permute=True)
    c.input_pos = c.seq_lens - 1
    for b in range(len(lens)):
        slot, pos = int(c.batch_idx[b]), int(c.input_pos[b])
        row = int(c.page_table[slot, pos // 16]) * 16 + pos % 16
        c.k_pool[row] = float("nan")
        c.v_pool[row] = float("nan")
    kp, vp, out, lse, err = run_fused(c)
    assert err == 0
    ek, ev, ref_o, ref_l, _, _ = oracle_decode_step(c)
    assert np.array_equal(bf16_bits(kp), ek) and np.array_equal(bf16_bits(vp), ev)
    assert_attention_close(out, lse, ref_o, ref_l)


@pytest.mark.parametrize("hq,hkv", [(8, 8), (16, 8), (32, 4), (8, 2)])
def test_fused_other_gqa_groups(hq, hkv):
    lens = [1, 15, 16, 17, 31, 32, 33, 100, 257, 1000]
    c = W.custom_decode(33, lens, hq=hq, hkv=hkv, page_size=32, permute=True)
    c.input_pos = c.seq_lens - 1
    kp, vp, out, lse, err = run_fused(c)
    ek, ev, ref_o, ref_l, bad_tok, bad_rows = oracle_decode_step(c)
    assert err == 0 and not bad_tok and not bad_rows
    assert np.array_equal(bf16_bits(kp), ek) and np.array_equal(bf16_bits(vp), ev)
    assert_attention_close(out, lse, ref_o, ref_l, tag=f"G={hq // hkv}")


def test_bad_page_for_new_token_is_flagged_other_rows_exact():
    c = W.custom_decode(35, [40, 300, 90], hq=32, hkv=8, page_size=128, permute=True)
    c.input_pos = c.seq_lens - 1
    slot = int(c.batch_idx[1])
    c.page_table[slot, 299 // 128] = -1      # the page that would take row 1's new token
    kp, vp, out, lse, err = run_fused(c)
    assert err & binding.DEV_ERR_BAD_PAGE
    ek, ev, ref_o, ref_l, bad_tok, bad_rows = oracle_decode_step(c)
    assert bad_tok == [1] and bad_rows == [1]
    assert np.array_equal(bf16_bits(kp), ek) and np.array_equal(bf16_bits(vp), ev)
    assert_attention_close(out, lse, ref_o, ref_l, rows=[0, 2])


@pytest.mark.parametrize("ps", [48, 256])
def test_fused_other_page_sizes(ps):
    """The new token's slot through the page table for page sizes that are
    not 128: pools bit-exact, attention against the oracle, and the same bits
    as the two-call step."""
    lens = [1, 16, ps, ps + 1, 2 * ps - 1, 500]
    c = W.custom_decode(33, lens, hq=32, hkv=8, page_size=ps, permute=True)
    kp, vp, out, lse, err = run_fused(c)
    ek, ev, ref_o, ref_l, bad_tok, bad_rows = oracle_decode_step(c)
    assert err == 0 and not bad_tok and not bad_rows
    assert np.array_equal(bf16_bits(kp), ek) and np.array_equal(bf16_bits(vp), ev)
    assert_attention_close(out, lse, ref_o, ref_l, tag=f"fused ps={ps}")
    k2, v2, o2, l2, e2 = run_decode_step(c)
    assert e2 == 0
    assert torch.equal(kp, k2) and torch.equal(vp, v2)
    assert torch.equal(out, o2) and torch.equal(lse, l2)


def test_results_written_straight_into_pinned_host_memory():
    """out and lse may be pinned host memory (the kernels write them with
    plain stores): the same bits as device buffers, with no copy."""
    c = W.qwen3_b64_decode(2, permute=True)
    k1, v1, o1, l1, e1 = run_fused(c)
    kp, vp = gpu(c.k_pool), gpu(c.v_pool)
    out_h = torch.zeros((c.batch, c.num_q_heads, c.head_dim), dtype=torch.bfloat16).pin_memory()
    lse_h = torch.zeros((c.batch, c.num_q_heads), dtype=torch.float32).pin_memory()
    err = new_dev_err()
    binding.pkv_decode_append_attention(kp, vp, gpu(c.page_table), gpu(c.q), gpu(c.k_new),
                                        gpu(c.v_new), gpu(c.batch_idx), gpu(c.seq_lens),
                                        c.page_size, c.scale, out=out_h, lse=lse_h, dev_err=err)
    torch.cuda.synchronize()
    assert e1 == 0 and int(err.item()) == 0
    assert torch.equal(out_h, o1) and torch.equal(lse_h, l1)


def test_fused_batches_above_512_rows():
    """777 rows run as two launches of at most 389 rows: each appends and
    attends its own rows. Pools and outputs equal the two-call step's bits
    and the oracle's."""
    lens = torch.randint(1, 150, (777,), generator=torch.Generator().manual_seed(12)).tolist()
    c = W.custom_decode(12, lens, hq=32, hkv=8, page_size=16, permute=True)
    _live_rows_decode_convention(c)
    k1, v1, o1, l1, e1 = run_fused(c)
    k2, v2, o2, l2, e2 = run_decode_step(c)
    assert e1 == 0 and e2 == 0
    assert torch.equal(k1, k2) and torch.equal(v1, v2)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    ek, ev, ref_o, ref_l, bad_tok, bad_rows = oracle_decode_step(c)
    assert not bad_tok and not bad_rows
    assert np.array_equal(bf16_bits(k1), ek) and np.array_equal(bf16_bits(v1), ev)
    assert_attention_close(o1, l1, ref_o, ref_l, tag="fused 777 rows")
