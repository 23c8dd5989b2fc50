"""pkv_mixed_attention on the GPU: a step of prefill chunks and decode tokens
in one call, the decode tokens (runs of one) served by the split-KV decode
kernels and the rest by the chunked prefill. Every token is compared with the
oracle's paged_prefill_attention (the full-size step over all host cores);
edge cases cover every page size, lone tokens at the ends of the packing and
next to each other, runs of two (not routed), padding, more lone tokens than
the 512 the decode side takes, NaN in stale slots, and bad entries."""

import numpy as np
import pytest
import torch

import oracle.paged_attention as orc
from paged_kv_gqa_pkv_gb300 import binding
from paged_kv_gqa_pkv_gb300 import workloads as W
from paged_kv_gqa_pkv_gb300.workloads import bf16_bits
from tests import oracle_pool
from tests.parity import assert_attention_close, gpu, new_dev_err

pytestmark = pytest.mark.gpu


def run_mixed(c, table=None):
    kp, vp = gpu(c.k_pool), gpu(c.v_pool)
    pt = gpu(c.page_table if table is None else table)
    bidx, pos = gpu(c.batch_idx), gpu(c.input_pos)
    err = new_dev_err()
    binding.pkv_append(kp, vp, pt, gpu(c.k_new), gpu(c.v_new), bidx, pos, c.page_size,
                       dev_err=err)
    out, lse = binding.pkv_mixed_attention(kp, vp, pt, gpu(c.q), bidx, pos, c.page_size,
                                           c.scale, dev_err=err)
    torch.cuda.synchronize()
    return kp.cpu(), vp.cpu(), out.cpu(), lse.cpu(), int(err.item())


def oracle_mixed(c, rows=None, table=None):
    t = (c.page_table if table is None else table).numpy()
    kb, vb, bad_tok = orc.append(bf16_bits(c.k_pool), bf16_bits(c.v_pool), t, bf16_bits(c.k_new),
                                 bf16_bits(c.v_new), c.batch_idx.numpy(), c.input_pos.numpy(),
                                 c.page_size)
    out, lse, bad = orc.paged_prefill_attention(bf16_bits(c.q), kb, vb, t, c.batch_idx.numpy(),
                                                c.input_pos.numpy(), c.page_size, c.scale,
                                                rows=rows)
    return out, lse, bad_tok, bad


def test_full_size_mixed_step_every_row():
    """16 chunks of 512 over prefixes U[512, 4096] and 48 decode tokens over
    prefixes U[512, 2048], shuffled: every token of every head."""
    c = W.chunked_prefill(0)
    _, _, out, lse, err = run_mixed(c)
    t = c.page_table.numpy()
    kb, vb, bad_tok = orc.append(bf16_bits(c.k_pool), bf16_bits(c.v_pool), t, bf16_bits(c.k_new),
                                 bf16_bits(c.v_new), c.batch_idx.numpy(), c.input_pos.numpy(),
                                 c.page_size)
    assert err == 0 and not bad_tok
    ro_bits, rl, bad = oracle_pool.paged_prefill_all_rows(
        bf16_bits(c.q), kb, vb, t, c.batch_idx.numpy(), c.input_pos.numpy(), c.page_size,
        c.scale)
    assert not bad
    assert_attention_close(out, lse, orc.bf16_bits_to_f64(ro_bits), rl, tag="mixed full")


@pytest.mark.parametrize("ps", [16, 32, 64, 128, 256])
def test_every_page_size_lone_tokens_at_the_edges(ps):
    # slots in packed order (shuffle off): a lone token first and last, two
    # lone tokens side by side, a run of two (not routed), chunks between
    c = W.chunked_prefill(11, prefix_lens=[40, 0, 300, 129, 700, 16, 5, 250],
                          chunk_lens=[1, 90, 1, 1, 2, 140, 33, 1], page_size=ps, hq=16, hkv=4,
                          shuffle=False, n_pad=3)
    _, _, out, lse, err = run_mixed(c)
    ref_o, ref_l, bad_tok, bad = oracle_mixed(c)
    assert err == 0 and not bad_tok and not bad
    assert_attention_close(out, lse, ref_o, ref_l, tag=f"ps={ps}")
    assert torch.all(out[-3:] == 0) and torch.all(torch.isneginf(lse[-3:]))


def test_agrees_with_the_chunked_prefill_call():
    c = W.chunked_prefill(12, n_chunks=3, chunk=200, prefix_lo=10, prefix_hi=900, n_decode=20,
                          decode_lo=1, decode_hi=600, hq=32, hkv=8)
    _, _, out, lse, err = run_mixed(c)
    kp, vp = gpu(c.k_pool), gpu(c.v_pool)
    pt, bidx, pos = gpu(c.page_table), gpu(c.batch_idx), gpu(c.input_pos)
    binding.pkv_append(kp, vp, pt, gpu(c.k_new), gpu(c.v_new), bidx, pos, c.page_size)
    o2, l2 = binding.pkv_prefill_paged_attention(kp, vp, pt, gpu(c.q), bidx, pos, c.page_size,
                                                 c.scale)
    torch.cuda.synchronize()
    ref_o, ref_l, _, bad = oracle_mixed(c)
    assert err == 0 and not bad
    assert_attention_close(out, lse, ref_o, ref_l, tag="mixed")
    assert_attention_close(o2.cpu(), l2.cpu(), ref_o, ref_l, tag="chunked")


def test_more_lone_tokens_than_the_decode_side_takes():
    """600 decode tokens: the first 512 go to the decode kernels, the rest
    stay with the chunked prefill; every token is still exact."""
    c = W.chunked_prefill(13, n_chunks=2, chunk=130, prefix_lo=0, prefix_hi=300, n_decode=600,
                          decode_lo=1, decode_hi=200, hq=8, hkv=2, page_size=16)
    _, _, out, lse, err = run_mixed(c)
    ref_o, ref_l, bad_tok, bad = oracle_mixed(c)
    assert err == 0 and not bad_tok and not bad
    assert_attention_close(out, lse, ref_o, ref_l, tag="600 lone")


def test_stale_slots_hold_nan():
    c = W.chunked_prefill(14, n_chunks=3, chunk=100, prefix_lo=50, prefix_hi=500, n_decode=10,
                          decode_lo=1, decode_hi=400, hq=16, hkv=4, page_size=64,
                          fill=float("nan"))
    _, _, out, lse, err = run_mixed(c)
    ref_o, ref_l, bad_tok, bad = oracle_mixed(c)
    assert err == 0 and not bad_tok and not bad
    assert_attention_close(out, lse, ref_o, ref_l, tag="nan stale")


def test_bad_entries_flagged_on_both_paths():
    c = W.chunked_prefill(6, prefix_lens=[100, 300, 20, 60], chunk_lens=[30, 40, 50, 1],
                          page_size=32, hq=16, hkv=4, shuffle=False)
    table = c.page_table.clone()
    table[2, 3] = -1                 # slot 2 positions 96..127: inside its prefix
    b = c.batch_idx.clone()
    p = c.input_pos.clone()
    b[5] = 99                        # now a lone token (routed) with a slot past the table
    p[80] = 10 ** 6                  # a chunk token with a position past the table
    last = c.n_tokens - 1
    p[last] = -1                     # the lone decode token of slot 4 with a bad position
    c.batch_idx, c.input_pos = b, p
    kp, vp, out, lse, err = run_mixed(c, table=table)
    assert err & binding.DEV_ERR_BAD_PAGE and err & binding.DEV_ERR_BAD_SLOT
    assert err & binding.DEV_ERR_BAD_POS
    for r in (5, 80, last):
        assert torch.all(out[r] == 0) and torch.all(torch.isneginf(lse[r]))
    ok_rows = [i for i in range(c.n_tokens) if int(b[i]) in (1, 3) and i not in (5, 80)]
    ref_o, ref_l, _, bad = oracle_mixed(c, rows=ok_rows, table=table)
    assert not bad
    assert_attention_close(out, lse, ref_o, ref_l, rows=ok_rows)


def test_workspace_checked_and_reused_across_calls():
    c = W.chunked_prefill(15, n_chunks=2, chunk=64, prefix_lo=1, prefix_hi=200, n_decode=5,
                          decode_lo=1, decode_hi=300, hq=8, hkv=2, page_size=16)
    kp, vp = gpu(c.k_pool), gpu(c.v_pool)
    pt, bidx, pos = gpu(c.page_table), gpu(c.batch_idx), gpu(c.input_pos)
    binding.pkv_append(kp, vp, pt, gpu(c.k_new), gpu(c.v_new), bidx, pos, c.page_size)
    n = binding.pkv_mixed_workspace_size(kp, pt, c.page_size, c.n_tokens, c.num_q_heads)
    with pytest.raises(binding.PkvError) as e:
        binding.pkv_mixed_attention(kp, vp, pt, gpu(c.q), bidx, pos, c.page_size, c.scale,
                                    workspace=torch.empty(n - 256, dtype=torch.uint8,
                                                          device="cuda"))
    assert e.value.status == 4
    ws = torch.full((n,), 0xAB, dtype=torch.uint8, device="cuda")   # stale contents
    o1, l1 = binding.pkv_mixed_attention(kp, vp, pt, gpu(c.q), bidx, pos, c.page_size, c.scale,
                                         workspace=ws)
    o2, l2 = binding.pkv_mixed_attention(kp, vp, pt, gpu(c.q), bidx, pos, c.page_size, c.scale,
                                         workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    ref_o, ref_l, _, bad = oracle_mixed(c)
    assert not bad
    assert_attention_close(o1.cpu(), l1.cpu(), ref_o, ref_l)


def test_more_than_768_query_tiles_round_robin():
    """200 chunks of 512 tokens and 30 decode tokens: 800 listed query tiles,
    past the sorted schedule's limit, so the prefill kernel deals them
    round-robin; sampled tokens (every decode token, the ends of every chunk
    and 400 others) against the oracle."""
    c = W.chunked_prefill(14, n_chunks=200, chunk=512, prefix_lo=0, prefix_hi=256, n_decode=30,
                          decode_lo=1, decode_hi=600, hq=8, hkv=2)
    _, _, out, lse, err = run_mixed(c)
    assert err == 0
    b = c.batch_idx.numpy()
    edges = np.flatnonzero(np.diff(b))
    rows = {0, len(b) - 1}
    rows.update(edges.tolist())
    rows.update((edges + 1).tolist())
    rows.update(np.random.default_rng(14).choice(len(b), 400, replace=False).tolist())
    rows = sorted(rows)
    ro, rl, bad_tok, bad = oracle_mixed(c, rows=rows)
    assert not bad_tok and not bad
    assert_attention_close(out, lse, ro, rl, rows=rows, tag="mixed 800 tiles")
