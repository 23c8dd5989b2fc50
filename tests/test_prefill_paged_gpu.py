"""Chunked prefill over the paged cache (``pkv_prefill_paged_attention``) on
the GPU against the oracle's ``paged_prefill_attention``: the chunks' K/V are
appended first (``pkv_append``), then every packed token attends its slot's
keys 0..input_pos through the pages. Every token is compared: the full-size
step runs the oracle over all host cores."""

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


def run_chunked(c, table=None):
    """Append the chunk K/V, then paged prefill, on the GPU. Returns CPU
    (k_pool, v_pool, out, lse, dev_err)."""
    kp, vp = gpu(c.k_pool), gpu(c.v_pool)
    pt = gpu(c.page_table if table is None else table)
    bidx, pos = gpu(c.batch_idx), gpu(c.input_pos)
    err = new_dev_err()
    binding.pkv_append(kp, vp, pt, gpu(c.k_new), gpu(c.v_new), bidx, pos, c.page_size,
                       dev_err=err)
    out, lse = binding.pkv_prefill_paged_attention(kp, vp, pt, gpu(c.q), bidx, pos, c.page_size,
                                                   c.scale, dev_err=err)
    torch.cuda.synchronize()
    return kp.cpu(), vp.cpu(), out.cpu(), lse.cpu(), int(err.item())


def oracle_chunked(c, rows=None, table=None):
    t = (c.page_table if table is None else table).numpy()
    kb, vb, bad_tok = orc.append(bf16_bits(c.k_pool), bf16_bits(c.v_pool), t, bf16_bits(c.k_new),
                                 bf16_bits(c.v_new), c.batch_idx.numpy(), c.input_pos.numpy(),
                                 c.page_size)
    out, lse, bad = orc.paged_prefill_attention(bf16_bits(c.q), kb, vb, t, c.batch_idx.numpy(),
                                                c.input_pos.numpy(), c.page_size, c.scale,
                                                rows=rows)
    return out, lse, bad_tok, bad


def test_mixed_chunked_step_full_size_every_row():
    """16 chunks of 512 tokens over prefixes U[512, 4096] plus 48 decode
    tokens, shuffled (the default chunked workload, page 128): every token of
    every head against the oracle, run over all host cores."""
    c = W.chunked_prefill(0)
    kp, vp, out, lse, err = run_chunked(c)
    t = c.page_table.numpy()
    kb, vb, bad_tok = orc.append(bf16_bits(c.k_pool), bf16_bits(c.v_pool), t, bf16_bits(c.k_new),
                                 bf16_bits(c.v_new), c.batch_idx.numpy(), c.input_pos.numpy(),
                                 c.page_size)
    assert err == 0 and not bad_tok
    assert np.array_equal(bf16_bits(kp), kb) and np.array_equal(bf16_bits(vp), vb)
    ro_bits, rl, bad = oracle_pool.paged_prefill_all_rows(
        bf16_bits(c.q), kb, vb, t, c.batch_idx.numpy(), c.input_pos.numpy(), c.page_size,
        c.scale)
    assert not bad and not np.isnan(rl).any()
    assert_attention_close(out, lse, orc.bf16_bits_to_f64(ro_bits), rl, tag="chunked full")


@pytest.mark.parametrize("ps", [16, 32, 64, 128, 256])
def test_every_page_size(ps):
    c = W.chunked_prefill(1, prefix_lens=[0, 5, 300, 129, 700, 16], chunk_lens=[20, 1, 140, 1, 77, 33],
                          page_size=ps, hq=16, hkv=4, n_pad=5)
    _, _, out, lse, err = run_chunked(c)
    ref_o, ref_l, bad_tok, bad = oracle_chunked(c)
    assert err == 0 and not bad_tok and not bad
    assert_attention_close(out, lse, ref_o, ref_l, tag=f"ps={ps}")


@pytest.mark.parametrize("hq,hkv", [(8, 8), (16, 8), (32, 8), (16, 2)])
def test_gqa_groups(hq, hkv):
    c = W.chunked_prefill(2, prefix_lens=[40, 0, 260, 1], chunk_lens=[90, 130, 3, 200], hq=hq,
                          hkv=hkv, page_size=128)
    _, _, out, lse, err = run_chunked(c)
    ref_o, ref_l, bad_tok, bad = oracle_chunked(c)
    assert err == 0 and not bad_tok and not bad
    assert_attention_close(out, lse, ref_o, ref_l, tag=f"G={hq // hkv}")


def test_stale_slots_hold_nan():
    """Every pool row past the prefixes starts as NaN: the chunks' own rows are
    written by the append, the rest (tails of the last pages) must never reach
    a result."""
    c = W.chunked_prefill(3, prefix_lens=[37, 200, 0], chunk_lens=[50, 1, 100], page_size=64,
                          hq=32, hkv=8, fill=float("nan"))
    _, _, out, lse, err = run_chunked(c)
    ref_o, ref_l, bad_tok, bad = oracle_chunked(c)
    assert err == 0 and not bad_tok and not bad
    assert_attention_close(out, lse, ref_o, ref_l)


def test_many_runs_in_one_tile_and_a_split_run():
    """40 decode tokens of different slots and two chunks in the first tiles;
    one slot's chunk split in two parts around other slots' tokens."""
    pre = [int(x) for x in np.random.default_rng(4).integers(1, 600, 40)] + [100, 0]
    chunks = [1] * 40 + [70, 60]
    c = W.chunked_prefill(4, prefix_lens=pre, chunk_lens=chunks, page_size=16, hq=16, hkv=8,
                          shuffle=True)
    # move the last 25 tokens of slot 41's chunk after the next few tokens
    b = c.batch_idx.numpy()
    idx = np.nonzero(b == 41)[0]
    order = list(range(len(b)))
    tail = order[idx[-25]:idx[-1] + 1]
    rest = [i for i in order if i not in tail]
    cut = rest.index(idx[-26]) + 4
    order = rest[:cut] + tail + rest[cut:]
    for name in ("q", "k_new", "v_new", "batch_idx", "input_pos"):
        setattr(c, name, getattr(c, name)[order].contiguous())
    _, _, out, lse, err = run_chunked(c)
    ref_o, ref_l, bad_tok, bad = oracle_chunked(c)
    assert err == 0 and not bad_tok and not bad
    assert_attention_close(out, lse, ref_o, ref_l)


def test_one_token_per_slot_agrees_with_decode():
    c = W.custom_decode(5, [33, 1, 400, 129, 1000, 17], hq=32, hkv=8, page_size=128, permute=True)
    kp, vp, pt = gpu(c.k_pool), gpu(c.v_pool), gpu(c.page_table)
    bidx, pos = gpu(c.batch_idx), gpu(c.input_pos)
    binding.pkv_append(kp, vp, pt, gpu(c.k_new), gpu(c.v_new), bidx, pos, 128)
    o1, l1 = binding.pkv_prefill_paged_attention(kp, vp, pt, gpu(c.q), bidx, pos, 128, c.scale)
    o2, l2 = binding.pkv_decode_attention(kp, vp, pt, gpu(c.q), bidx, gpu(c.seq_lens), 128,
                                          c.scale)
    torch.cuda.synchronize()
    assert (o1.float() - o2.float()).abs().max().item() <= 2e-2
    assert (l1 - l2).abs().max().item() <= 1e-3


def test_bad_entries_flagged_other_tokens_exact():
    c = W.chunked_prefill(6, prefix_lens=[100, 300, 20], chunk_lens=[30, 40, 50], page_size=32,
                          hq=16, hkv=4, shuffle=False)
    table = c.page_table.clone()
    table[2, 3] = -1                 # slot 2 positions 96..127: inside its prefix
    b = c.batch_idx.clone()
    p = c.input_pos.clone()
    b[5] = 99                        # slot past the table
    p[80] = 10 ** 6                  # position past the table
    c.batch_idx, c.input_pos = b, p
    kp, vp, out, lse, err = run_chunked(c, table=table)
    assert err & binding.DEV_ERR_BAD_PAGE and err & binding.DEV_ERR_BAD_SLOT
    assert err & binding.DEV_ERR_BAD_POS
    assert torch.all(out[[5, 80]] == 0) and torch.all(torch.isneginf(lse[[5, 80]]))
    ok_rows = [i for i in range(c.n_tokens) if int(b[i]) in (1, 3) and i not in (5, 80)]
    ref_o, ref_l, _, bad = oracle_chunked(c, rows=ok_rows, table=table)
    assert not bad
    assert_attention_close(out, lse, ref_o, ref_l, rows=ok_rows)


@pytest.mark.parametrize("offset_elems", [0, 8], ids=["out_32B_aligned", "out_16B_offset"])
def test_output_alignment_paths(offset_elems):
    """out needs only 16-byte alignment: a 32-byte-aligned buffer and one at
    a 16-byte offset both match the oracle, and nothing outside out is
    written."""
    c = W.chunked_prefill(5, prefix_lens=[100, 300, 0], chunk_lens=[140, 60, 33], page_size=64,
                          hq=16, hkv=4)
    kp, vp, pt = gpu(c.k_pool), gpu(c.v_pool), gpu(c.page_table)
    bidx, pos = gpu(c.batch_idx), gpu(c.input_pos)
    err = new_dev_err()
    binding.pkv_append(kp, vp, pt, gpu(c.k_new), gpu(c.v_new), bidx, pos, c.page_size,
                       dev_err=err)
    T, hq, d = c.q.shape
    buf = torch.full((T * hq * d + 16,), float("nan"), dtype=torch.bfloat16, device="cuda")
    out = buf[offset_elems:offset_elems + T * hq * d].view(T, hq, d)
    assert out.data_ptr() % 32 == (0 if offset_elems == 0 else 16)
    _, lse = binding.pkv_prefill_paged_attention(kp, vp, pt, gpu(c.q), bidx, pos, c.page_size,
                                                 c.scale, out=out, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ro, rl, bad_tok, bad = oracle_chunked(c)
    assert not bad_tok and not bad
    assert_attention_close(out.cpu(), lse.cpu(), ro, rl, tag=f"out offset {offset_elems}")
    # nothing written outside out
    rest = torch.cat([buf[:offset_elems], buf[offset_elems + T * hq * d:]]).cpu()
    assert torch.isnan(rest.float()).all()


def _sampled_tokens(c, n_random, seed):
    """First and last token of every run of one slot, and n_random others."""
    b = c.batch_idx.numpy()
    edges = np.flatnonzero(np.diff(b)) if len(b) > 1 else np.zeros(0, dtype=np.int64)
    rows = {0, len(b) - 1}
    rows.update(edges.tolist())
    rows.update((edges + 1).tolist())
    rng = np.random.default_rng(seed)
    rows.update(rng.choice(len(b), min(n_random, len(b)), replace=False).tolist())
    return sorted(rows)


def test_item_schedule_groups_of_many_tiles():
    """Items are dealt by estimated cost with the tiles of one run of equal
    slots kept together, costliest first: runs of 32, 6, 2 and 1 query tiles
    and a run of two tokens, shuffled, page 64."""
    c = W.chunked_prefill(12, prefix_lens=[100, 3000, 0, 50, 700, 9],
                          chunk_lens=[4096, 700, 129, 2, 300, 1], hq=8, hkv=2, page_size=64)
    _, _, out, lse, err = run_chunked(c)
    assert err == 0
    rows = _sampled_tokens(c, 600, 12)
    ro, rl, bad_tok, bad = oracle_chunked(c, rows=rows)
    assert not bad_tok and not bad
    assert_attention_close(out, lse, ro, rl, rows=rows, tag="groups")


def test_item_schedule_round_robin_above_768_tiles():
    """200 chunks of 512 tokens (800 query tiles) over prefixes U[0, 256]:
    past the sorted schedule's 768 tiles the items are dealt round-robin."""
    c = W.chunked_prefill(13, n_chunks=200, chunk=512, prefix_lo=0, prefix_hi=256, n_decode=0,
                          hq=8, hkv=2)
    assert (c.n_tokens + 127) // 128 == 800
    _, _, out, lse, err = run_chunked(c)
    assert err == 0
    rows = _sampled_tokens(c, 400, 13)
    ro, rl, bad_tok, bad = oracle_chunked(c, rows=rows)
    assert not bad_tok and not bad
    assert_attention_close(out, lse, ro, rl, rows=rows, tag="800 tiles")


def test_item_schedule_one_head_items():
    """GQA group 1 (one head per item): 40 chunks of 512 over prefixes
    U[0, 3000] (160 query tiles) on sampled tokens."""
    c = W.chunked_prefill(15, n_chunks=40, chunk=512, prefix_lo=0, prefix_hi=3000, n_decode=0,
                          hq=8, hkv=8)
    _, _, out, lse, err = run_chunked(c)
    assert err == 0
    rows = _sampled_tokens(c, 400, 15)
    ro, rl, bad_tok, bad = oracle_chunked(c, rows=rows)
    assert not bad_tok and not bad
    assert_attention_close(out, lse, ro, rl, rows=rows, tag="G=1 chunks")
