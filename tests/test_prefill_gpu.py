"""K4 tcgen05 packed document-causal prefill on the GPU against the float64
oracle: small cases in full, the 64-document workload at full size on
every row, padding tokens, other GQA groups, a packing that breaks the
precondition, and a run of changing token counts in one process."""

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


def _run(case, bidx=None, pos=None):
    bidx = case.batch_idx if bidx is None else bidx
    pos = case.input_pos if pos is None else pos
    err = new_dev_err()
    out, lse = binding.pkv_prefill_attention(gpu(case.q), gpu(case.k), gpu(case.v), gpu(bidx),
                                             gpu(pos), case.scale, dev_err=err)
    torch.cuda.synchronize()
    return out.cpu(), lse.cpu(), int(err.item())


def _oracle(case, rows=None, bidx=None, pos=None):
    bidx = case.batch_idx if bidx is None else bidx
    pos = case.input_pos if pos is None else pos
    return orc.prefill_attention(bf16_bits(case.q), bf16_bits(case.k), bf16_bits(case.v),
                                 bidx.numpy(), pos.numpy(), case.scale, rows=rows)


def test_tiny_single_document():
    c = W.packed_prefill(1, doc_lens=[5], hq=8, hkv=2)
    out, lse, err = _run(c)
    ro, rl = _oracle(c)
    assert err == 0
    assert_attention_close(out, lse, ro, rl, tag="5 tokens")


@pytest.mark.parametrize("doc_lens", [[1, 5, 130, 17, 256, 3], [128], [129], [300, 1, 1, 77],
                                      [1] * 40, [700]])
def test_small_packings(doc_lens):
    c = W.packed_prefill(2, doc_lens=doc_lens, hq=8, hkv=2)
    out, lse, err = _run(c)
    ro, rl = _oracle(c)
    assert err == 0
    assert_attention_close(out, lse, ro, rl, tag=str(doc_lens))


@pytest.mark.parametrize("hq,hkv", [(8, 8), (16, 8), (32, 4)])
def test_other_gqa_groups(hq, hkv):
    c = W.packed_prefill(3, doc_lens=[200, 57, 129], hq=hq, hkv=hkv)
    out, lse, err = _run(c)
    ro, rl = _oracle(c)
    assert err == 0
    assert_attention_close(out, lse, ro, rl, tag=f"G={hq // hkv}")


def test_padding_tokens_give_zero():
    """The pages pad the packing to a multiple of the block size with slot-0
    tokens at position 0; those rows attend nothing."""
    c = W.packed_prefill(4, doc_lens=[100, 90], hq=8, hkv=2)
    T = c.n_tokens
    pad = 66
    import copy
    c2 = copy.copy(c)
    gen = torch.Generator().manual_seed(9)
    c2.q = torch.cat([c.q, torch.randn((pad, 8, 128), generator=gen).to(torch.bfloat16)])
    c2.k = torch.cat([c.k, torch.randn((pad, 2, 128), generator=gen).to(torch.bfloat16)])
    c2.v = torch.cat([c.v, torch.randn((pad, 2, 128), generator=gen).to(torch.bfloat16)])
    c2.batch_idx = torch.cat([c.batch_idx, torch.zeros(pad, dtype=torch.int32)])
    c2.input_pos = torch.cat([c.input_pos, torch.zeros(pad, dtype=torch.int32)])
    out, lse, err = _run(c2)
    assert err == 0
    assert torch.all(out[T:] == 0) and torch.all(torch.isneginf(lse[T:]))
    ro, rl = _oracle(c2)
    assert_attention_close(out, lse, ro, rl)


def test_full_size_64_documents_every_row():
    """The 64-document workload (lengths uniform in [64, 1024], T = 32 718) in
    the launch configuration the bench times; every row of every head is
    compared with the oracle (run over all host cores, a document per task)."""
    c = W.packed_prefill(0)
    out, lse, err = _run(c)
    assert err == 0
    ro_bits, rl = oracle_pool.prefill_all_rows(bf16_bits(c.q), bf16_bits(c.k), bf16_bits(c.v),
                                               c.batch_idx.numpy(), c.input_pos.numpy(),
                                               c.scale)
    assert not np.isnan(rl).any()
    assert_attention_close(out, lse, orc.bf16_bits_to_f64(ro_bits), rl, tag="64 docs")


def test_layout_violation_is_flagged():
    c = W.packed_prefill(5, doc_lens=[40, 40], hq=8, hkv=2)
    pos = c.input_pos.clone()
    pos[50] = 3                      # breaks the 0, 1, 2, ... numbering
    out, lse, err = _run(c, pos=pos)
    assert err & binding.DEV_ERR_LAYOUT
    rows = list(range(40))           # the first document is untouched
    ro, rl = _oracle(c, rows=rows, pos=pos)
    assert_attention_close(out, lse, ro, rl, rows=rows)


def test_changing_token_counts_in_one_process():
    """A small packing, a large one, then small again: nothing may be
    specialised on the first shape (the pages hit exactly this with a cached
    mask kernel; "flex_paged_attention.py" commit log)."""
    for lens in ([17, 3], [900, 400, 1024, 64, 300], [5, 9, 2]):
        c = W.packed_prefill(6, doc_lens=lens, hq=32, hkv=8)
        out, lse, err = _run(c)
        assert err == 0
        ro, rl = _oracle(c)
        assert_attention_close(out, lse, ro, rl, tag=str(lens))


def test_prefill_rejects_bad_host_arguments():
    c = W.packed_prefill(7, doc_lens=[10], hq=8, hkv=2)
    with pytest.raises(binding.PkvError) as e:
        binding.pkv_prefill_attention(gpu(c.q), gpu(c.k), gpu(c.v), gpu(c.batch_idx),
                                      gpu(c.input_pos), -0.1)
    assert e.value.status == 1


def _sampled_rows(case, n_random, seed):
    """Every document's first and last rows and n_random others."""
    rows = set()
    start = 0
    for n in case.doc_lens:
        rows.update((start, start + n - 1))
        start += n
    rng = np.random.default_rng(seed)
    rows.update(rng.choice(case.n_tokens, n_random, replace=False).tolist())
    return sorted(rows)


@pytest.mark.parametrize("n_tiles", [330, 768, 769])
def test_item_schedule_sorted_windows_and_round_robin(n_tiles):
    """The items are sorted by estimated cost within windows of eight rounds
    (here 304 query tiles: one head pair per item, 152 SMs) up to 768 query
    tiles and dealt round-robin above: a last window cut short (330), the
    limit (768) and one tile past it (769). Documents of U[64, 1200] tokens;
    every document's first and last rows and 400 others against the oracle."""
    T = n_tiles * 128 - 37
    rng = np.random.default_rng(n_tiles)
    lens = []
    while sum(lens) < T:
        lens.append(int(rng.integers(64, 1201)))
    lens[-1] = T - sum(lens[:-1])
    c = W.packed_prefill(9, doc_lens=lens, hq=8, hkv=2)
    assert c.n_tokens == T and (T + 127) // 128 == n_tiles
    out, lse, err = _run(c)
    assert err == 0
    rows = _sampled_rows(c, 400, n_tiles)
    ro, rl = _oracle(c, rows=rows)
    assert_attention_close(out, lse, ro, rl, rows=rows, tag=f"{n_tiles} tiles")


def test_item_schedule_one_head_items():
    """GQA group 1 (one head per item, 16 items per query tile): the sort
    windows are then 8 * 152 / 16 = 76 tiles; 300 query tiles of documents
    U[64, 1200] on sampled rows."""
    T = 300 * 128 - 5
    rng = np.random.default_rng(300)
    lens = []
    while sum(lens) < T:
        lens.append(int(rng.integers(64, 1201)))
    lens[-1] = T - sum(lens[:-1])
    c = W.packed_prefill(10, doc_lens=lens, hq=16, hkv=16)
    out, lse, err = _run(c)
    assert err == 0
    rows = _sampled_rows(c, 400, 300)
    ro, rl = _oracle(c, rows=rows)
    assert_attention_close(out, lse, ro, rl, rows=rows, tag="G=1")
