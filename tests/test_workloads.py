"""The seeded workload generators: reproducible, and shaped like the
workloads they stand in for."""

import torch

from paged_kv_gqa_pkv_gb300 import workloads as W


def _check_table(case, lens):
    t = case.page_table
    assert t.dtype == torch.int32 and torch.all(t[0] == -1)
    used = []
    for s, n in enumerate(lens, start=1):
        nb = -(-n // case.page_size)
        row = t[s]
        assert torch.all(row[:nb] >= 1) and torch.all(row[:nb] < case.num_pages)
        assert torch.all(row[nb:] == -1)
        used += row[:nb].tolist()
    assert len(used) == len(set(used)), "a page was handed out twice"
    assert 0 not in used


def test_tiny_decode_shape_and_determinism():
    a, b = W.tiny_decode(0), W.tiny_decode(0)
    assert torch.equal(a.q, b.q) and torch.equal(a.k_pool, b.k_pool)
    assert torch.equal(a.page_table, b.page_table)
    assert a.seq_lens.tolist() == [18, 65, 101, 131]
    assert a.input_pos.tolist() == [17, 64, 100, 130]
    assert a.num_pages == 32 and a.page_size == 16
    assert (a.num_q_heads, a.num_kv_heads, a.head_dim) == (8, 2, 128)
    _check_table(a, a.seq_lens.tolist())
    assert not torch.equal(W.tiny_decode(1).q, a.q)


def test_qwen3_b64_decode_ranges():
    for permute in (False, True):
        c = W.qwen3_b64_decode(0, permute=permute)
        lens = c.seq_lens.tolist()
        assert c.batch == 64 and min(lens) >= 512 and max(lens) <= 1024
        _check_table(c, lens)
        if not permute:
            for s, n in enumerate(lens, start=1):
                nb = -(-n // 128)
                r = c.page_table[s, :nb]
                assert torch.equal(r, r[0] + torch.arange(nb, dtype=torch.int32))
    # the two runs draw the same lengths (same seed), different page orders
    a, b = W.qwen3_b64_decode(0, False), W.qwen3_b64_decode(0, True)
    assert torch.equal(a.seq_lens, b.seq_lens)
    assert not torch.equal(a.page_table, b.page_table)


def test_padded_bucket_rows():
    c = W.padded_bucket_decode(0)
    assert c.batch == 64
    assert torch.all(c.batch_idx[:40] > 0) and torch.all(c.batch_idx[40:] == 0)
    lens = c.seq_lens[:40].tolist()
    assert min(lens) >= 1 and max(lens) <= 2048
    _check_table(c, lens)


def test_packed_prefill_layout():
    c = W.packed_prefill(0, n_docs=6, lo=3, hi=40)
    T = c.n_tokens
    assert T == sum(c.doc_lens)
    start = 0
    for s, n in enumerate(c.doc_lens, start=1):
        assert torch.all(c.batch_idx[start:start + n] == s)
        assert torch.equal(c.input_pos[start:start + n], torch.arange(n, dtype=torch.int32))
        start += n
    _check_table(c, c.doc_lens)


def test_full_size_prefill_token_count():
    c = W.packed_prefill(0)
    assert len(c.doc_lens) == 64 and min(c.doc_lens) >= 64 and max(c.doc_lens) <= 1024
    assert 25_000 < c.n_tokens < 45_000
