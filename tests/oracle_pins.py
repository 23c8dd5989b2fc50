"""Checks that pin the float64 oracle to facts other than itself.

Each ``check_*`` takes the oracle module (``oracle.paged_attention``, or a
copy with a planted mistake) and raises ``AssertionError`` when the oracle
disagrees with a fixed fact:

* library special cases: PyTorch's float64 ``scaled_dot_product_attention``
  (dense softmax attention with grouped-query heads, causal or with an
  explicit mask), PyTorch's float32->bf16 and bf16->float64 conversions, and
  a NumPy fancy-index scatter;
* closed forms: one key, n identical keys, documents of one token;
* invariants: permuting physical pages, splitting a document, interleaving
  documents in the packing, and decode at a document's last token agreeing
  with prefill.

The LSE is pinned through the library routine with a probe key: appending a
key of all zeros (score 0 for every head) whose value is a one-hot extra
column makes the library's output in that column equal exp(-lse'), where
lse' = log(exp(lse) + 1). Solving gives lse = log(1/w - 1).
"""

from __future__ import annotations

import math

import numpy as np
import torch
import torch.nn.functional as F

D = 128


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _rand_bf16(gen, shape) -> torch.Tensor:
    return torch.randn(shape, generator=gen, dtype=torch.float32).to(torch.bfloat16)


def _sdpa_with_probe(q, k, v, mask=None):
    """Library attention plus probe-derived LSE.

    q [Hq, L, E], k [Hkv, S, E], v [Hkv, S, E] float64; mask [L, S] bool
    (True = may attend) or None. Returns (out [Hq, L, E], lse [Hq, L])."""
    hkv, S, E = k.shape
    kz = torch.cat([torch.zeros(hkv, 1, E, dtype=k.dtype), k], dim=1)
    vz = torch.cat([v, torch.zeros(hkv, S, 1, dtype=v.dtype)], dim=2)
    probe_v = torch.zeros(hkv, 1, E + 1, dtype=v.dtype)
    probe_v[..., E] = 1.0
    vz = torch.cat([probe_v, vz], dim=1)
    if mask is not None:
        L = mask.shape[0]
        mz = torch.cat([torch.ones(L, 1, dtype=torch.bool), mask], dim=1)
    else:
        mz = None
    scale = 1.0 / math.sqrt(E)
    with_probe = F.scaled_dot_product_attention(
        q[None], kz[None], vz[None], attn_mask=mz, scale=scale,
        enable_gqa=True)[0]
    w = with_probe[..., E]
    lse = torch.log(1.0 / w - 1.0)
    plain = F.scaled_dot_product_attention(
        q[None], k[None], v[None],
        attn_mask=mask, scale=scale, enable_gqa=True)[0]
    return plain, lse


# ---------------------------------------------------------------- bf16 ----

def check_bf16_conversions(orc):
    all_bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    mine = orc.bf16_bits_to_f64(all_bits)
    lib = torch.from_numpy(all_bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(lib)
    assert np.array_equal(np.isnan(mine), nan)
    assert np.array_equal(mine[~nan], lib[~nan])

    gen = torch.Generator().manual_seed(7)
    x32 = torch.randn(200000, generator=gen) * torch.exp2(torch.randint(-140, 120, (200000,), generator=gen).float())
    # exact ties on the bf16 grid: odd multiples of half an ulp
    ties = (1.0 + (2 * torch.arange(0, 256) + 1).float() * 2.0 ** -8) * 2.0 ** torch.randint(-100, 100, (256,)).float()
    x32 = torch.cat([x32, ties, -ties]).to(torch.float32)
    x32 = x32[torch.isfinite(x32)]
    lib_bits = _bits(x32.to(torch.bfloat16))
    mine_bits = orc.f64_to_bf16_bits(x32.to(torch.float64).numpy())
    assert np.array_equal(lib_bits, mine_bits)

    fixed = {
        1.0: 0x3F80, -2.0: 0xC000, 1.0 + 2.0 ** -8: 0x3F80,
        1.0 + 3 * 2.0 ** -8: 0x3F82, 2.0 ** -133: 0x0001,
        float.fromhex("0x1.fep127"): 0x7F7F, 2.0 ** 128: 0x7F80,
        # direct rounding from float64: just above the tie, so up. Rounding
        # through float32 first would land on the tie and go to even.
        1.0 + 2.0 ** -8 + 2.0 ** -30: 0x3F81,
    }
    got = orc.f64_to_bf16_bits(np.array(list(fixed.keys())))
    assert [int(b) for b in got] == list(fixed.values()), [hex(int(b)) for b in got]


# -------------------------------------------------------------- append ----

def check_append_scatter(orc):
    gen = torch.Generator().manual_seed(11)
    ps, P, hkv, maxb, nb = 16, 24, 2, 6, 5
    pool_k = np.random.default_rng(1).integers(0, 65536, (P * ps, hkv, D), dtype=np.uint16)
    pool_v = np.random.default_rng(2).integers(0, 65536, (P * ps, hkv, D), dtype=np.uint16)
    perm = (torch.randperm(P - 1, generator=gen) + 1).numpy()
    table = np.full((maxb, nb), -1, dtype=np.int32)
    table[1:, :4] = perm[:20].reshape(5, 4)
    table[0, :] = 0             # padding slot routed to the reserved page 0
    table[3, 2] = -1            # an unreserved entry inside a sequence
    table[4, 1] = P + 3         # an entry past the pool
    N = 40
    rng = np.random.default_rng(3)
    bidx = rng.integers(0, maxb, N).astype(np.int32)
    pos = rng.integers(0, 4 * ps, N).astype(np.int32)
    pos[:3] = [5 * ps, nb * ps + 1, 3]      # block past the table
    bidx[2] = maxb                           # slot past the table
    # positions unique per slot, so later writes never overwrite earlier ones
    seen = set()
    for i in range(N):
        while (int(bidx[i]), int(pos[i])) in seen:
            pos[i] = (pos[i] + 1) % (4 * ps)
        seen.add((int(bidx[i]), int(pos[i])))
    k_new = rng.integers(0, 65536, (N, hkv, D), dtype=np.uint16)
    v_new = rng.integers(0, 65536, (N, hkv, D), dtype=np.uint16)

    ko, vo, bad = orc.append(pool_k, pool_v, table, k_new, v_new, bidx, pos, ps)

    # independent: vectorised address formula + NumPy fancy-index scatter
    ek, ev = pool_k.copy(), pool_v.copy()
    in_table = (bidx >= 0) & (bidx < maxb) & (pos // ps < nb)
    page = np.full(N, -1, dtype=np.int64)
    page[in_table] = table[bidx[in_table], pos[in_table] // ps]
    ok = in_table & (page >= 0) & (page < P)
    live = ok & (bidx != 0)
    rows = page[live] * ps + pos[live] % ps
    ek[rows] = k_new[live]
    ev[rows] = v_new[live]
    assert np.array_equal(ko, ek) and np.array_equal(vo, ev)
    assert sorted(bad) == sorted(np.nonzero(~ok & (bidx != 0))[0].tolist())
    assert len(bad) >= 4
    # the padding slot is never written: page 0 rows are untouched
    assert np.array_equal(ko[:ps], pool_k[:ps])


# -------------------------------------------------------------- decode ----

def _sequential_case(seed, lens, hq, hkv, ps, start_page=1, slack_pages=2):
    """Decode inputs whose slots own consecutive pages, so logical keys of a
    slot are one contiguous run of the pool (readable without the table)."""
    gen = torch.Generator().manual_seed(seed)
    blocks = [-(-n // ps) for n in lens]
    P = start_page + sum(blocks) + slack_pages
    table = np.full((len(lens) + 1, max(max(blocks), 1)), -1, dtype=np.int32)
    starts = []
    nxt = start_page
    for s, nbk in enumerate(blocks, start=1):
        table[s, :nbk] = np.arange(nxt, nxt + nbk)
        starts.append(nxt * ps)
        nxt += nbk
    kp = _rand_bf16(gen, (P * ps, hkv, D))
    vp = _rand_bf16(gen, (P * ps, hkv, D))
    q = _rand_bf16(gen, (len(lens), hq, D))
    return dict(kp=kp, vp=vp, q=q, table=table, starts=starts, ps=ps, P=P,
                bidx=np.arange(1, len(lens) + 1, dtype=np.int32),
                lens=np.asarray(lens, dtype=np.int32))


def check_decode_matches_library(orc):
    for (hq, hkv, ps, lens) in [(8, 2, 16, [1, 5, 16, 17, 40]),
                                (4, 4, 32, [3, 64, 33]),
                                (6, 2, 16, [31, 2])]:
        c = _sequential_case(5, lens, hq, hkv, ps)
        out, lse, bad = orc.decode_attention(
            _bits(c["q"]), _bits(c["kp"]), _bits(c["vp"]), c["table"],
            c["bidx"], c["lens"], ps, 1.0 / math.sqrt(D))
        assert not bad
        for b, n in enumerate(lens):
            s0 = c["starts"][b]
            K = c["kp"][s0:s0 + n].to(torch.float64).permute(1, 0, 2)  # [Hkv, n, D]
            V = c["vp"][s0:s0 + n].to(torch.float64).permute(1, 0, 2)
            Q = c["q"][b].to(torch.float64)[:, None, :]                # [Hq, 1, D]
            ref_o, ref_lse = _sdpa_with_probe(Q, K, V)
            assert np.allclose(out[b], ref_o[:, 0].numpy(), atol=1e-12, rtol=0)
            assert np.allclose(lse[b], ref_lse[:, 0].numpy(), atol=1e-9, rtol=0)


def check_permutation_invariance(orc):
    hq, hkv, ps = 8, 2, 16
    lens = [18, 65, 101, 131]
    c = _sequential_case(9, lens, hq, hkv, ps, slack_pages=5)
    args = (_bits(c["q"]),)
    kb, vb = _bits(c["kp"]), _bits(c["vp"])
    o1, l1, _ = orc.decode_attention(args[0], kb, vb, c["table"], c["bidx"],
                                     c["lens"], ps, 1.0 / math.sqrt(D))
    # move every physical page p to sigma(p) and rewrite the table
    rng = np.random.default_rng(4)
    P = c["P"]
    sigma = np.concatenate([[0], rng.permutation(np.arange(1, P))])
    kb2, vb2 = np.empty_like(kb), np.empty_like(vb)
    for p in range(P):
        kb2[sigma[p] * ps:(sigma[p] + 1) * ps] = kb[p * ps:(p + 1) * ps]
        vb2[sigma[p] * ps:(sigma[p] + 1) * ps] = vb[p * ps:(p + 1) * ps]
    t2 = np.where(c["table"] >= 0, sigma[np.maximum(c["table"], 0)], -1).astype(np.int32)
    assert not np.array_equal(t2, c["table"])
    o2, l2, _ = orc.decode_attention(args[0], kb2, vb2, t2, c["bidx"],
                                     c["lens"], ps, 1.0 / math.sqrt(D))
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def check_single_key(orc):
    hq, hkv, ps = 8, 2, 16
    c = _sequential_case(13, [1, 1, 1], hq, hkv, ps)
    out, lse, _ = orc.decode_attention(
        _bits(c["q"]), _bits(c["kp"]), _bits(c["vp"]), c["table"], c["bidx"],
        c["lens"], ps, 1.0 / math.sqrt(D))
    g = hq // hkv
    for b in range(3):
        row = c["starts"][b]
        for h in range(hq):
            v = c["vp"][row, h // g].to(torch.float64).numpy()
            assert np.array_equal(out[b, h], v)
            qk = math.fsum((c["q"][b, h].to(torch.float64) *
                            c["kp"][row, h // g].to(torch.float64)).tolist())
            assert abs(lse[b, h] - qk / math.sqrt(D)) <= 1e-12 * max(1.0, abs(qk))


def check_identical_keys(orc):
    """n copies of one (k, v): out = v and lse = s + ln n for every n."""
    hq, hkv, ps = 4, 2, 16
    gen = torch.Generator().manual_seed(17)
    kr, vr = _rand_bf16(gen, (hkv, D)), _rand_bf16(gen, (hkv, D))
    lens = [1, 2, 7, 16, 33]
    c = _sequential_case(17, lens, hq, hkv, ps)
    kp, vp = c["kp"].clone(), c["vp"].clone()
    kp[:] = kr
    vp[:] = vr
    out, lse, _ = orc.decode_attention(
        _bits(c["q"]), _bits(kp), _bits(vp), c["table"], c["bidx"], c["lens"],
        ps, 1.0 / math.sqrt(D))
    g = hq // hkv
    for b, n in enumerate(lens):
        for h in range(hq):
            v = vr[h // g].to(torch.float64).numpy()
            assert np.allclose(out[b, h], v, atol=1e-14, rtol=1e-14)
            s = math.fsum((c["q"][b, h].to(torch.float64) *
                           kr[h // g].to(torch.float64)).tolist()) / math.sqrt(D)
            assert abs(lse[b, h] - (s + math.log(n))) <= 1e-12


def check_all_masked(orc):
    hq, hkv, ps = 8, 2, 16
    c = _sequential_case(19, [5, 9, 3], hq, hkv, ps)
    bidx = np.array([0, 2, 0, 3], dtype=np.int32)     # slot 0 = padding
    lens = np.array([1, 0, 7, 3], dtype=np.int32)     # row 1: no keys
    q = _rand_bf16(torch.Generator().manual_seed(1), (4, hq, D))
    out, lse, bad = orc.decode_attention(
        _bits(q), _bits(c["kp"]), _bits(c["vp"]), c["table"], bidx, lens, ps,
        1.0 / math.sqrt(D))
    assert not bad
    for b in (0, 1, 2):
        assert np.all(out[b] == 0.0) and not np.any(np.isnan(out[b]))
        assert np.all(np.isneginf(lse[b]))
    assert np.all(np.isfinite(lse[3]))


def check_unaddressable_rows_flagged(orc):
    hq, hkv, ps = 4, 2, 16
    c = _sequential_case(23, [20, 20], hq, hkv, ps)
    table = c["table"].copy()
    table[2, 1] = -1
    out, lse, bad = orc.decode_attention(
        _bits(c["q"]), _bits(c["kp"]), _bits(c["vp"]), table, c["bidx"],
        c["lens"], ps, 1.0 / math.sqrt(D))
    assert bad == [1]
    assert np.all(np.isfinite(out[0]))


# ------------------------------------------------------------- prefill ----

def _prefill_inputs(seed, doc_lens, hq=8, hkv=2):
    gen = torch.Generator().manual_seed(seed)
    T = sum(doc_lens)
    q = _rand_bf16(gen, (T, hq, D))
    k = _rand_bf16(gen, (T, hkv, D))
    v = _rand_bf16(gen, (T, hkv, D))
    bidx = np.concatenate([np.full(n, s + 1) for s, n in enumerate(doc_lens)]).astype(np.int32)
    pos = np.concatenate([np.arange(n) for n in doc_lens]).astype(np.int32)
    return q, k, v, bidx, pos


def check_prefill_single_doc_causal(orc):
    for n, hq, hkv in [(1, 4, 2), (37, 8, 2), (130, 4, 4)]:
        q, k, v, bidx, pos = _prefill_inputs(29, [n], hq, hkv)
        out, lse = orc.prefill_attention(_bits(q), _bits(k), _bits(v), bidx,
                                         pos, 1.0 / math.sqrt(D))
        Q = q.to(torch.float64).permute(1, 0, 2)
        K = k.to(torch.float64).permute(1, 0, 2)
        V = v.to(torch.float64).permute(1, 0, 2)
        ref = F.scaled_dot_product_attention(Q[None], K[None], V[None],
                                             is_causal=True, enable_gqa=True,
                                             scale=1.0 / math.sqrt(D))[0]
        assert np.allclose(out, ref.permute(1, 0, 2).numpy(), atol=1e-12, rtol=0)
        causal = torch.ones(n, n, dtype=torch.bool).tril()
        _, ref_lse = _sdpa_with_probe(Q, K, V, mask=causal)
        assert np.allclose(lse, ref_lse.T.numpy(), atol=1e-9, rtol=0)


def check_prefill_length_one_docs(orc):
    hq, hkv = 8, 2
    q, k, v, bidx, pos = _prefill_inputs(31, [1] * 9, hq, hkv)
    out, lse = orc.prefill_attention(_bits(q), _bits(k), _bits(v), bidx, pos,
                                     1.0 / math.sqrt(D))
    g = hq // hkv
    for i in range(9):
        for h in range(hq):
            assert np.array_equal(out[i, h], v[i, h // g].to(torch.float64).numpy())
            s = math.fsum((q[i, h].to(torch.float64) *
                           k[i, h // g].to(torch.float64)).tolist()) / math.sqrt(D)
            assert abs(lse[i, h] - s) <= 1e-12


def check_prefill_split_document(orc):
    q, k, v, bidx, pos = _prefill_inputs(37, [50])
    scale = 1.0 / math.sqrt(D)
    o1, l1 = orc.prefill_attention(_bits(q), _bits(k), _bits(v), bidx, pos, scale)
    b2, p2 = bidx.copy(), pos.copy()
    b2[20:] = 2
    p2[20:] = np.arange(30)
    o2, l2 = orc.prefill_attention(_bits(q), _bits(k), _bits(v), b2, p2, scale)
    assert np.array_equal(o1[:20], o2[:20]) and np.array_equal(l1[:20], l2[:20])
    assert not np.allclose(o1[21:], o2[21:])
    # the first token after the split sees only itself
    assert np.array_equal(o2[20, 0], v[20, 0].to(torch.float64).numpy())


def check_prefill_interleaved_documents(orc):
    """Masking is by slot and position, not by packed index: shuffling the
    packed order only permutes the result rows."""
    q, k, v, bidx, pos = _prefill_inputs(41, [23, 17, 9])
    scale = 1.0 / math.sqrt(D)
    o1, l1 = orc.prefill_attention(_bits(q), _bits(k), _bits(v), bidx, pos, scale)
    perm = np.random.default_rng(5).permutation(len(bidx))
    o2, l2 = orc.prefill_attention(_bits(q[perm]), _bits(k[perm]), _bits(v[perm]),
                                   bidx[perm], pos[perm], scale)
    assert np.allclose(o2, o1[perm], atol=1e-13, rtol=0)
    assert np.allclose(l2, l1[perm], atol=1e-12, rtol=0)
    # padding tokens (slot 0) attend nothing and are attended by nobody
    b3 = bidx.copy()
    b3[5] = 0
    o3, l3 = orc.prefill_attention(_bits(q), _bits(k), _bits(v), b3, pos, scale)
    assert np.all(o3[5] == 0.0) and np.all(np.isneginf(l3[5]))
    assert np.array_equal(o3[:5], o1[:5])
    assert not np.allclose(o3[6:23], o1[6:23])


def check_prefill_decode_consistency(orc):
    """The last token of a document, prefilled, equals a decode step over the
    document's k/v appended into a paged pool."""
    hq, hkv, ps = 8, 2, 16
    lens = [19, 40, 7]
    q, k, v, bidx, pos = _prefill_inputs(43, lens, hq, hkv)
    scale = 1.0 / math.sqrt(D)
    o_pre, l_pre = orc.prefill_attention(_bits(q), _bits(k), _bits(v), bidx, pos, scale)
    P = 1 + sum(-(-n // ps) for n in lens) + 3
    table = np.full((len(lens) + 1, 4), -1, dtype=np.int32)
    pages = np.random.default_rng(6).permutation(np.arange(1, P))
    j = 0
    for s, n in enumerate(lens, start=1):
        nbk = -(-n // ps)
        table[s, :nbk] = pages[j:j + nbk]
        j += nbk
    zeros = np.zeros((P * ps, hkv, D), dtype=np.uint16)
    kp, vp, bad = orc.append(zeros, zeros, table, _bits(k), _bits(v), bidx, pos, ps)
    assert not bad
    last = np.cumsum(lens) - 1
    o_dec, l_dec, bad = orc.decode_attention(
        _bits(q[last]), kp, vp, table, bidx[last], np.asarray(lens), ps, scale)
    assert not bad
    assert np.array_equal(o_dec, o_pre[last]) and np.array_equal(l_dec, l_pre[last])


ALL_CHECKS = [
    check_bf16_conversions,
    check_append_scatter,
    check_decode_matches_library,
    check_permutation_invariance,
    check_single_key,
    check_identical_keys,
    check_all_masked,
    check_unaddressable_rows_flagged,
    check_prefill_single_doc_causal,
    check_prefill_length_one_docs,
    check_prefill_split_document,
    check_prefill_interleaved_documents,
    check_prefill_decode_consistency,
]


# ---------------------------------------------------------------- rope ----

def check_rope_closed_forms(orc):
    gen = torch.Generator().manual_seed(47)
    N, H = 6, 3
    x = _bits(_rand_bf16(gen, (N, H, D)))
    xf = orc.bf16_bits_to_f64(x)
    half = D // 2
    pos = np.arange(N)
    # angle 0: identity
    c0, s0 = np.ones((N, half)), np.zeros((N, half))
    assert np.array_equal(orc.rope(x, pos, c0, s0), xf)
    # angle 90 degrees: (x1, x2) -> (-x2, x1)
    c9, s9 = np.zeros((N, half)), np.ones((N, half))
    r = orc.rope(x, pos, c9, s9)
    assert np.array_equal(r[..., :half], -xf[..., half:]) and np.array_equal(r[..., half:], xf[..., :half])
    # a rotation keeps each (d, d + D/2) pair's length, for any angles
    ang = np.random.default_rng(1).uniform(-7, 7, (N, half))
    r = orc.rope(x, pos, np.cos(ang), np.sin(ang))
    n_in = xf[..., :half] ** 2 + xf[..., half:] ** 2
    n_out = r[..., :half] ** 2 + r[..., half:] ** 2
    assert np.allclose(n_in, n_out, rtol=1e-12, atol=1e-12)


def check_rope_relative_position(orc):
    """With the standard table, <rope(q, m), rope(k, n)> depends only on m - n."""
    from paged_kv_gqa_pkv_gb300.workloads import rope_tables
    cos_t, sin_t = rope_tables(64)
    gen = torch.Generator().manual_seed(53)
    q = _bits(_rand_bf16(gen, (1, 1, D)))
    k = _bits(_rand_bf16(gen, (1, 1, D)))
    def dot(m, n):
        return float(np.sum(orc.rope(q, np.array([m]), cos_t.numpy(), sin_t.numpy()) *
                            orc.rope(k, np.array([n]), cos_t.numpy(), sin_t.numpy())))
    for m, n in [(9, 4), (30, 2), (17, 17)]:
        assert abs(dot(m, n) - dot(m + 13, n + 13)) < 1e-5 * (1 + abs(dot(m, n)))
    assert abs(dot(9, 4) - dot(4, 9)) > 1e-3   # but it does depend on the sign of m - n


def check_append_rope(orc):
    gen = torch.Generator().manual_seed(59)
    ps, P, hkv = 16, 10, 2
    from paged_kv_gqa_pkv_gb300.workloads import rope_tables
    cos_t, sin_t = rope_tables(40)
    kp = _bits(_rand_bf16(gen, (P * ps, hkv, D)))
    vp = _bits(_rand_bf16(gen, (P * ps, hkv, D)))
    table = np.full((3, 4), -1, dtype=np.int32)
    table[1, :2] = [3, 5]
    table[2, :3] = [7, 1, 2]
    bidx = np.array([1, 2, 0, 2, 1], dtype=np.int32)
    pos = np.array([0, 33, 3, 39, 40], dtype=np.int32)   # 40: past the table
    kn = _bits(_rand_bf16(gen, (5, hkv, D)))
    vn = _bits(_rand_bf16(gen, (5, hkv, D)))
    ko, vo, bad = orc.append_rope(kp, vp, table, kn, vn, bidx, pos, ps, cos_t.numpy(),
                                  sin_t.numpy())
    assert bad == [4]
    # position 0 is the identity rotation: the raw row lands unchanged
    assert np.array_equal(ko[3 * ps + 0], kn[0])
    rot = orc.f64_to_bf16_bits(orc.rope(kn[1:2], pos[1:2], cos_t.numpy(), sin_t.numpy()))[0]
    assert np.array_equal(ko[2 * ps + 33 % ps], rot) and np.array_equal(vo[2 * ps + 1], vn[1])
    assert not np.array_equal(rot, kn[1])


ALL_CHECKS += [check_rope_closed_forms, check_rope_relative_position, check_append_rope]


# -------------------------------------------------------------- k_norm ----

def check_k_norm_closed_forms(orc):
    # x = (3, 4, 0, ..., 0): mean of squares 25/D, so out = w * x * sqrt(D) / 5
    x = np.zeros((1, 1, D), dtype=np.float32)
    x[0, 0, 0], x[0, 0, 1] = 3.0, 4.0
    xb = _bits(torch.from_numpy(x).to(torch.bfloat16))
    w = np.linspace(0.5, 1.5, D)
    r = orc.k_norm(xb, w, 0.0)
    want = np.zeros(D)
    want[0], want[1] = 3.0 * w[0] * math.sqrt(D) / 5.0, 4.0 * w[1] * math.sqrt(D) / 5.0
    assert np.allclose(r[0, 0], want, rtol=1e-15, atol=0)
    # a constant head a: out = w * a / sqrt(a^2 + eps), eps included
    a, eps = 0.375, 0.5
    xc = _bits(torch.full((2, 3, D), a).to(torch.bfloat16))
    rc = orc.k_norm(xc, w, eps)
    assert np.allclose(rc, np.broadcast_to(w * a / math.sqrt(a * a + eps), rc.shape),
                       rtol=1e-15, atol=0)
    # all-zero head with eps > 0: zeros, not NaN
    z = orc.k_norm(np.zeros((1, 2, D), dtype=np.uint16), w, 1e-6)
    assert np.array_equal(z, np.zeros((1, 2, D)))


def check_k_norm_invariants(orc):
    gen = torch.Generator().manual_seed(61)
    x = _bits(_rand_bf16(gen, (5, 4, D)))
    # unit weight, eps 0: every head comes out with root-mean-square exactly 1
    r = orc.k_norm(x, np.ones(D), 0.0)
    assert np.allclose(np.sqrt(np.mean(r * r, axis=-1)), 1.0, rtol=1e-14)
    # scaling a head by a power of two (exact in bf16) leaves it unchanged at eps 0
    x2 = _bits(torch.from_numpy(orc.bf16_bits_to_f64(x) * 2.0).to(torch.bfloat16))
    w = np.random.default_rng(3).uniform(0.5, 1.5, D)
    assert np.array_equal(orc.k_norm(x2, w, 0.0), orc.k_norm(x, w, 0.0))
    # the weight multiplies its own dim: two weights differing in one dim
    # change that dim only
    w2 = w.copy()
    w2[77] *= 3.0
    d = orc.k_norm(x, w2, 1e-6) - orc.k_norm(x, w, 1e-6)
    assert np.count_nonzero(d[..., np.arange(D) != 77]) == 0
    assert np.count_nonzero(d[..., 77]) == d[..., 77].size


def check_append_rope_k_norm(orc):
    """append_rope with k_norm against the same arithmetic written another
    way: the norm through np.linalg.norm, the rotation as complex
    multiplication (x1 + i x2) * exp(i theta), one rounding at the end."""
    gen = torch.Generator().manual_seed(67)
    ps, P, hkv = 16, 10, 2
    from paged_kv_gqa_pkv_gb300.workloads import rope_tables
    cos_t, sin_t = rope_tables(40)
    kp = _bits(_rand_bf16(gen, (P * ps, hkv, D)))
    vp = _bits(_rand_bf16(gen, (P * ps, hkv, D)))
    table = np.full((3, 4), -1, dtype=np.int32)
    table[1, :2] = [3, 5]
    table[2, :3] = [7, 1, 2]
    bidx = np.array([1, 2, 0, 2], dtype=np.int32)
    pos = np.array([0, 33, 3, 39], dtype=np.int32)
    kn = _bits(_rand_bf16(gen, (4, hkv, D)) * 3.0)
    vn = _bits(_rand_bf16(gen, (4, hkv, D)))
    w = np.random.default_rng(5).uniform(0.25, 2.0, D)   # not symmetric in d, d + D/2
    eps = 1e-6
    ko, vo, bad = orc.append_rope(kp, vp, table, kn, vn, bidx, pos, ps, cos_t.numpy(),
                                  sin_t.numpy(), k_norm_weight=w, k_norm_eps=eps)
    assert bad == []
    half = D // 2
    for i, row in [(0, 3 * ps + 0), (1, 2 * ps + 33 % ps), (3, 2 * ps + 39 % ps)]:
        xf = orc.bf16_bits_to_f64(kn[i])                       # [hkv, D]
        rms = np.linalg.norm(xf, axis=-1, keepdims=True) / math.sqrt(D)
        y = w * xf / np.sqrt(rms * rms + eps)
        theta = np.arctan2(sin_t.numpy()[pos[i]].astype(np.float64),
                           cos_t.numpy()[pos[i]].astype(np.float64))
        mag = np.hypot(sin_t.numpy()[pos[i]].astype(np.float64),
                       cos_t.numpy()[pos[i]].astype(np.float64))
        zc = (y[:, :half] + 1j * y[:, half:]) * (mag * np.exp(1j * theta))
        want = np.concatenate([zc.real, zc.imag], axis=-1)
        got = orc.bf16_bits_to_f64(ko[row])
        ulp = np.abs(np.asarray(want)) * 2.0 ** -8 + 1e-30
        assert np.all(np.abs(got - want) <= ulp)
        assert np.array_equal(vo[row], vn[i])
    # position 0 rotates by nothing: the row is k_norm(k) rounded once
    assert np.array_equal(ko[3 * ps], orc.f64_to_bf16_bits(orc.k_norm(kn[0:1], w, eps))[0])


ALL_CHECKS += [check_k_norm_closed_forms, check_k_norm_invariants, check_append_rope_k_norm]


# ---------------------------------------------------- paged (chunked) prefill --

def _chunk_case(orc, prefix_lens, chunk_lens, page_size, seed, hq=8, hkv=2, shuffle=True,
                n_pad=0):
    from paged_kv_gqa_pkv_gb300 import workloads as W
    c = W.chunked_prefill(seed, prefix_lens=prefix_lens, chunk_lens=chunk_lens, hq=hq, hkv=hkv,
                          page_size=page_size, shuffle=shuffle, n_pad=n_pad)
    kp, vp, bad = orc.append(_bits(c.k_pool), _bits(c.v_pool), c.page_table.numpy(),
                             _bits(c.k_new), _bits(c.v_new), c.batch_idx.numpy(),
                             c.input_pos.numpy(), c.page_size)
    assert bad == []
    return c, kp, vp


def check_paged_prefill_against_library(orc):
    """One sequence with a 37-token prefix and a 29-token chunk: the chunk's
    queries against the library's attention over the whole dense sequence,
    masked by position."""
    c, kp, vp = _chunk_case(orc, [37], [29], 16, 73, shuffle=False)
    out, lse, bad = orc.paged_prefill_attention(_bits(c.q), kp, vp, c.page_table.numpy(),
                                                c.batch_idx.numpy(), c.input_pos.numpy(),
                                                c.page_size, c.scale)
    assert bad == []
    n = 37 + 29
    rows = [int(c.page_table[1, t // 16]) * 16 + t % 16 for t in range(n)]
    K = torch.from_numpy(orc.bf16_bits_to_f64(kp[rows])).permute(1, 0, 2)     # [Hkv, n, D]
    V = torch.from_numpy(orc.bf16_bits_to_f64(vp[rows])).permute(1, 0, 2)
    Q = torch.from_numpy(orc.bf16_bits_to_f64(_bits(c.q))).permute(1, 0, 2)   # [Hq, 29, D]
    pos = c.input_pos.numpy()
    mask = torch.from_numpy(np.arange(n)[None, :] <= pos[:, None])
    ref_o, ref_l = _sdpa_with_probe(Q, K, V, mask)
    assert np.allclose(out, ref_o.permute(1, 0, 2).numpy(), rtol=0, atol=1e-12)
    assert np.allclose(lse, ref_l.permute(1, 0).numpy(), rtol=0, atol=1e-10)


def check_paged_prefill_reduces_to_packed_prefill(orc):
    """Empty prefixes, chunks appended to the pages: exactly the packed
    document-causal prefill over the same tokens."""
    c, kp, vp = _chunk_case(orc, [0, 0, 0], [20, 1, 45], 16, 79, shuffle=False)
    out, lse, bad = orc.paged_prefill_attention(_bits(c.q), kp, vp, c.page_table.numpy(),
                                                c.batch_idx.numpy(), c.input_pos.numpy(),
                                                c.page_size, c.scale)
    ref_o, ref_l = orc.prefill_attention(_bits(c.q), _bits(c.k_new), _bits(c.v_new),
                                         c.batch_idx.numpy(), c.input_pos.numpy(), c.scale)
    assert bad == []
    assert np.allclose(out, ref_o, rtol=0, atol=1e-12)
    assert np.allclose(lse, ref_l, rtol=0, atol=1e-12)


def check_paged_prefill_chunking_invariance(orc):
    """A 70-token sequence in one chunk, or as chunks of 30 then 40 (the
    first appended before the second is attended): the same results."""
    from paged_kv_gqa_pkv_gb300 import workloads as W
    whole, kp, vp = _chunk_case(orc, [0], [70], 16, 83, shuffle=False)
    o_all, l_all, _ = orc.paged_prefill_attention(_bits(whole.q), kp, vp,
                                                  whole.page_table.numpy(),
                                                  whole.batch_idx.numpy(),
                                                  whole.input_pos.numpy(), 16, whole.scale)
    # chunk 2 of 40 tokens over a 30-token prefix: the same pools (the
    # prefix's K/V are the first chunk's), queries 30..69
    sel = np.arange(30, 70)
    o2, l2, bad = orc.paged_prefill_attention(_bits(whole.q)[sel], kp, vp,
                                              whole.page_table.numpy(),
                                              whole.batch_idx.numpy()[sel],
                                              whole.input_pos.numpy()[sel], 16, whole.scale)
    assert bad == []
    assert np.array_equal(o2, o_all[sel]) and np.array_equal(l2, l_all[sel])


def check_paged_prefill_one_token_is_decode(orc):
    """A chunk of one token per sequence is a decode step."""
    c, kp, vp = _chunk_case(orc, [5, 0, 40, 17], [1, 1, 1, 1], 16, 89)
    out, lse, bad = orc.paged_prefill_attention(_bits(c.q), kp, vp, c.page_table.numpy(),
                                                c.batch_idx.numpy(), c.input_pos.numpy(),
                                                c.page_size, c.scale)
    d_o, d_l, d_bad = orc.decode_attention(_bits(c.q), kp, vp, c.page_table.numpy(),
                                           c.batch_idx.numpy(), c.input_pos.numpy() + 1,
                                           c.page_size, c.scale)
    assert bad == [] and d_bad == []
    assert np.array_equal(out, d_o) and np.array_equal(lse, d_l)


def check_paged_prefill_order_and_edges(orc):
    """Shuffling the packed order permutes the results; padding tokens give
    0 / -inf; an unreserved page inside a token's keys makes it a bad row."""
    c, kp, vp = _chunk_case(orc, [10, 33, 0], [7, 12, 19], 16, 97, shuffle=True, n_pad=3)
    args = (kp, vp, c.page_table.numpy())
    out, lse, bad = orc.paged_prefill_attention(_bits(c.q), *args, c.batch_idx.numpy(),
                                                c.input_pos.numpy(), 16, c.scale)
    assert bad == []
    perm = np.random.default_rng(7).permutation(c.n_tokens)
    o_p, l_p, _ = orc.paged_prefill_attention(_bits(c.q)[perm], *args, c.batch_idx.numpy()[perm],
                                              c.input_pos.numpy()[perm], 16, c.scale)
    assert np.array_equal(o_p, out[perm]) and np.array_equal(l_p, lse[perm])
    pad = c.batch_idx.numpy() == 0
    assert pad.sum() == 3 and np.all(out[pad] == 0) and np.all(np.isneginf(lse[pad]))
    table = c.page_table.numpy().copy()
    table[2, 1] = -1                    # slot 2 positions 16..31: its prefix of 33
    _, _, bad2 = orc.paged_prefill_attention(_bits(c.q), kp, vp, table, c.batch_idx.numpy(),
                                             c.input_pos.numpy(), 16, c.scale)
    assert sorted(bad2) == sorted(np.nonzero(c.batch_idx.numpy() == 2)[0].tolist())


ALL_CHECKS += [check_paged_prefill_against_library, check_paged_prefill_reduces_to_packed_prefill,
               check_paged_prefill_chunking_invariance, check_paged_prefill_one_token_is_decode,
               check_paged_prefill_order_and_edges]
