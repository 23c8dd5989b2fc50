"""Plain, slow, float64 CPU oracle for attention over a paged KV cache.

TEST INFRASTRUCTURE ONLY: used by ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py``. The product path never imports it.

What the method computes (sources are the pages' own titles and sections):

* The KV cache of one layer is one contiguous physical pool per tensor (K and
  V), addressed by a page table that maps (logical batch slot, logical block)
  to a physical page; batch slot 0 and page 0 are reserved as no-op padding
  ("flex_paged_attention.py" commit log, section "Why this works", items 1
  and 3). Pools here are token-major ``[num_pages*page_size, H_kv, D]``.
* A new token's K/V row is written to
  ``page_table[b, pos // page_size] * page_size + pos % page_size``; a write
  through an unreserved entry is an error ("flex_paged_attention.py" commit
  log, the paragraph on ``k_cache[addr] = k_val`` under "Files";
  "qwen3_flex_inference.py", ``capture_decode_cudagraph``).
* Decode: one query token per sequence attends to logical keys
  ``kv_idx <= input_pos`` of its own batch slot ("qwen3_flex_inference.py",
  ``_decode_block_mask``, the ``causal_offset`` mask), with grouped-query
  heads ("qwen3_flex_inference.py", attention ``forward``, ``enable_gqa``).
  ``seq_lens[b] = input_pos[b] + 1`` keys are attended.
* Prefill: all prompts are packed into one sequence and token i may attend
  token j iff both carry the same (non-zero) batch slot and
  ``input_pos[j] <= input_pos[i]`` ("qwen3_flex_inference.py", ``_prefill``,
  document-causal mask).
* A row whose keys are all masked returns zeros, not NaN
  ("flex_vs_vllm.md", "What broke correctness and had to be dropped",
  ROWS_GUARANTEED_SAFE).

* Before the cache write, k goes through the model's per-head ``k_norm`` and
  the rotate-half rotary embedding ("qwen3_flex_inference.py", attention
  ``forward`` and ``_apply_rotary``).

Readings where the pages are silent (each is listed in the design notes):
the LSE is the natural log of sum_t exp(scale * q.k_t); the q head h reads
kv head h // (H_q / H_kv); rows of batch slot 0 or with no keys give
out = 0 and lse = -inf; an append whose batch slot is 0 is skipped;
``k_norm`` is the Qwen3 family's RMSNorm over the head dims (the pages name
the module, not its formula), and normalisation and rotation are exact with
one rounding to bf16 at the end.

Representation: bf16 tensors are numpy ``uint16`` arrays of raw bf16 bit
patterns; every arithmetic step is float64. Results are float64; callers that
compare against bf16 hardware output round with ``f64_to_bf16_bits``.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(closed forms, library special cases, invariants, brute force) and the pins'
power is checked by ``tests/test_oracle_mutations.py``.
"""

from __future__ import annotations

import math

import numpy as np


# --------------------------------------------------------------------------
# bf16 <-> float64 (exact widening; round-to-nearest-even narrowing)
# --------------------------------------------------------------------------

def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact value of bf16 bit patterns: bf16 is the top half of an IEEE
    binary32, so shifting the 16 bits into the high half gives the float32
    with the same value, which float64 holds exactly."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    with np.errstate(invalid="ignore"):   # NaN patterns stay NaN
        return b.view(np.float32).astype(np.float64)


def f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float64 values to bf16 (8 significant bits, 8-bit exponent) with
    round-to-nearest, ties-to-even, in one step from float64 (no detour
    through float32, so no double rounding). Returns uint16 bit patterns."""
    x = np.asarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.float64)
    finite = np.isfinite(x)
    xf = np.where(finite, x, 0.0)
    # Quantum of the bf16 grid at |x|: 2^(e-8) for normal numbers with
    # |x| in [2^(e-1), 2^e); fixed at 2^-133 in the subnormal range.
    _, e = np.frexp(xf)
    e = np.maximum(e, -125)           # bf16 min normal is 2^-126 = 2^(-125-1)
    quantum = np.ldexp(1.0, e - 8)
    r = np.rint(xf / quantum) * quantum  # np.rint rounds half to even
    max_bf16 = float.fromhex("0x1.fep127")
    r = np.where(np.abs(r) > max_bf16, np.copysign(np.inf, xf), r)
    out[...] = np.where(finite, r, x)
    f32 = out.astype(np.float32)        # exact: every value is on the bf16 grid
    bits = (f32.view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    # NaN stays NaN (canonical quiet NaN)
    bits = np.where(np.isnan(x), np.uint16(0x7FC0), bits)
    return bits


# --------------------------------------------------------------------------
# Page-table addressing
# --------------------------------------------------------------------------

def physical_slot(page_table: np.ndarray, slot: int, pos: int, page_size: int,
                  num_pages: int):
    """Physical row of logical position ``pos`` of batch slot ``slot``:
    ``page_table[slot, pos // page_size] * page_size + pos % page_size``.
    Returns None when the address cannot be formed: slot or block outside the
    table, or a page entry that is not a reserved page in ``[0, num_pages)``
    (-1 marks "not reserved")."""
    if slot < 0 or slot >= page_table.shape[0] or pos < 0:
        return None
    block = pos // page_size
    if block >= page_table.shape[1]:
        return None
    page = int(page_table[slot, block])
    if page < 0 or page >= num_pages:
        return None
    return page * page_size + pos % page_size


# --------------------------------------------------------------------------
# KV append
# --------------------------------------------------------------------------

def append(k_pool: np.ndarray, v_pool: np.ndarray, page_table: np.ndarray,
           k_new: np.ndarray, v_new: np.ndarray, batch_idx: np.ndarray,
           input_pos: np.ndarray, page_size: int):
    """Write each new token's K and V row into the pools through the page
    table (the cache ``update`` step before attention; "qwen3_flex_inference.py",
    attention ``forward``, "Write to paged KV cache").

    Token i with slot ``batch_idx[i]`` and position ``input_pos[i]`` copies the
    raw bf16 bytes of ``k_new[i]`` / ``v_new[i]`` (shape ``[H_kv, D]``) to the
    pool row given by ``physical_slot``. Slot 0 is the padding slot and is not
    written. A token whose address cannot be formed is not written and is
    reported.

    Returns ``(k_pool_out, v_pool_out, bad_tokens)`` where the pools are new
    arrays and ``bad_tokens`` lists the indices of tokens that were skipped for
    an invalid address.
    """
    k_out = np.array(k_pool, dtype=np.uint16, copy=True)
    v_out = np.array(v_pool, dtype=np.uint16, copy=True)
    num_pages = k_out.shape[0] // page_size
    bad = []
    for i in range(len(batch_idx)):
        slot = int(batch_idx[i])
        if slot == 0:
            continue
        row = physical_slot(page_table, slot, int(input_pos[i]), page_size,
                            num_pages)
        if row is None:
            bad.append(i)
            continue
        k_out[row] = k_new[i]
        v_out[row] = v_new[i]
    return k_out, v_out, bad


def k_norm(x: np.ndarray, weight: np.ndarray, eps: float) -> np.ndarray:
    """Per-head RMS normalisation of K, the step the model applies to each
    head of k just before the rotary embedding ("qwen3_flex_inference.py",
    attention ``forward``: ``k = self.k_norm(self.k_proj(...).view(...,
    head_dim))``, then ``_apply_rotary``). The pages name the module only; its
    formula is the Qwen3 family's RMSNorm over the head dims with a learned
    per-dim weight:
    ``out[d] = weight[d] * x[d] / sqrt(mean over d' of x[d']**2 + eps)``.

    ``x`` is bf16 bits ``[N, H, D]``, ``weight`` ``[D]`` (any float type).
    Returns float64, unrounded: the rotation that follows works on the exact
    value and the result is rounded to bf16 once, at the end.
    """
    xf = bf16_bits_to_f64(x)
    w = np.asarray(weight, dtype=np.float64)
    ms = np.mean(xf * xf, axis=-1, keepdims=True)
    return w * (xf / np.sqrt(ms + float(eps)))


def rope(x: np.ndarray, positions: np.ndarray, cos_table: np.ndarray,
         sin_table: np.ndarray) -> np.ndarray:
    """Rotary position embedding in the rotate-half form the pages apply to q
    and k before the cache write ("qwen3_flex_inference.py", ``_apply_rotary``:
    ``x * cos + rotate_half(x) * sin`` with ``rotate_half(x) = cat(-x2, x1)``).

    ``x`` is bf16 bits ``[N, H, D]``; token i uses row ``positions[i]`` of the
    tables ``cos_table``/``sin_table`` (``[L, D/2]``, the half-width table: the
    full-width cos/sin repeat it for the second half). For each head, with
    ``x1 = x[:D/2]``, ``x2 = x[D/2:]``, ``c = cos[p]``, ``s = sin[p]``:
    ``out1 = x1*c - x2*s`` and ``out2 = x2*c + x1*s``. Returns float64.
    """
    return rope_f64(bf16_bits_to_f64(x), positions, cos_table, sin_table)


def rope_f64(xf: np.ndarray, positions: np.ndarray, cos_table: np.ndarray,
             sin_table: np.ndarray) -> np.ndarray:
    """``rope`` on float64 input ``[N, H, D]`` (e.g. the output of ``k_norm``)."""
    half = xf.shape[-1] // 2
    c = np.asarray(cos_table, dtype=np.float64)[np.asarray(positions, dtype=np.int64)]
    s = np.asarray(sin_table, dtype=np.float64)[np.asarray(positions, dtype=np.int64)]
    c = c[:, None, :]
    s = s[:, None, :]
    x1, x2 = xf[..., :half], xf[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def append_rope(k_pool: np.ndarray, v_pool: np.ndarray, page_table: np.ndarray,
                k_new: np.ndarray, v_new: np.ndarray, batch_idx: np.ndarray,
                input_pos: np.ndarray, page_size: int, cos_table: np.ndarray,
                sin_table: np.ndarray, k_norm_weight=None, k_norm_eps: float = 1e-6):
    """KV append with the rotary embedding applied to K first: K rows are
    ``rope(k_new)`` rounded to bf16 (nearest even), V rows are copied as
    they are. With ``k_norm_weight`` given, K is first normalised per head
    (``k_norm``) and the rotation acts on the exact normalised value: K rows
    are ``rope(k_norm(k_new))`` rounded to bf16 once. A token whose position
    has no table row is reported and not written. Returns
    ``(k_pool_out, v_pool_out, bad_tokens)``."""
    n = len(batch_idx)
    pos = np.asarray(input_pos, dtype=np.int64)
    in_table = (pos >= 0) & (pos < len(cos_table))
    k_rot = np.array(k_new, dtype=np.uint16, copy=True)
    if in_table.any():
        if k_norm_weight is None:
            kf = bf16_bits_to_f64(k_new[in_table])
        else:
            kf = k_norm(k_new[in_table], k_norm_weight, k_norm_eps)
        k_rot[in_table] = f64_to_bf16_bits(rope_f64(kf, pos[in_table], cos_table, sin_table))
    keep = [i for i in range(n) if in_table[i] or int(batch_idx[i]) == 0]
    k_out, v_out, bad = append(k_pool, v_pool, page_table, k_rot[keep], v_new[keep],
                               np.asarray(batch_idx)[keep], pos[keep], page_size)
    bad = sorted([keep[i] for i in bad] +
                 [i for i in range(n) if not in_table[i] and int(batch_idx[i]) != 0])
    return k_out, v_out, bad


# --------------------------------------------------------------------------
# Attention
# --------------------------------------------------------------------------

def gather_logical(pool: np.ndarray, page_table: np.ndarray, slot: int, n: int,
                   page_size: int):
    """Logical keys 0..n-1 of batch slot ``slot`` read through the page table,
    as float64 ``[n, H_kv, D]``. Returns None if any address within the first
    n positions cannot be formed (the result of such a row is unspecified)."""
    num_pages = pool.shape[0] // page_size
    rows = []
    for t in range(n):
        r = physical_slot(page_table, slot, t, page_size, num_pages)
        if r is None:
            return None
        rows.append(r)
    return bf16_bits_to_f64(pool[np.asarray(rows, dtype=np.int64)])


def attend(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float):
    """Exact softmax attention of query heads ``q`` (float64 ``[H_q, D]``) over
    keys ``K`` and values ``V`` (float64 ``[n, H_kv, D]``).

    Query head h reads kv head ``h // (H_q // H_kv)`` (grouped-query heads,
    consecutive q heads share one kv head). For each head:
    ``s_t = scale * sum_d q[h, d] K[t, kvh, d]``; ``lse = log sum_t exp(s_t)``
    (evaluated as ``m + log sum_t exp(s_t - m)`` with ``m = max_t s_t``);
    ``out = sum_t exp(s_t - lse) V[t, kvh]``. With no keys: out = 0 and
    lse = -inf.

    Returns ``(out [H_q, D], lse [H_q])`` in float64.
    """
    hq, d = q.shape
    n = K.shape[0]
    out = np.zeros((hq, d), dtype=np.float64)
    lse = np.full((hq,), -np.inf, dtype=np.float64)
    if n == 0:
        return out, lse
    hkv = K.shape[1]
    group = hq // hkv
    for h in range(hq):
        kvh = h // group
        s = scale * (K[:, kvh, :] @ q[h])
        m = np.max(s)
        lse[h] = m + math.log(np.sum(np.exp(s - m)))
        p = np.exp(s - lse[h])
        out[h] = p @ V[:, kvh, :]
    return out, lse


def decode_attention(q: np.ndarray, k_pool: np.ndarray, v_pool: np.ndarray,
                     page_table: np.ndarray, batch_idx: np.ndarray,
                     seq_lens: np.ndarray, page_size: int, scale: float,
                     rows=None):
    """GQA decode over the paged cache: row b (one query token, ``q[b]`` of
    shape ``[H_q, D]`` bf16 bits) attends the first ``seq_lens[b]`` logical
    keys of batch slot ``batch_idx[b]`` ("qwen3_flex_inference.py",
    ``_decode_block_mask`` / ``causal_offset``: keys ``kv_idx <= input_pos``).
    Rows with slot 0 (padding) or no keys give out 0, lse -inf.

    ``rows`` optionally restricts the computation to a subset of rows (the
    others are left NaN). Rows whose keys cannot all be addressed are NaN and
    listed in the returned ``bad_rows``.

    Returns ``(out [B, H_q, D], lse [B, H_q], bad_rows)`` in float64.
    """
    B, hq, d = q.shape
    out = np.full((B, hq, d), np.nan)
    lse = np.full((B, hq), np.nan)
    bad = []
    for b in (range(B) if rows is None else rows):
        slot = int(batch_idx[b])
        n = int(seq_lens[b])
        if slot == 0 or n <= 0:
            out[b] = 0.0
            lse[b] = -np.inf
            continue
        K = gather_logical(k_pool, page_table, slot, n, page_size)
        V = gather_logical(v_pool, page_table, slot, n, page_size)
        if K is None or V is None:
            bad.append(b)
            continue
        out[b], lse[b] = attend(bf16_bits_to_f64(q[b]), K, V, scale)
    return out, lse, bad


def paged_prefill_attention(q: np.ndarray, k_pool: np.ndarray, v_pool: np.ndarray,
                            page_table: np.ndarray, batch_idx: np.ndarray,
                            input_pos: np.ndarray, page_size: int, scale: float, rows=None):
    """Chunked prefill over the paged cache: packed query token i (``q[i]``,
    ``[H_q, D]`` bf16 bits) attends the logical keys ``0..input_pos[i]`` of its
    batch slot ``batch_idx[i]``, read through the page table, the token's own
    chunk included (its K/V were appended first). This is the step the pages
    leave on the table: prefill that reads its earlier context from the pages,
    so that prefill chunks and decode tokens can share one pass
    ("flex_vs_vllm.md", "What's left on the table", chunked prefill; the
    prefill there reads the packed fresh k/v instead,
    "qwen3_flex_inference.py", ``_prefill``). The rule per token is the
    decode rule (``_decode_block_mask``, ``causal_offset``: ``kv_idx <=
    input_pos``); tokens need no particular order or packing.

    Tokens of slot 0 give out 0, lse -inf. Tokens whose keys cannot all be
    addressed (a position past the table, an unreserved entry) are NaN and
    listed in the returned ``bad_rows``. ``rows`` optionally restricts the
    computation to some tokens (the others stay NaN).

    Returns ``(out [T, H_q, D], lse [T, H_q], bad_rows)`` in float64.
    """
    T, hq, d = q.shape
    out = np.full((T, hq, d), np.nan)
    lse = np.full((T, hq), np.nan)
    bad = []
    for i in (range(T) if rows is None else rows):
        slot = int(batch_idx[i])
        if slot == 0:
            out[i] = 0.0
            lse[i] = -np.inf
            continue
        n = int(input_pos[i]) + 1
        if n <= 0:
            bad.append(i)
            continue
        K = gather_logical(k_pool, page_table, slot, n, page_size)
        V = gather_logical(v_pool, page_table, slot, n, page_size)
        if K is None or V is None:
            bad.append(i)
            continue
        out[i], lse[i] = attend(bf16_bits_to_f64(q[i]), K, V, scale)
    return out, lse, bad


def prefill_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray,
                      batch_idx: np.ndarray, input_pos: np.ndarray,
                      scale: float, rows=None):
    """Packed document-causal prefill ("qwen3_flex_inference.py", ``_prefill``).

    ``q`` is ``[T, H_q, D]``, ``k``/``v`` are ``[T, H_kv, D]`` (bf16 bits) for T
    packed tokens. Token i may attend token j iff
    ``batch_idx[j] == batch_idx[i] != 0`` and ``input_pos[j] <= input_pos[i]``.
    Attention reads the packed fresh k/v, not the pages. Tokens of slot 0
    (padding) give out 0, lse -inf.

    Tokens are grouped by batch slot (pairs across slots are masked by the
    definition) and each query row is attended with ``attend`` over its allowed
    keys in packed order. ``rows`` optionally restricts the query rows
    computed (others NaN).

    Returns ``(out [T, H_q, D], lse [T, H_q])`` in float64.
    """
    T, hq, d = q.shape
    out = np.full((T, hq, d), np.nan)
    lse = np.full((T, hq), np.nan)
    want = np.zeros(T, dtype=bool)
    if rows is None:
        want[:] = True
    else:
        want[np.asarray(rows, dtype=np.int64)] = True
    bidx = np.asarray(batch_idx, dtype=np.int64)
    pos = np.asarray(input_pos, dtype=np.int64)
    qf = bf16_bits_to_f64(q)
    kf = bf16_bits_to_f64(k)
    vf = bf16_bits_to_f64(v)
    pad = want & (bidx == 0)
    out[pad] = 0.0
    lse[pad] = -np.inf
    for slot in np.unique(bidx[want & (bidx != 0)]):
        members = np.nonzero(bidx == slot)[0]
        for i in members:
            if not want[i]:
                continue
            keys = members[pos[members] <= pos[i]]
            out[i], lse[i] = attend(qf[i], kf[keys], vf[keys], scale)
    return out, lse
