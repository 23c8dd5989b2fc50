"""Power of the oracle pins: each test plants one plausible mistake in a copy
of an oracle function (on the CPU) and requires that some pin fails.

A mistake that no pin catches would mean the pins cannot vouch for the
oracle, so every planted mistake here must be caught."""

import math

import numpy as np
import pytest

import oracle.paged_attention as orc
from tests import oracle_pins


def _caught(monkeypatch, name, fn):
    monkeypatch.setattr(orc, name, fn)
    failures = []
    for check in oracle_pins.ALL_CHECKS:
        try:
            check(orc)
        except Exception as e:  # noqa: BLE001 - any failure counts as caught
            failures.append((check.__name__, type(e).__name__))
    return failures


def _attend_variant(head_map=None, use_scale=True, add_max=True, swap_kv=False,
                    drop_last=False):
    def attend(q, K, V, scale):
        hq, d = q.shape
        n = K.shape[0] - (1 if drop_last and K.shape[0] > 1 else 0)
        out = np.zeros((hq, d))
        lse = np.full((hq,), -np.inf)
        if n == 0:
            return out, lse
        hkv = K.shape[1]
        g = hq // hkv
        for h in range(hq):
            kvh = head_map(h, g, hkv) if head_map else h // g
            KK, VV = (V, K) if swap_kv else (K, V)
            s = (scale if use_scale else 1.0) * (KK[:n, kvh, :] @ q[h])
            m = np.max(s)
            lse[h] = (m if add_max else 0.0) + math.log(np.sum(np.exp(s - m)))
            p = np.exp(s - (m + math.log(np.sum(np.exp(s - m)))))
            out[h] = p @ VV[:n, kvh, :]
        return out, lse
    return attend


MUTANTS = {
    "gqa_head_modulo": ("attend", _attend_variant(head_map=lambda h, g, hkv: h % hkv)),
    "no_scale": ("attend", _attend_variant(use_scale=False)),
    "lse_without_max": ("attend", _attend_variant(add_max=False)),
    "k_v_swapped": ("attend", _attend_variant(swap_kv=True)),
    "last_key_dropped": ("attend", _attend_variant(drop_last=True)),
}


def _physical_slot_swapped(page_table, slot, pos, page_size, num_pages):
    if slot < 0 or slot >= page_table.shape[0] or pos < 0:
        return None
    block = pos % page_size                 # planted: block and offset swapped
    if block >= page_table.shape[1]:
        return None
    page = int(page_table[slot, block])
    if page < 0 or page >= num_pages:
        return None
    return page * page_size + pos // page_size


def _physical_slot_no_range_check(page_table, slot, pos, page_size, num_pages):
    page = int(page_table[slot, pos // page_size])
    return page * page_size + pos % page_size   # planted: -1 not rejected


def _append_writes_padding(k_pool, v_pool, page_table, k_new, v_new, batch_idx,
                           input_pos, page_size):
    k_out, v_out = k_pool.copy(), v_pool.copy()
    P = k_out.shape[0] // page_size
    bad = []
    for i in range(len(batch_idx)):
        r = orc.physical_slot(page_table, int(batch_idx[i]), int(input_pos[i]),
                              page_size, P)
        if r is None:
            if int(batch_idx[i]) != 0:
                bad.append(i)
            continue
        k_out[r] = k_new[i]             # planted: slot 0 rows are written too
        v_out[r] = v_new[i]
    return k_out, v_out, bad


_real_decode = orc.decode_attention
_real_prefill = orc.prefill_attention
_real_round = orc.f64_to_bf16_bits


def _decode_off_by_one(q, kp, vp, table, bidx, lens, ps, scale, rows=None):
    return _real_decode(q, kp, vp, table, bidx, np.asarray(lens) - 1, ps, scale, rows)


def _decode_nan_on_empty(q, kp, vp, table, bidx, lens, ps, scale, rows=None):
    out, lse, bad = _real_decode(q, kp, vp, table, bidx, lens, ps, scale, rows)
    empty = (np.asarray(bidx) == 0) | (np.asarray(lens) <= 0)
    out[empty] = np.nan                  # planted: empty rows give NaN
    return out, lse, bad


def _decode_ignores_slot(q, kp, vp, table, bidx, lens, ps, scale, rows=None):
    # planted: row b reads slot b+1 instead of batch_idx[b]
    return _real_decode(q, kp, vp, table, np.arange(1, len(bidx) + 1), lens,
                        ps, scale, rows)


def _prefill_strict_causal(q, k, v, bidx, pos, scale, rows=None):
    # planted: keys with pos < pos_i only (the diagonal is dropped); done by
    # shifting every query position down by one within its document
    return _real_prefill(q, k, v, bidx, np.asarray(pos), scale, rows) \
        if False else _strict(q, k, v, bidx, pos, scale)


def _strict(q, k, v, bidx, pos, scale):
    T, hq, d = q.shape
    out = np.zeros((T, hq, d))
    lse = np.full((T, hq), -np.inf)
    qf, kf, vf = (orc.bf16_bits_to_f64(x) for x in (q, k, v))
    for i in range(T):
        if bidx[i] == 0:
            continue
        keys = np.nonzero((bidx == bidx[i]) & (pos < pos[i]))[0]
        out[i], lse[i] = orc.attend(qf[i], kf[keys], vf[keys], scale)
    return out, lse


def _prefill_across_documents(q, k, v, bidx, pos, scale, rows=None):
    # planted: the document boundary is ignored (plain causal over the packing)
    T = len(bidx)
    return _real_prefill(q, k, v, np.where(np.asarray(bidx) != 0, 1, 0),
                         np.arange(T), scale, rows)


def _round_truncate(x):
    x = np.asarray(x, dtype=np.float64)
    return (x.astype(np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def _round_via_f32(x):
    x = np.asarray(x, dtype=np.float64)
    import torch
    t = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _rope_sign_flipped(x, positions, cos_table, sin_table):
    xf = orc.bf16_bits_to_f64(x)
    half = xf.shape[-1] // 2
    c = np.asarray(cos_table, dtype=np.float64)[np.asarray(positions)][:, None, :]
    s_ = np.asarray(sin_table, dtype=np.float64)[np.asarray(positions)][:, None, :]
    x1, x2 = xf[..., :half], xf[..., half:]
    return np.concatenate([x1 * c + x2 * s_, x2 * c - x1 * s_], axis=-1)   # planted: sign


def _rope_interleaved(x, positions, cos_table, sin_table):
    xf = orc.bf16_bits_to_f64(x)
    c = np.asarray(cos_table, dtype=np.float64)[np.asarray(positions)][:, None, :]
    s_ = np.asarray(sin_table, dtype=np.float64)[np.asarray(positions)][:, None, :]
    x1, x2 = xf[..., 0::2], xf[..., 1::2]          # planted: pairs (2i, 2i+1)
    out = np.empty_like(xf)
    out[..., 0::2] = x1 * c - x2 * s_
    out[..., 1::2] = x2 * c + x1 * s_
    return out


_real_append_rope = orc.append_rope


def _append_rope_on_v(k_pool, v_pool, table, k_new, v_new, bidx, pos, ps, cos_t, sin_t):
    # planted: the rotation is applied to V as well
    ok = (np.asarray(pos) >= 0) & (np.asarray(pos) < len(cos_t))
    v_rot = np.array(v_new, copy=True)
    v_rot[ok] = orc.f64_to_bf16_bits(orc.rope(v_new[ok], np.asarray(pos)[ok], cos_t, sin_t))
    return _real_append_rope(k_pool, v_pool, table, k_new, v_rot, bidx, pos, ps, cos_t, sin_t)


def _k_norm_sum(x, weight, eps):
    xf = orc.bf16_bits_to_f64(x)
    return np.asarray(weight, dtype=np.float64) * xf / np.sqrt(
        np.sum(xf * xf, axis=-1, keepdims=True) + eps)            # planted: sum, not mean


def _k_norm_no_eps(x, weight, eps):
    xf = orc.bf16_bits_to_f64(x)
    ms = np.mean(xf * xf, axis=-1, keepdims=True)
    with np.errstate(invalid="ignore", divide="ignore"):
        return np.asarray(weight, dtype=np.float64) * xf / np.sqrt(ms)   # planted: eps dropped


def _k_norm_weight_reversed(x, weight, eps):
    xf = orc.bf16_bits_to_f64(x)
    ms = np.mean(xf * xf, axis=-1, keepdims=True)
    return np.asarray(weight, dtype=np.float64)[::-1] * xf / np.sqrt(ms + eps)   # planted


def _append_rope_norm_after(k_pool, v_pool, table, k_new, v_new, bidx, pos, ps, cos_t, sin_t,
                            k_norm_weight=None, k_norm_eps=1e-6):
    # planted: the rotation first, the normalisation (and its weight) after it
    if k_norm_weight is None:
        return _real_append_rope(k_pool, v_pool, table, k_new, v_new, bidx, pos, ps, cos_t,
                                 sin_t)
    posa = np.asarray(pos, dtype=np.int64)
    ok = (posa >= 0) & (posa < len(cos_t))
    k2 = np.array(k_new, copy=True)
    r = orc.rope(k_new[ok], posa[ok], cos_t, sin_t)
    ms = np.mean(r * r, axis=-1, keepdims=True)
    k2[ok] = orc.f64_to_bf16_bits(np.asarray(k_norm_weight) * r / np.sqrt(ms + k_norm_eps))
    zero = np.zeros_like(cos_t)
    one = np.ones_like(cos_t)
    return _real_append_rope(k_pool, v_pool, table, k2, v_new, bidx, pos, ps, one, zero)


def _paged_prefill_variant(excl_own=False, slot_of=None, skip_first=False):
    def fn(q, k_pool, v_pool, page_table, batch_idx, input_pos, page_size, scale, rows=None):
        T, hq, d = q.shape
        out = np.full((T, hq, d), np.nan)
        lse = np.full((T, hq), np.nan)
        bad = []
        for i in (range(T) if rows is None else rows):
            slot = int(batch_idx[i]) if slot_of is None else slot_of(batch_idx, i)
            if slot == 0:
                out[i], lse[i] = 0.0, -np.inf
                continue
            n = int(input_pos[i]) + (0 if excl_own else 1)
            K = orc.gather_logical(k_pool, page_table, slot, n, page_size)
            V = orc.gather_logical(v_pool, page_table, slot, n, page_size)
            if K is None or V is None or n <= 0:
                bad.append(i)
                continue
            if skip_first and n > 1:
                K, V = K[1:], V[1:]
            out[i], lse[i] = orc.attend(orc.bf16_bits_to_f64(q[i]), K, V, scale)
        return out, lse, bad
    return fn


MUTANTS.update({
    "paged_prefill_excludes_own_token": ("paged_prefill_attention",
                                         _paged_prefill_variant(excl_own=True)),
    "paged_prefill_first_tokens_slot": ("paged_prefill_attention",
                                        _paged_prefill_variant(
                                            slot_of=lambda b, i: int(b[0]) if int(b[i]) else 0)),
    "paged_prefill_drops_first_key": ("paged_prefill_attention",
                                      _paged_prefill_variant(skip_first=True)),
    "k_norm_sum_not_mean": ("k_norm", _k_norm_sum),
    "k_norm_drops_eps": ("k_norm", _k_norm_no_eps),
    "k_norm_weight_reversed": ("k_norm", _k_norm_weight_reversed),
    "append_rope_norm_after_rotation": ("append_rope", _append_rope_norm_after),
    "rope_sign_flipped": ("rope", _rope_sign_flipped),
    "rope_interleaved_pairs": ("rope", _rope_interleaved),
    "append_rope_rotates_v": ("append_rope", _append_rope_on_v),
    "page_formula_swapped": ("physical_slot", _physical_slot_swapped),
    "unreserved_page_accepted": ("physical_slot", _physical_slot_no_range_check),
    "append_writes_padding_slot": ("append", _append_writes_padding),
    "decode_seq_len_off_by_one": ("decode_attention", _decode_off_by_one),
    "decode_empty_rows_nan": ("decode_attention", _decode_nan_on_empty),
    "decode_ignores_batch_idx": ("decode_attention", _decode_ignores_slot),
    "prefill_strict_causal": ("prefill_attention", _prefill_strict_causal),
    "prefill_ignores_documents": ("prefill_attention", _prefill_across_documents),
    "bf16_truncation": ("f64_to_bf16_bits", _round_truncate),
    "bf16_double_rounding": ("f64_to_bf16_bits", _round_via_f32),
})


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_planted_mistake_is_caught(monkeypatch, mutant):
    name, fn = MUTANTS[mutant]
    failures = _caught(monkeypatch, name, fn)
    assert failures, f"no pin caught the planted mistake {mutant!r}"
