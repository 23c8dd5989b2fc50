"""pkv_append_rope on the GPU against the oracle's append_rope.

Pool bytes the call must not rotate (V rows, untouched rows, skipped tokens)
are compared bit for bit. Rotated K rows come from fp32 arithmetic on the GPU
and float64 in the oracle, both rounded to bf16 with ties to even: they may
differ by one bf16 ulp when the exact value sits within fp32 error of a
rounding boundary, so the bar is at most one ulp anywhere and at least 99.9 %
of elements identical."""

import numpy as np
import pytest
import torch

import oracle.paged_attention as orc
from paged_kv_gqa_pkv_gb300 import binding
from paged_kv_gqa_pkv_gb300 import workloads as W
from paged_kv_gqa_pkv_gb300.workloads import bf16_bits, rope_tables
from tests.parity import assert_attention_close, gpu, new_dev_err

pytestmark = pytest.mark.gpu


def _ulp_gap(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Distance in bf16 ulps between bit patterns (monotone integer map)."""
    def key(x):
        x = x.astype(np.int32)
        return np.where(x & 0x8000, 0x8000 - (x & 0x7FFF), 0x8000 + x)
    return np.abs(key(a) - key(b))


def _run(case, k_new, v_new, bidx, pos, cos_t, sin_t):
    kp, vp = gpu(case.k_pool), gpu(case.v_pool)
    err = new_dev_err()
    binding.pkv_append_rope(kp, vp, gpu(case.page_table), gpu(k_new), gpu(v_new), gpu(bidx),
                            gpu(pos), case.page_size, gpu(cos_t), gpu(sin_t), dev_err=err)
    torch.cuda.synchronize()
    return bf16_bits(kp.cpu()), bf16_bits(vp.cpu()), int(err.item())


def _compare(kb, vb, ek, ev):
    assert np.array_equal(vb, ev), "V rows must be a plain copy"
    gap = _ulp_gap(kb, ek)
    assert gap.max() <= 1, f"K differs by {gap.max()} ulps"
    assert (gap == 0).mean() >= 0.999


@pytest.mark.parametrize("maker", [W.qwen3_b64_decode, W.padded_bucket_decode])
def test_decode_step_append_rope(maker):
    c = maker(0)
    cos_t, sin_t = rope_tables(4096)
    kb, vb, err = _run(c, c.k_new, c.v_new, c.batch_idx, c.input_pos, cos_t, sin_t)
    ek, ev, bad = orc.append_rope(bf16_bits(c.k_pool), bf16_bits(c.v_pool), c.page_table.numpy(),
                                  bf16_bits(c.k_new), bf16_bits(c.v_new), c.batch_idx.numpy(),
                                  c.input_pos.numpy(), c.page_size, cos_t.numpy(), sin_t.numpy())
    assert err == 0 and not bad
    _compare(kb, vb, ek, ev)


def test_prefill_append_rope_full_size():
    c = W.packed_prefill(0)
    cos_t, sin_t = rope_tables(1024)
    kb, vb, err = _run(c, c.k, c.v, c.batch_idx, c.input_pos, cos_t, sin_t)
    ek, ev, bad = orc.append_rope(bf16_bits(c.k_pool), bf16_bits(c.v_pool), c.page_table.numpy(),
                                  bf16_bits(c.k), bf16_bits(c.v), c.batch_idx.numpy(),
                                  c.input_pos.numpy(), c.page_size, cos_t.numpy(), sin_t.numpy())
    assert err == 0 and not bad
    _compare(kb, vb, ek, ev)


def test_positions_past_the_table_are_flagged_and_skipped():
    c = W.tiny_decode(0)
    cos_t, sin_t = rope_tables(100)   # rows with input_pos 100 and 130 have no angles
    kb, vb, err = _run(c, c.k_new, c.v_new, c.batch_idx, c.input_pos, cos_t, sin_t)
    ek, ev, bad = orc.append_rope(bf16_bits(c.k_pool), bf16_bits(c.v_pool), c.page_table.numpy(),
                                  bf16_bits(c.k_new), bf16_bits(c.v_new), c.batch_idx.numpy(),
                                  c.input_pos.numpy(), c.page_size, cos_t.numpy(), sin_t.numpy())
    assert bad == [2, 3] and err & binding.DEV_ERR_BAD_POS
    _compare(kb, vb, ek, ev)


def test_decode_after_rope_append_matches_oracle():
    c = W.qwen3_b64_decode(0, permute=True)
    cos_t, sin_t = rope_tables(2048)
    kp, vp, pt = gpu(c.k_pool), gpu(c.v_pool), gpu(c.page_table)
    bidx, pos, lens = gpu(c.batch_idx), gpu(c.input_pos), gpu(c.seq_lens)
    binding.pkv_append_rope(kp, vp, pt, gpu(c.k_new), gpu(c.v_new), bidx, pos, c.page_size,
                            gpu(cos_t), gpu(sin_t))
    out, lse = binding.pkv_decode_attention(kp, vp, pt, gpu(c.q), bidx, lens, c.page_size, c.scale)
    torch.cuda.synchronize()
    ek, ev, bad = orc.append_rope(bf16_bits(c.k_pool), bf16_bits(c.v_pool), c.page_table.numpy(),
                                  bf16_bits(c.k_new), bf16_bits(c.v_new), c.batch_idx.numpy(),
                                  c.input_pos.numpy(), c.page_size, cos_t.numpy(), sin_t.numpy())
    ro, rl, bad_rows = orc.decode_attention(bf16_bits(c.q), ek, ev, c.page_table.numpy(),
                                            c.batch_idx.numpy(), c.seq_lens.numpy(), c.page_size,
                                            c.scale)
    assert not bad and not bad_rows
    assert_attention_close(out.cpu(), lse.cpu(), ro, rl, tag="decode after rope append")


# ------------------------------------------------------------------ k_norm --
# With k_norm the rotation acts on an fp32 approximation of the normalised
# head, so the products are no longer exact: the bar is the correctly rounded
# value up to fp32-level error. Every element lies within half a bf16 ulp of
# the exact float64 value plus 2^-20 of its head's largest value, and at
# least 99.9 % of elements equal the oracle's rounding.

def _knorm_weight(seed):
    return torch.from_numpy(np.random.default_rng(seed).uniform(0.25, 2.0, 128).astype(np.float32))


def _check_knorm(case, k_new, bidx, pos, cos_t, sin_t, w, eps, kb, vb, ek, ev):
    assert np.array_equal(vb, ev), "V rows must be a plain copy"
    gap = _ulp_gap(kb, ek)
    assert (gap == 0).mean() >= 0.999
    live = [i for i in range(len(bidx)) if int(bidx[i]) != 0]
    exact = orc.rope_f64(orc.k_norm(bf16_bits(k_new)[live], w.numpy(), eps),
                         pos.numpy()[live], cos_t.numpy(), sin_t.numpy())
    num_pages = case.k_pool.shape[0] // case.page_size
    rows = [orc.physical_slot(case.page_table.numpy(), int(bidx[i]), int(pos[i]),
                              case.page_size, num_pages) for i in live]
    got = orc.bf16_bits_to_f64(kb[np.asarray(rows)])
    scale = np.max(np.abs(exact), axis=-1, keepdims=True)
    half_ulp = np.ldexp(1.0, np.frexp(np.abs(exact))[1] - 9)    # half of 2^(e-8)
    assert np.all(np.abs(got - exact) <= half_ulp + scale * 2.0 ** -20)


@pytest.mark.parametrize("maker", [W.qwen3_b64_decode, W.padded_bucket_decode])
def test_decode_step_append_knorm_rope(maker):
    c = maker(0)
    cos_t, sin_t = rope_tables(4096)
    w, eps = _knorm_weight(1), 1e-6
    kp, vp = gpu(c.k_pool), gpu(c.v_pool)
    err = new_dev_err()
    binding.pkv_append_rope(kp, vp, gpu(c.page_table), gpu(c.k_new), gpu(c.v_new),
                            gpu(c.batch_idx), gpu(c.input_pos), c.page_size, gpu(cos_t),
                            gpu(sin_t), k_norm_weight=gpu(w), k_norm_eps=eps, dev_err=err)
    torch.cuda.synchronize()
    kb, vb = bf16_bits(kp.cpu()), bf16_bits(vp.cpu())
    ek, ev, bad = orc.append_rope(bf16_bits(c.k_pool), bf16_bits(c.v_pool), c.page_table.numpy(),
                                  bf16_bits(c.k_new), bf16_bits(c.v_new), c.batch_idx.numpy(),
                                  c.input_pos.numpy(), c.page_size, cos_t.numpy(), sin_t.numpy(),
                                  k_norm_weight=w.numpy(), k_norm_eps=eps)
    assert int(err.item()) == 0 and not bad
    _check_knorm(c, c.k_new, c.batch_idx, c.input_pos, cos_t, sin_t, w, eps, kb, vb, ek, ev)


def test_prefill_append_knorm_rope_full_size():
    c = W.packed_prefill(0)
    cos_t, sin_t = rope_tables(1024)
    w, eps = _knorm_weight(2), 1e-6
    kp, vp = gpu(c.k_pool), gpu(c.v_pool)
    err = new_dev_err()
    binding.pkv_append_rope(kp, vp, gpu(c.page_table), gpu(c.k), gpu(c.v), gpu(c.batch_idx),
                            gpu(c.input_pos), c.page_size, gpu(cos_t), gpu(sin_t),
                            k_norm_weight=gpu(w), k_norm_eps=eps, dev_err=err)
    torch.cuda.synchronize()
    kb, vb = bf16_bits(kp.cpu()), bf16_bits(vp.cpu())
    ek, ev, bad = orc.append_rope(bf16_bits(c.k_pool), bf16_bits(c.v_pool), c.page_table.numpy(),
                                  bf16_bits(c.k), bf16_bits(c.v), c.batch_idx.numpy(),
                                  c.input_pos.numpy(), c.page_size, cos_t.numpy(), sin_t.numpy(),
                                  k_norm_weight=w.numpy(), k_norm_eps=eps)
    assert int(err.item()) == 0 and not bad
    _check_knorm(c, c.k, c.batch_idx, c.input_pos, cos_t, sin_t, w, eps, kb, vb, ek, ev)


def test_knorm_with_large_eps_and_zero_heads():
    """A large eps (it dominates small heads) and heads that are all zero
    (zero out, no NaN), with two kv heads so the 8-lane groups do not fill
    the warp."""
    gen = torch.Generator().manual_seed(71)
    ps, P, hkv = 16, 12, 2
    kp0 = torch.randn((P * ps, hkv, 128), generator=gen).to(torch.bfloat16)
    vp0 = torch.randn((P * ps, hkv, 128), generator=gen).to(torch.bfloat16)
    table = torch.full((4, 4), -1, dtype=torch.int32)
    table[1:, :3] = (torch.randperm(P - 1, generator=gen)[:9] + 1).view(3, 3).int()
    table[0, :] = 0
    bidx = torch.tensor([1, 2, 3, 0, 2], dtype=torch.int32)
    pos = torch.tensor([5, 17, 40, 2, 33], dtype=torch.int32)
    kn = (torch.randn((5, hkv, 128), generator=gen) * 0.01).to(torch.bfloat16)
    kn[2, 1] = 0
    vn = torch.randn((5, hkv, 128), generator=gen).to(torch.bfloat16)
    cos_t, sin_t = rope_tables(64)
    w, eps = _knorm_weight(3), 0.5

    class C:
        pass
    c = C()
    c.k_pool, c.v_pool, c.page_table, c.page_size = kp0, vp0, table, ps
    kp, vp = gpu(kp0), gpu(vp0)
    err = new_dev_err()
    binding.pkv_append_rope(kp, vp, gpu(table), gpu(kn), gpu(vn), gpu(bidx), gpu(pos), ps,
                            gpu(cos_t), gpu(sin_t), k_norm_weight=gpu(w), k_norm_eps=eps,
                            dev_err=err)
    torch.cuda.synchronize()
    kb, vb = bf16_bits(kp.cpu()), bf16_bits(vp.cpu())
    ek, ev, bad = orc.append_rope(bf16_bits(kp0), bf16_bits(vp0), table.numpy(), bf16_bits(kn),
                                  bf16_bits(vn), bidx.numpy(), pos.numpy(), ps, cos_t.numpy(),
                                  sin_t.numpy(), k_norm_weight=w.numpy(), k_norm_eps=eps)
    assert int(err.item()) == 0 and not bad
    _check_knorm(c, kn, bidx, pos, cos_t, sin_t, w, eps, kb, vb, ek, ev)
    assert not np.isnan(orc.bf16_bits_to_f64(kb)).any()
