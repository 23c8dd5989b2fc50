"""Seeded random sweeps on the GPU against the float64 oracle: each case
draws its shape (GQA group, page size, batch, length mix, page order,
padding) from a fixed seed, so the sweep covers combinations the hand-written
cases do not, and a failure names the seed that reproduces it."""

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

GROUPS = [(8, 8), (16, 8), (32, 8), (16, 2), (32, 4), (8, 1), (64, 8)]


def _decode_shape(seed):
    rng = np.random.default_rng(1000 + seed)
    hq, hkv = GROUPS[rng.integers(len(GROUPS))]
    ps = int(rng.choice([16, 32, 48, 64, 128, 256]))
    b = int(rng.integers(1, 41))
    # log-uniform lengths up to ~3000 (each row attends at least the token
    # it appends; empty rows come from the padding slots), with tile and
    # page edges
    lens = np.exp(rng.uniform(0, np.log(3000), size=b)).astype(int).tolist()
    for k in rng.choice(b, size=min(b, 3), replace=False):
        lens[k] = int(rng.choice([1, 16, 17, ps, ps + 1]))
    return dict(hq=int(hq), hkv=int(hkv), page_size=ps, lens=lens,
                n_pad=int(rng.integers(0, 4)), permute=bool(rng.integers(2)))


@pytest.mark.parametrize("seed", range(12))
def test_decode_random_shapes(seed):
    s = _decode_shape(seed)
    c = W.custom_decode(seed, s["lens"], hq=s["hq"], hkv=s["hkv"], page_size=s["page_size"],
                        n_pad=s["n_pad"], permute=s["permute"])
    kp, vp, out, lse, err = run_decode_step(c)
    ek, ev, ref_o, ref_l, bad_tok, bad_rows = oracle_decode_step(c)
    assert err == 0 and not bad_tok and not bad_rows, (seed, s)
    assert np.array_equal(bf16_bits(kp), ek) and np.array_equal(bf16_bits(vp), ev), (seed, s)
    assert_attention_close(out, lse, ref_o, ref_l, tag=f"decode seed {seed} {s}")
    # the same step as one fused call gives the same bits
    kpf, vpf = gpu(c.k_pool), gpu(c.v_pool)
    errf = new_dev_err()
    of, lf = binding.pkv_decode_append_attention(
        kpf, vpf, gpu(c.page_table), gpu(c.q), gpu(c.k_new), gpu(c.v_new), gpu(c.batch_idx),
        gpu(c.seq_lens), c.page_size, c.scale, dev_err=errf)
    torch.cuda.synchronize()
    assert int(errf.item()) == 0
    assert torch.equal(kpf.cpu(), kp) and torch.equal(vpf.cpu(), vp)
    assert torch.equal(of.cpu(), out) and torch.equal(lf.cpu(), lse)


@pytest.mark.parametrize("seed", range(6))
def test_packed_prefill_random_packings(seed):
    rng = np.random.default_rng(2000 + seed)
    hq, hkv = GROUPS[rng.integers(len(GROUPS))]
    n_docs = int(rng.integers(1, 13))
    lo = int(rng.integers(1, 64))
    hi = int(rng.integers(lo, 400))
    pc = W.packed_prefill(seed, n_docs=n_docs, lo=lo, hi=hi, hq=int(hq), hkv=int(hkv))
    err = new_dev_err()
    out, lse = binding.pkv_prefill_attention(gpu(pc.q), gpu(pc.k), gpu(pc.v), gpu(pc.batch_idx),
                                             gpu(pc.input_pos), pc.scale, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ro, rl = orc.prefill_attention(bf16_bits(pc.q), bf16_bits(pc.k), bf16_bits(pc.v),
                                   pc.batch_idx.numpy(), pc.input_pos.numpy(), pc.scale)
    assert_attention_close(out.cpu(), lse.cpu(), ro, rl,
                           tag=f"prefill seed {seed} docs {n_docs} U[{lo},{hi}] {hq}/{hkv}")


@pytest.mark.parametrize("seed", range(6))
def test_chunked_prefill_random_steps(seed):
    rng = np.random.default_rng(3000 + seed)
    hq, hkv = GROUPS[rng.integers(len(GROUPS))]
    ps = int(rng.choice([16, 32, 64, 128, 256]))
    n = int(rng.integers(1, 9))
    prefix = [int(x) for x in rng.integers(0, 900, size=n)]
    chunk = [int(rng.choice([1, int(rng.integers(1, 300))])) for _ in range(n)]
    c = W.chunked_prefill(seed, prefix_lens=prefix, chunk_lens=chunk, page_size=ps, hq=int(hq),
                          hkv=int(hkv), n_pad=int(rng.integers(0, 3)),
                          shuffle=bool(rng.integers(2)), permute=bool(rng.integers(2)))
    kp, vp, pt = gpu(c.k_pool), gpu(c.v_pool), gpu(c.page_table)
    bidx, pos = gpu(c.batch_idx), gpu(c.input_pos)
    err = new_dev_err()
    binding.pkv_append(kp, vp, pt, gpu(c.k_new), gpu(c.v_new), bidx, pos, c.page_size,
                       dev_err=err)
    out, lse = binding.pkv_prefill_paged_attention(kp, vp, pt, gpu(c.q), bidx, pos, c.page_size,
                                                   c.scale, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    kb, vb, bad_tok = orc.append(bf16_bits(c.k_pool), bf16_bits(c.v_pool), c.page_table.numpy(),
                                 bf16_bits(c.k_new), bf16_bits(c.v_new), c.batch_idx.numpy(),
                                 c.input_pos.numpy(), c.page_size)
    ro, rl, bad = orc.paged_prefill_attention(bf16_bits(c.q), kb, vb, c.page_table.numpy(),
                                              c.batch_idx.numpy(), c.input_pos.numpy(),
                                              c.page_size, c.scale)
    assert not bad_tok and not bad
    assert np.array_equal(bf16_bits(kp.cpu()), kb) and np.array_equal(bf16_bits(vp.cpu()), vb)
    assert_attention_close(out.cpu(), lse.cpu(), ro, rl,
                           tag=f"chunked seed {seed} ps {ps} prefix {prefix} chunk {chunk}")
