"""Helpers for comparing the CUDA path (through the C ABI) with the oracle.

Tolerances for attention follow the stated bar: on the bf16 output,
max-abs error <= 2e-2 and mean-abs error <= 2e-3 against the oracle's float64
result rounded to bf16; on the fp32 LSE, abs error <= 1e-3 where finite, and
-inf exactly where the oracle has -inf. Append and addressing are bit-exact.
"""

from __future__ import annotations

import numpy as np
import torch

import oracle.paged_attention as orc
from paged_kv_gqa_pkv_gb300 import binding
from paged_kv_gqa_pkv_gb300.workloads import bf16_bits

OUT_MAX_ABS = 2e-2
OUT_MEAN_ABS = 2e-3
LSE_ABS = 1e-3


def gpu(t: torch.Tensor) -> torch.Tensor:
    return t.to("cuda", non_blocking=False).contiguous()


def new_dev_err() -> torch.Tensor:
    return torch.zeros(1, dtype=torch.int32, device="cuda")


def run_decode_step(case, append: bool = True, dev_err=None):
    """Append the case's new tokens, then decode, on the GPU through the C
    ABI. Returns CPU tensors (k_pool, v_pool, out, lse, dev_err value)."""
    kp, vp = gpu(case.k_pool), gpu(case.v_pool)
    table = gpu(case.page_table)
    bidx, pos, lens = gpu(case.batch_idx), gpu(case.input_pos), gpu(case.seq_lens)
    err = new_dev_err() if dev_err is None else dev_err
    if append:
        binding.pkv_append(kp, vp, table, gpu(case.k_new), gpu(case.v_new), bidx, pos,
                           case.page_size, dev_err=err)
    out, lse = binding.pkv_decode_attention(kp, vp, table, gpu(case.q), bidx, lens,
                                            case.page_size, case.scale, dev_err=err)
    torch.cuda.synchronize()
    return kp.cpu(), vp.cpu(), out.cpu(), lse.cpu(), int(err.item())


def oracle_decode_step(case, append: bool = True, rows=None):
    """The oracle's append then decode on the case. Returns
    (k_bits, v_bits, out_f64, lse_f64, bad_tokens, bad_rows)."""
    kb, vb = bf16_bits(case.k_pool), bf16_bits(case.v_pool)
    table = case.page_table.numpy()
    bad_tok = []
    if append:
        kb, vb, bad_tok = orc.append(kb, vb, table, bf16_bits(case.k_new), bf16_bits(case.v_new),
                                     case.batch_idx.numpy(), case.input_pos.numpy(),
                                     case.page_size)
    out, lse, bad_rows = orc.decode_attention(bf16_bits(case.q), kb, vb, table,
                                              case.batch_idx.numpy(), case.seq_lens.numpy(),
                                              case.page_size, case.scale, rows=rows)
    return kb, vb, out, lse, bad_tok, bad_rows


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.float64).numpy()


def attention_errors(out_gpu: torch.Tensor, lse_gpu: torch.Tensor, out_ref: np.ndarray,
                     lse_ref: np.ndarray, rows=None):
    """(max_abs, mean_abs, lse_max_abs) over `rows` (default all), after
    checking that -inf and NaN patterns agree."""
    o = bf16_to_f64(out_gpu)
    l = lse_gpu.to(torch.float64).numpy()
    ref_o = orc.bf16_bits_to_f64(orc.f64_to_bf16_bits(out_ref))
    if rows is not None:
        o, l, ref_o, lse_ref = o[rows], l[rows], ref_o[rows], lse_ref[rows]
    assert not np.isnan(o).any(), "GPU output has NaN"
    assert not np.isnan(l).any(), "GPU lse has NaN"
    assert not np.isnan(ref_o).any() and not np.isnan(lse_ref).any(), "oracle rows missing"
    ninf_ref = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(l), ninf_ref), "-inf LSE rows differ"
    assert np.all(o[ninf_ref] == 0.0), "rows with no keys must be exactly 0"
    err = np.abs(o - ref_o)
    fin = ~ninf_ref
    lse_err = np.abs(l[fin] - lse_ref[fin]).max() if fin.any() else 0.0
    return float(err.max()), float(err.mean()), float(lse_err)


def assert_attention_close(out_gpu, lse_gpu, out_ref, lse_ref, rows=None, tag=""):
    mx, mean, lerr = attention_errors(out_gpu, lse_gpu, out_ref, lse_ref, rows)
    assert mx <= OUT_MAX_ABS, f"{tag} max-abs {mx:.3g} > {OUT_MAX_ABS}"
    assert mean <= OUT_MEAN_ABS, f"{tag} mean-abs {mean:.3g} > {OUT_MEAN_ABS}"
    assert lerr <= LSE_ABS, f"{tag} lse abs {lerr:.3g} > {LSE_ABS}"
    return mx, mean, lerr
