"""The oracle over every row of a full-size workload, on all host cores.

The oracle is a per-row float64 loop; a full-size packed prefill (32 718
rows) or chunked step (8 240 rows over ~100 k cached keys) takes minutes on
one core. Rows are independent, so the work is cut into tasks (a document's
tokens for the packed prefill, runs of tokens for the chunked step) and run
by a process pool started with ``spawn`` (never forked from a process that
has touched CUDA). The large read-only inputs are placed once in shared
memory and every worker maps them. The arithmetic is the oracle's own:
each task calls ``oracle.prefill_attention`` or
``oracle.paged_prefill_attention`` unchanged, on the task's query rows.

* Packed prefill: a token attends only tokens of its own document, so the
  oracle run on one document's slice of the packing gives exactly that
  document's rows of the whole run.
* Chunked prefill: a token's result depends on its own q row, slot and
  position and on the pools and table, so the oracle run on a subset of
  query rows (with the whole pools) gives exactly those rows.

Results come back as the oracle's float64 output rounded to bf16 (bits) and
its float64 LSE.
"""

from __future__ import annotations

import multiprocessing as mp
import os
from multiprocessing import shared_memory

import numpy as np

import oracle.paged_attention as orc

_W = {}   # per-worker views of the shared arrays


def workers() -> int:
    return max(1, min(16, os.cpu_count() or 1))


class _Shared:
    """Named numpy arrays copied once into shared memory."""

    def __init__(self, arrays: dict):
        self.blocks, self.spec = [], {}
        for name, a in arrays.items():
            a = np.ascontiguousarray(a)
            shm = shared_memory.SharedMemory(create=True, size=max(1, a.nbytes))
            np.ndarray(a.shape, a.dtype, buffer=shm.buf)[...] = a
            self.blocks.append(shm)
            self.spec[name] = (shm.name, a.shape, a.dtype.str)

    def close(self):
        for shm in self.blocks:
            shm.close()
            shm.unlink()


def _attach(spec, extra):
    global _W
    _W = {"_shm": []}
    for name, (shm_name, shape, dt) in spec.items():
        shm = shared_memory.SharedMemory(name=shm_name)
        _W["_shm"].append(shm)
        _W[name] = np.ndarray(shape, np.dtype(dt), buffer=shm.buf)
    _W.update(extra)


def _prefill_task(span):
    lo, hi = span
    out, lse = orc.prefill_attention(_W["q"][lo:hi], _W["k"][lo:hi], _W["v"][lo:hi],
                                     _W["bidx"][lo:hi], _W["pos"][lo:hi], _W["scale"])
    return lo, hi, orc.f64_to_bf16_bits(out), lse


def _paged_task(rows):
    rows = np.asarray(rows, dtype=np.int64)
    out, lse, bad = orc.paged_prefill_attention(
        _W["q"][rows], _W["kb"], _W["vb"], _W["table"], _W["bidx"][rows], _W["pos"][rows],
        _W["page_size"], _W["scale"])
    return rows, orc.f64_to_bf16_bits(out), lse, [int(rows[i]) for i in bad]


def _restore(saved):
    for k, v in saved.items():
        if v is None:
            os.environ.pop(k, None)
        else:
            os.environ[k] = v


def _run(arrays, extra, fn, tasks):
    """Runs fn over tasks in a spawn pool with the arrays shared; yields results."""
    shared = _Shared(arrays)
    saved = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS",
                                            "MKL_NUM_THREADS")}
    try:
        for k in saved:                        # one BLAS thread per worker
            os.environ[k] = "1"
        ctx = mp.get_context("spawn")
        pool = ctx.Pool(min(workers(), len(tasks)), initializer=_attach,
                        initargs=(shared.spec, extra))
        _restore(saved)
        with pool:
            yield from pool.imap_unordered(fn, tasks)
    finally:
        _restore(saved)
        shared.close()


def prefill_all_rows(q, k, v, batch_idx, input_pos, scale):
    """oracle.prefill_attention on every row of a packing whose documents are
    contiguous runs of equal batch_idx. Inputs are bf16 bits (numpy uint16)
    and int arrays. Returns (out_bits uint16 [T, Hq, D], lse float64 [T, Hq])."""
    bidx = np.asarray(batch_idx)
    T = len(bidx)
    starts = [0] + [i for i in range(1, T) if bidx[i] != bidx[i - 1]] + [T]
    spans = [(starts[j], starts[j + 1]) for j in range(len(starts) - 1)]
    if len(set(int(bidx[lo]) for lo, _ in spans)) != len(spans):
        raise ValueError("a document is split over several runs of the packing")
    spans.sort(key=lambda s: -(s[1] - s[0]))            # longest first
    out = np.zeros(q.shape, dtype=np.uint16)
    lse = np.full(q.shape[:2], np.nan)
    for lo, hi, o, l in _run({"q": q, "k": k, "v": v, "bidx": bidx,
                              "pos": np.asarray(input_pos)}, {"scale": float(scale)},
                             _prefill_task, spans):
        out[lo:hi], lse[lo:hi] = o, l
    return out, lse


def paged_prefill_all_rows(q, k_pool, v_pool, page_table, batch_idx, input_pos, page_size,
                           scale, rows_per_task=48):
    """oracle.paged_prefill_attention on every token, the pools as given (the
    chunks' K/V already appended). Returns (out_bits, lse, bad_rows)."""
    T = q.shape[0]
    pos = np.asarray(input_pos)
    order = np.argsort(-pos, kind="stable")             # most keys first
    tasks = [order[i:i + rows_per_task].tolist() for i in range(0, T, rows_per_task)]
    out = np.zeros(q.shape, dtype=np.uint16)
    lse = np.full(q.shape[:2], np.nan)
    bad = []
    for rows, o, l, b in _run({"q": q, "kb": k_pool, "vb": v_pool, "table": page_table,
                               "bidx": np.asarray(batch_idx), "pos": pos},
                              {"scale": float(scale), "page_size": int(page_size)},
                              _paged_task, tasks):
        out[rows], lse[rows] = o, l
        bad += b
    return out, lse, sorted(bad)
