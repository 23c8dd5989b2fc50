"""Thin ctypes binding over libpkv.so (C ABI in include/pkv.h).

Argument marshalling only: shapes are read from the tensors, outputs are
allocated with PyTorch when the caller passes none, and every computation
runs in the library's CUDA kernels on the caller's current stream. There is
no fallback: if ``libpkv.so`` is missing or fails to load, every call raises.
Tensors live on the GPU, except that the decode calls also take q,
batch_idx, seq_lens, k_new, v_new, out and lse as pinned host tensors, which
the kernels read or write over the host link (no copy).

Functions keep the names of the C entry points: ``pkv_append``,
``pkv_append_rope``, ``pkv_decode_workspace_size``, ``pkv_decode_attention``,
``pkv_decode_append_attention``, ``pkv_decode_attention_static_scratch``,
``pkv_prefill_attention``, ``pkv_prefill_paged_attention``,
``pkv_mixed_workspace_size``, ``pkv_mixed_attention``,
``pkv_stage_from_host``, ``pkv_status_string``,
``pkv_status_from_device_error`` and ``pkv_last_cuda_error_string``.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libpkv.so")

PKV_OK = 0
STATUS_NAMES = {0: "PKV_OK", 1: "PKV_ERR_ARG", 2: "PKV_ERR_ALIGN",
                3: "PKV_ERR_BAD_PAGE", 4: "PKV_ERR_WORKSPACE", 5: "PKV_ERR_CUDA",
                6: "PKV_ERR_DEVICE", 7: "PKV_ERR_BAD_INPUT"}
DEV_ERR_BAD_PAGE = 0x1
DEV_ERR_BAD_SLOT = 0x2
DEV_ERR_BAD_POS = 0x4
DEV_ERR_LAYOUT = 0x8
DEV_ERR_TIMEOUT = 0x10

EXPORTED = ("pkv_append", "pkv_append_rope", "pkv_decode_workspace_size", "pkv_decode_attention",
            "pkv_decode_append_attention", "pkv_decode_attention_static_scratch",
            "pkv_prefill_paged_attention",
            "pkv_prefill_attention", "pkv_mixed_workspace_size", "pkv_mixed_attention",
            "pkv_stage_from_host", "pkv_status_string",
            "pkv_status_from_device_error", "pkv_last_cuda_error_string")


class PkvError(RuntimeError):
    """A libpkv call returned a status other than PKV_OK."""

    def __init__(self, func: str, status: int):
        self.status = status
        detail = status_string(status)
        if status == 5:
            detail += ": " + load_library().pkv_last_cuda_error_string().decode()
        super().__init__(f"{func}: {STATUS_NAMES.get(status, status)} ({detail})")


class CacheDesc(ctypes.Structure):
    _fields_ = [("num_pages", ctypes.c_int), ("page_size", ctypes.c_int),
                ("num_kv_heads", ctypes.c_int), ("head_dim", ctypes.c_int),
                ("max_batch", ctypes.c_int), ("max_blocks", ctypes.c_int)]


_lib = None


def load_library() -> ctypes.CDLL:
    """Loads the in-tree libpkv.so (built by ``paged_kv_gqa_pkv_gb300.build``)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                           "`python -m paged_kv_gqa_pkv_gb300.build`")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32p, f32p = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p
    c_int, c_float, c_size = ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    desc_p = ctypes.POINTER(CacheDesc)
    lib.pkv_append.argtypes = [desc_p, vp, vp, i32p, vp, vp, i32p, i32p, c_int, i32p, vp]
    lib.pkv_append.restype = c_int
    lib.pkv_append_rope.argtypes = [desc_p, vp, vp, i32p, vp, vp, i32p, i32p, c_int, f32p, f32p,
                                    c_int, f32p, c_float, i32p, vp]
    lib.pkv_append_rope.restype = c_int
    lib.pkv_decode_workspace_size.argtypes = [desc_p, c_int, c_int, c_int]
    lib.pkv_decode_workspace_size.restype = c_size
    lib.pkv_decode_attention.argtypes = [desc_p, vp, vp, i32p, vp, c_int, i32p, i32p, c_int,
                                         c_float, vp, f32p, vp, c_size, i32p, vp]
    lib.pkv_decode_attention.restype = c_int
    lib.pkv_decode_append_attention.argtypes = [desc_p, vp, vp, i32p, vp, c_int, vp, vp, i32p,
                                                i32p, c_int, c_float, vp, f32p, vp, c_size, i32p,
                                                vp]
    lib.pkv_decode_append_attention.restype = c_int
    lib.pkv_prefill_paged_attention.argtypes = [desc_p, vp, vp, i32p, vp, c_int, i32p, i32p,
                                                c_int, c_float, vp, f32p, i32p, vp]
    lib.pkv_prefill_paged_attention.restype = c_int
    lib.pkv_prefill_attention.argtypes = [vp, vp, vp, c_int, c_int, c_int, i32p, i32p, c_int,
                                          c_float, vp, f32p, i32p, vp]
    lib.pkv_prefill_attention.restype = c_int
    lib.pkv_decode_attention_static_scratch.argtypes = [desc_p, vp, vp, i32p, vp, c_int, i32p,
                                                        i32p, c_int, c_float, vp, f32p, i32p,
                                                        vp]
    lib.pkv_decode_attention_static_scratch.restype = c_int
    lib.pkv_mixed_workspace_size.argtypes = [desc_p, c_int, c_int]
    lib.pkv_mixed_workspace_size.restype = c_size
    lib.pkv_mixed_attention.argtypes = [desc_p, vp, vp, i32p, vp, c_int, i32p, i32p, c_int,
                                        c_float, vp, f32p, vp, c_size, i32p, vp]
    lib.pkv_mixed_attention.restype = c_int
    lib.pkv_stage_from_host.argtypes = [vp, vp, c_size, vp]
    lib.pkv_stage_from_host.restype = c_int
    lib.pkv_status_string.argtypes = [c_int]
    lib.pkv_status_string.restype = ctypes.c_char_p
    lib.pkv_last_cuda_error_string.argtypes = []
    lib.pkv_last_cuda_error_string.restype = ctypes.c_char_p
    lib.pkv_status_from_device_error.argtypes = [ctypes.c_int32]
    lib.pkv_status_from_device_error.restype = c_int
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load_library().pkv_status_string(int(status)).decode()


pkv_status_string = status_string


def pkv_status_from_device_error(dev_err_word: int) -> int:
    """Status for a dev_err word read back after the stream synchronised:
    PKV_OK when 0, PKV_ERR_BAD_PAGE when the bad-page bit is set, else
    PKV_ERR_BAD_INPUT."""
    return int(load_library().pkv_status_from_device_error(int(dev_err_word)))


def pkv_last_cuda_error_string() -> str:
    """Text of the CUDA error behind the last PKV_ERR_CUDA of this process."""
    return load_library().pkv_last_cuda_error_string().decode()


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _need(t: torch.Tensor, name: str, dtype: torch.dtype, ndim: int, host_ok: bool = False):
    """A contiguous tensor of `dtype` and rank `ndim` on the GPU, or (with
    host_ok) in pinned host memory, which the decode kernels read over the
    host link."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    where_ok = t.is_cuda or (host_ok and t.device.type == "cpu" and t.is_pinned())
    if t.dtype != dtype or t.dim() != ndim or not where_ok or not t.is_contiguous():
        kind = "CUDA or pinned host" if host_ok else "CUDA"
        raise ValueError(f"{name}: expected a contiguous {kind} {dtype} tensor of rank {ndim}, "
                         f"got {t.dtype} {tuple(t.shape)} on {t.device}")


def cache_desc(k_pool: torch.Tensor, page_table: torch.Tensor, page_size: int) -> CacheDesc:
    rows, hkv, d = k_pool.shape
    if rows % page_size:
        raise ValueError("pool rows must be a multiple of page_size")
    return CacheDesc(rows // page_size, page_size, hkv, d, page_table.shape[0],
                     page_table.shape[1])


def _check(func: str, status: int):
    if status != PKV_OK:
        raise PkvError(func, status)


def pkv_append(k_pool, v_pool, page_table, k_new, v_new, batch_idx, input_pos,
               page_size: int, dev_err=None, stream=None) -> None:
    """Writes k_new/v_new [N, H_kv, D] into the pools through the page table."""
    for name, t, dt, nd in (("k_pool", k_pool, torch.bfloat16, 3),
                            ("v_pool", v_pool, torch.bfloat16, 3),
                            ("page_table", page_table, torch.int32, 2),
                            ("k_new", k_new, torch.bfloat16, 3),
                            ("v_new", v_new, torch.bfloat16, 3),
                            ("batch_idx", batch_idx, torch.int32, 1),
                            ("input_pos", input_pos, torch.int32, 1)):
        _need(t, name, dt, nd)
    desc = cache_desc(k_pool, page_table, page_size)
    st = load_library().pkv_append(
        ctypes.byref(desc), _ptr(k_pool), _ptr(v_pool), _ptr(page_table), _ptr(k_new),
        _ptr(v_new), _ptr(batch_idx), _ptr(input_pos), int(batch_idx.numel()),
        _ptr(dev_err), _stream(stream))
    _check("pkv_append", st)


def pkv_append_rope(k_pool, v_pool, page_table, k_new, v_new, batch_idx, input_pos,
                    page_size: int, rope_cos, rope_sin, k_norm_weight=None,
                    k_norm_eps: float = 1e-6, dev_err=None, stream=None) -> None:
    """pkv_append with the rotary embedding (and, given ``k_norm_weight``
    fp32 [D], the per-head k_norm before it) applied to K; rope_cos/rope_sin
    are fp32 [L, D/2] tables indexed by position."""
    for name, t, dt, nd in (("k_pool", k_pool, torch.bfloat16, 3),
                            ("v_pool", v_pool, torch.bfloat16, 3),
                            ("page_table", page_table, torch.int32, 2),
                            ("k_new", k_new, torch.bfloat16, 3),
                            ("v_new", v_new, torch.bfloat16, 3),
                            ("batch_idx", batch_idx, torch.int32, 1),
                            ("input_pos", input_pos, torch.int32, 1),
                            ("rope_cos", rope_cos, torch.float32, 2),
                            ("rope_sin", rope_sin, torch.float32, 2)):
        _need(t, name, dt, nd)
    if rope_cos.shape != rope_sin.shape or rope_cos.shape[1] * 2 != k_new.shape[2]:
        raise ValueError("rope tables must both be [L, D/2]")
    if k_norm_weight is not None:
        _need(k_norm_weight, "k_norm_weight", torch.float32, 1)
        if k_norm_weight.shape[0] != k_new.shape[2]:
            raise ValueError("k_norm_weight must be [D]")
    desc = cache_desc(k_pool, page_table, page_size)
    st = load_library().pkv_append_rope(
        ctypes.byref(desc), _ptr(k_pool), _ptr(v_pool), _ptr(page_table), _ptr(k_new),
        _ptr(v_new), _ptr(batch_idx), _ptr(input_pos), int(batch_idx.numel()), _ptr(rope_cos),
        _ptr(rope_sin), int(rope_cos.shape[0]), _ptr(k_norm_weight), float(k_norm_eps),
        _ptr(dev_err), _stream(stream))
    _check("pkv_append_rope", st)


def pkv_decode_workspace_size(k_pool, page_table, page_size: int, batch: int,
                              num_q_heads: int, max_seq_len: int = 0) -> int:
    desc = cache_desc(k_pool, page_table, page_size)
    n = load_library().pkv_decode_workspace_size(ctypes.byref(desc), batch, num_q_heads,
                                                 max_seq_len)
    if n == 0 and batch > 0:
        raise PkvError("pkv_decode_workspace_size", 1)
    return int(n)


def pkv_decode_attention(k_pool, v_pool, page_table, q, batch_idx, seq_lens,
                         page_size: int, scale: float, out=None, lse=None,
                         workspace=None, dev_err=None, stream=None):
    """Split-KV GQA decode. q [B, Hq, D] bf16 -> (out [B, Hq, D] bf16,
    lse [B, Hq] fp32). q, batch_idx and seq_lens may be pinned host tensors,
    and out/lse pinned host tensors too; the outputs default to the pools'
    device."""
    _need(q, "q", torch.bfloat16, 3, host_ok=True)
    for name, t, dt, nd, h in (("k_pool", k_pool, torch.bfloat16, 3, False),
                               ("v_pool", v_pool, torch.bfloat16, 3, False),
                               ("page_table", page_table, torch.int32, 2, False),
                               ("batch_idx", batch_idx, torch.int32, 1, True),
                               ("seq_lens", seq_lens, torch.int32, 1, True)):
        _need(t, name, dt, nd, host_ok=h)
    B, hq, d = q.shape
    if out is None:
        out = torch.empty((B, hq, d), dtype=torch.bfloat16, device=k_pool.device)
    if lse is None:
        lse = torch.empty((B, hq), dtype=torch.float32, device=k_pool.device)
    desc = cache_desc(k_pool, page_table, page_size)
    lib = load_library()
    if workspace is None:
        n = lib.pkv_decode_workspace_size(ctypes.byref(desc), B, hq, 0)
        workspace = torch.empty(max(int(n), 256), dtype=torch.uint8, device=k_pool.device)
    st = lib.pkv_decode_attention(
        ctypes.byref(desc), _ptr(k_pool), _ptr(v_pool), _ptr(page_table), _ptr(q), hq,
        _ptr(batch_idx), _ptr(seq_lens), B, float(scale), _ptr(out), _ptr(lse),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(dev_err),
        _stream(stream))
    _check("pkv_decode_attention", st)
    return out, lse


def pkv_decode_append_attention(k_pool, v_pool, page_table, q, k_new, v_new, batch_idx,
                                seq_lens, page_size: int, scale: float, out=None, lse=None,
                                workspace=None, dev_err=None, stream=None):
    """One decode step in one call: row b's new token (k_new/v_new
    [B, Hkv, D] bf16) is written to position seq_lens[b] - 1 of its slot and
    attended with the rest. Returns (out [B, Hq, D] bf16, lse [B, Hq] fp32)."""
    _need(q, "q", torch.bfloat16, 3, host_ok=True)
    for name, t, dt, nd, h in (("k_pool", k_pool, torch.bfloat16, 3, False),
                               ("v_pool", v_pool, torch.bfloat16, 3, False),
                               ("k_new", k_new, torch.bfloat16, 3, True),
                               ("v_new", v_new, torch.bfloat16, 3, True),
                               ("page_table", page_table, torch.int32, 2, False),
                               ("batch_idx", batch_idx, torch.int32, 1, True),
                               ("seq_lens", seq_lens, torch.int32, 1, True)):
        _need(t, name, dt, nd, host_ok=h)
    B, hq, d = q.shape
    if k_new.shape != (B, k_pool.shape[1], d) or v_new.shape != k_new.shape:
        raise ValueError("k_new/v_new must be [B, Hkv, D]")
    if out is None:
        out = torch.empty((B, hq, d), dtype=torch.bfloat16, device=k_pool.device)
    if lse is None:
        lse = torch.empty((B, hq), dtype=torch.float32, device=k_pool.device)
    desc = cache_desc(k_pool, page_table, page_size)
    lib = load_library()
    if workspace is None:
        n = lib.pkv_decode_workspace_size(ctypes.byref(desc), B, hq, 0)
        workspace = torch.empty(max(int(n), 256), dtype=torch.uint8, device=k_pool.device)
    st = lib.pkv_decode_append_attention(
        ctypes.byref(desc), _ptr(k_pool), _ptr(v_pool), _ptr(page_table), _ptr(q), hq,
        _ptr(k_new), _ptr(v_new), _ptr(batch_idx), _ptr(seq_lens), B, float(scale), _ptr(out),
        _ptr(lse), _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(dev_err),
        _stream(stream))
    _check("pkv_decode_append_attention", st)
    return out, lse


def pkv_prefill_paged_attention(k_pool, v_pool, page_table, q, batch_idx, input_pos,
                                page_size: int, scale: float, out=None, lse=None, dev_err=None,
                                stream=None):
    """Chunked prefill over the paged cache: token i of q [T, Hq, D] attends
    its slot's keys 0..input_pos[i] through the page table (its own chunk
    appended first). Returns (out [T, Hq, D] bf16, lse [T, Hq] fp32)."""
    _need(q, "q", torch.bfloat16, 3)
    for name, t, dt, nd in (("k_pool", k_pool, torch.bfloat16, 3),
                            ("v_pool", v_pool, torch.bfloat16, 3),
                            ("page_table", page_table, torch.int32, 2),
                            ("batch_idx", batch_idx, torch.int32, 1),
                            ("input_pos", input_pos, torch.int32, 1)):
        _need(t, name, dt, nd)
    T, hq, d = q.shape
    if out is None:
        out = torch.empty((T, hq, d), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((T, hq), dtype=torch.float32, device=q.device)
    desc = cache_desc(k_pool, page_table, page_size)
    st = load_library().pkv_prefill_paged_attention(
        ctypes.byref(desc), _ptr(k_pool), _ptr(v_pool), _ptr(page_table), _ptr(q), hq,
        _ptr(batch_idx), _ptr(input_pos), T, float(scale), _ptr(out), _ptr(lse), _ptr(dev_err),
        _stream(stream))
    _check("pkv_prefill_paged_attention", st)
    return out, lse


def pkv_mixed_workspace_size(k_pool, page_table, page_size: int, n_tokens: int,
                             num_q_heads: int) -> int:
    desc = cache_desc(k_pool, page_table, page_size)
    n = load_library().pkv_mixed_workspace_size(ctypes.byref(desc), n_tokens, num_q_heads)
    if n == 0:
        raise PkvError("pkv_mixed_workspace_size", 1)
    return int(n)


def pkv_mixed_attention(k_pool, v_pool, page_table, q, batch_idx, input_pos, page_size: int,
                        scale: float, out=None, lse=None, workspace=None, dev_err=None,
                        stream=None):
    """A step of prefill chunks and decode tokens in one call: the results of
    ``pkv_prefill_paged_attention`` (token i of q [T, Hq, D] attends its
    slot's keys 0..input_pos[i]), with the decode tokens served by the
    split-KV decode kernels. Returns (out [T, Hq, D] bf16, lse [T, Hq] fp32)."""
    _need(q, "q", torch.bfloat16, 3)
    for name, t, dt, nd in (("k_pool", k_pool, torch.bfloat16, 3),
                            ("v_pool", v_pool, torch.bfloat16, 3),
                            ("page_table", page_table, torch.int32, 2),
                            ("batch_idx", batch_idx, torch.int32, 1),
                            ("input_pos", input_pos, torch.int32, 1)):
        _need(t, name, dt, nd)
    T, hq, d = q.shape
    if out is None:
        out = torch.empty((T, hq, d), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((T, hq), dtype=torch.float32, device=q.device)
    desc = cache_desc(k_pool, page_table, page_size)
    lib = load_library()
    if workspace is None:
        n = lib.pkv_mixed_workspace_size(ctypes.byref(desc), T, hq)
        workspace = torch.empty(max(int(n), 256), dtype=torch.uint8, device=q.device)
    st = lib.pkv_mixed_attention(
        ctypes.byref(desc), _ptr(k_pool), _ptr(v_pool), _ptr(page_table), _ptr(q), hq,
        _ptr(batch_idx), _ptr(input_pos), T, float(scale), _ptr(out), _ptr(lse), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(dev_err), _stream(stream))
    _check("pkv_mixed_attention", st)
    return out, lse


def pkv_decode_attention_static_scratch(k_pool, v_pool, page_table, q, batch_idx, seq_lens,
                                        page_size: int, scale: float, out=None, lse=None,
                                        dev_err=None, stream=None):
    """Decode for callers that cannot allocate device memory: same result as
    ``pkv_decode_attention``, with the library's built-in 8 MiB scratch array
    instead of a caller workspace (calls must not overlap on the GPU)."""
    _need(q, "q", torch.bfloat16, 3, host_ok=True)
    for name, t, dt, nd, h in (("k_pool", k_pool, torch.bfloat16, 3, False),
                               ("v_pool", v_pool, torch.bfloat16, 3, False),
                               ("page_table", page_table, torch.int32, 2, False),
                               ("batch_idx", batch_idx, torch.int32, 1, True),
                               ("seq_lens", seq_lens, torch.int32, 1, True)):
        _need(t, name, dt, nd, host_ok=h)
    B, hq, d = q.shape
    if out is None:
        out = torch.empty((B, hq, d), dtype=torch.bfloat16, device=k_pool.device)
    if lse is None:
        lse = torch.empty((B, hq), dtype=torch.float32, device=k_pool.device)
    desc = cache_desc(k_pool, page_table, page_size)
    st = load_library().pkv_decode_attention_static_scratch(
        ctypes.byref(desc), _ptr(k_pool), _ptr(v_pool), _ptr(page_table), _ptr(q), hq,
        _ptr(batch_idx), _ptr(seq_lens), B, float(scale), _ptr(out), _ptr(lse), _ptr(dev_err),
        _stream(stream))
    _check("pkv_decode_attention_static_scratch", st)
    return out, lse


def pkv_prefill_attention(q, k, v, batch_idx, input_pos, scale: float, out=None,
                          lse=None, dev_err=None, stream=None):
    """Packed document-causal prefill. q [T, Hq, D], k/v [T, H_kv, D] bf16 ->
    (out [T, Hq, D] bf16, lse [T, Hq] fp32)."""
    for name, t, dt, nd in (("q", q, torch.bfloat16, 3), ("k", k, torch.bfloat16, 3),
                            ("v", v, torch.bfloat16, 3),
                            ("batch_idx", batch_idx, torch.int32, 1),
                            ("input_pos", input_pos, torch.int32, 1)):
        _need(t, name, dt, nd)
    T, hq, d = q.shape
    if out is None:
        out = torch.empty((T, hq, d), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((T, hq), dtype=torch.float32, device=q.device)
    st = load_library().pkv_prefill_attention(
        _ptr(q), _ptr(k), _ptr(v), hq, k.shape[1], d, _ptr(batch_idx), _ptr(input_pos), T,
        float(scale), _ptr(out), _ptr(lse), _ptr(dev_err), _stream(stream))
    _check("pkv_prefill_attention", st)
    return out, lse


def pkv_stage_from_host(dst: torch.Tensor, src: torch.Tensor, stream=None) -> None:
    """Copies the bytes of ``src`` (pinned host memory) into ``dst`` (a CUDA
    tensor of the same byte size) with the GPU's own loads, on the current
    stream. Both contiguous, 16-byte aligned, size a multiple of 16 bytes."""
    for name, t in (("dst", dst), ("src", src)):
        if not isinstance(t, torch.Tensor) or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous tensor")
    if not dst.is_cuda:
        raise ValueError("dst must be a CUDA tensor")
    nbytes = src.numel() * src.element_size()
    if dst.numel() * dst.element_size() != nbytes:
        raise ValueError("dst and src must hold the same number of bytes")
    st = load_library().pkv_stage_from_host(_ptr(dst), _ptr(src), nbytes, _stream(stream))
    _check("pkv_stage_from_host", st)
