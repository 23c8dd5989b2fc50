"""The C ABI without a GPU: the library loads, exports every entry point
include/pkv.h declares, and its host-side validation rejects bad arguments
before touching the device."""

import ctypes
import os
import re

import pytest

from paged_kv_gqa_pkv_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "pkv.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_[a-z_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(binding.LIB_PATH):
        from paged_kv_gqa_pkv_gb300 import build
        build.build()
    return binding.load_library()


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert set(binding.EXPORTED) <= set(names)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in pkv.h but not exported"


def test_binding_has_a_function_of_each_declared_name():
    """The Python binding keeps the C names: one callable per declared entry
    point."""
    for n in _declared():
        assert callable(getattr(binding, n, None)), f"binding has no {n}"


def test_status_strings(lib):
    for s in range(8):
        assert binding.status_string(s) != "unknown status"
    assert binding.status_string(99) == "unknown status"
    assert lib.pkv_status_from_device_error(0) == 0
    assert lib.pkv_status_from_device_error(binding.DEV_ERR_BAD_PAGE | 4) == 3
    assert lib.pkv_status_from_device_error(binding.DEV_ERR_LAYOUT) == 7


def _desc(**kw):
    d = dict(num_pages=32, page_size=16, num_kv_heads=2, head_dim=128, max_batch=5,
             max_blocks=16)
    d.update(kw)
    return binding.CacheDesc(**d)


P = ctypes.c_void_p


@pytest.mark.parametrize("kw", [dict(head_dim=64), dict(page_size=24), dict(page_size=0),
                                dict(num_pages=0), dict(num_kv_heads=0), dict(max_blocks=0),
                                dict(num_pages=1 << 28, page_size=128)])
def test_append_rejects_bad_geometry(lib, kw):
    d = _desc(**kw)
    st = lib.pkv_append(ctypes.byref(d), P(256), P(256), P(256), P(256), P(256), P(256),
                        P(256), 4, None, None)
    assert st == 1


def test_append_rejects_null_and_misaligned(lib):
    d = _desc()
    assert lib.pkv_append(None, P(256), P(256), P(256), P(256), P(256), P(256), P(256), 4,
                          None, None) == 1
    assert lib.pkv_append(ctypes.byref(d), None, P(256), P(256), P(256), P(256), P(256),
                          P(256), 4, None, None) == 1
    assert lib.pkv_append(ctypes.byref(d), P(264), P(256), P(256), P(256), P(256), P(256),
                          P(256), 4, None, None) == 2
    assert lib.pkv_append(ctypes.byref(d), P(256), P(256), P(258), P(256), P(256), P(256),
                          P(256), 4, None, None) == 2
    assert lib.pkv_append(ctypes.byref(d), P(256), P(256), P(256), P(256), P(256), P(256),
                          P(256), -1, None, None) == 1
    # nothing to do is not an error, and touches nothing
    assert lib.pkv_append(ctypes.byref(d), None, None, None, None, None, None, None, 0,
                          None, None) == 0


def test_decode_rejects_bad_arguments(lib):
    d = _desc()
    args = lambda hq=8, batch=4, q=256, ws=256, wsb=1 << 20, scale=0.088: (  # noqa: E731
        ctypes.byref(d), P(256), P(256), P(256), P(q), hq, P(256), P(256), batch,
        ctypes.c_float(scale), P(256), P(256), P(ws), wsb, None, None)
    assert lib.pkv_decode_attention(*args(hq=6)) == 1          # group 3
    assert lib.pkv_decode_attention(*args(hq=32)) == 1         # group 16
    assert lib.pkv_decode_attention(*args(batch=-1)) == 1
    # any batch size is accepted (above 512 rows the call runs as several
    # launches): 100 000 rows pass the argument checks and stop at the
    # device check without a supported GPU, else at the 1 MiB workspace
    assert lib.pkv_decode_attention(*args(batch=100000)) in (4, 5)
    assert lib.pkv_decode_attention(*args(q=264)) == 2
    assert lib.pkv_decode_attention(*args(scale=float("nan"))) == 1
    assert lib.pkv_decode_attention(*args(batch=0)) == 0
    assert lib.pkv_decode_workspace_size(ctypes.byref(d), 4, 6, 0) == 0


def test_prefill_rejects_bad_arguments(lib):
    args = lambda hq=32, hkv=8, d=128, n=16, q=256: (  # noqa: E731
        P(q), P(256), P(256), hq, hkv, d, P(256), P(256), n, ctypes.c_float(0.088),
        P(256), P(256), None, None)
    assert lib.pkv_prefill_attention(*args(d=64)) == 1
    assert lib.pkv_prefill_attention(*args(hq=24)) == 1
    assert lib.pkv_prefill_attention(*args(n=-3)) == 1
    assert lib.pkv_prefill_attention(*args(q=250)) == 2
    assert lib.pkv_prefill_attention(*args(n=0)) == 0


def test_without_a_gpu_calls_fail_cleanly(lib):
    """Valid-looking arguments on a machine with no GPU: a CUDA or device
    status, never a crash."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    d = _desc()
    st = lib.pkv_append(ctypes.byref(d), P(256), P(256), P(256), P(256), P(256), P(256),
                        P(256), 4, None, None)
    assert st in (5, 6)


def test_append_rope_rejects_bad_arguments(lib):
    d = _desc()
    args = lambda cos=256, sin=256, n=4, L=32, w=0, eps=1e-6: (  # noqa: E731
        ctypes.byref(d), P(256), P(256), P(256), P(256), P(256), P(256), P(256), n, P(cos),
        P(sin), L, P(w) if w else None, ctypes.c_float(eps), None, None)
    assert lib.pkv_append_rope(*args(cos=0)) == 1
    assert lib.pkv_append_rope(*args(w=256, eps=-1.0)) == 1
    assert lib.pkv_append_rope(*args(w=256, eps=float("nan"))) == 1
    assert lib.pkv_append_rope(*args(w=264)) == 2
    assert lib.pkv_append_rope(*args(L=0)) == 1
    assert lib.pkv_append_rope(*args(sin=264)) == 2
    assert lib.pkv_append_rope(*args(n=-1)) == 1
    assert lib.pkv_append_rope(*args(n=0)) == 0


def test_decode_append_rejects_bad_arguments(lib):
    d = _desc()
    args = lambda kn=256, vn=256, hq=8, batch=4: (  # noqa: E731
        ctypes.byref(d), P(256), P(256), P(256), P(256), hq, P(kn), P(vn), P(256), P(256),
        batch, ctypes.c_float(0.088), P(256), P(256), P(256), 1 << 20, None, None)
    assert lib.pkv_decode_append_attention(*args(kn=0)) == 1
    assert lib.pkv_decode_append_attention(*args(vn=0)) == 1
    assert lib.pkv_decode_append_attention(*args(kn=264)) == 2
    assert lib.pkv_decode_append_attention(*args(hq=6)) == 1
    assert lib.pkv_decode_append_attention(*args(batch=0, kn=0, vn=0)) == 0


def test_prefill_paged_rejects_bad_arguments(lib):
    args = lambda ps=16, hq=8, n=16, q=256, scale=0.088: (  # noqa: E731
        ctypes.byref(_desc(page_size=ps)), P(256), P(256), P(256), P(q), hq, P(256), P(256), n,
        ctypes.c_float(scale), P(256), P(256), None, None)
    assert lib.pkv_prefill_paged_attention(*args(ps=48)) == 1      # tiles would straddle pages
    assert lib.pkv_prefill_paged_attention(*args(ps=24)) == 1      # not a multiple of 16
    assert lib.pkv_prefill_paged_attention(*args(hq=6)) == 1
    assert lib.pkv_prefill_paged_attention(*args(n=-1)) == 1
    assert lib.pkv_prefill_paged_attention(*args(scale=0.0)) == 1
    assert lib.pkv_prefill_paged_attention(*args(q=264)) == 2
    assert lib.pkv_prefill_paged_attention(*args(n=0)) == 0
    assert lib.pkv_prefill_paged_attention(*args(ps=256, n=0)) == 0


def test_stage_from_host_rejects_bad_arguments(lib):
    """Host checks run before any CUDA call: empty copies succeed, null
    pointers and sizes off the 16-byte grain are ARG, misaligned pointers
    ALIGN."""
    assert lib.pkv_stage_from_host(None, None, 0, None) == 0
    assert lib.pkv_stage_from_host(None, P(256), 32, None) == 1
    assert lib.pkv_stage_from_host(P(256), None, 32, None) == 1
    assert lib.pkv_stage_from_host(P(256), P(512), 24, None) == 1
    assert lib.pkv_stage_from_host(P(264), P(512), 32, None) == 2
    assert lib.pkv_stage_from_host(P(256), P(520), 32, None) == 2


def test_mixed_rejects_bad_arguments(lib):
    d = _desc()
    args = lambda ps=16, hq=8, n=4, q=256, ws=256: (  # noqa: E731
        ctypes.byref(_desc(page_size=ps)), P(256), P(256), P(256), P(q), hq, P(256), P(256), n,
        ctypes.c_float(0.088), P(256), P(256), P(ws), 1 << 20, None, None)
    assert lib.pkv_mixed_attention(*args(ps=48)) == 1      # page size the prefill side refuses
    assert lib.pkv_mixed_attention(*args(hq=12)) == 1      # GQA group of 6
    assert lib.pkv_mixed_attention(*args(n=-1)) == 1
    assert lib.pkv_mixed_attention(*args(n=0)) == 0
    assert lib.pkv_mixed_attention(*args(q=264)) == 2
    assert lib.pkv_mixed_workspace_size(ctypes.byref(d), -1, 8) == 0
