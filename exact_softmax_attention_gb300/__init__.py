"""Exact softmax attention for GB300 (sm_103a): Python binding of the C ABI in ``include/attn.h``.

The functions here only marshal arguments (tensor data pointers, sizes, the CUDA
stream) and call the native library; every step of the computation runs in its
CUDA kernels. There is no fallback: if the library is missing, importing this
package raises.

Tensors may be ``torch.Tensor`` objects (their ``data_ptr()`` is passed) or raw
integer device addresses. ``stream`` may be a ``torch.cuda.Stream``, an integer
``cudaStream_t`` handle, or ``None`` for the current PyTorch stream (the legacy
default stream when PyTorch is not in use).
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libattn_gb300.so")

ATTN_OK = 0
ATTN_ERR_NULL_PTR = -1
ATTN_ERR_BAD_SHAPE = -2
ATTN_ERR_ALIGN = -3
ATTN_ERR_UNSUPPORTED_ARCH = -4
ATTN_ERR_CUDA = -5
ATTN_ERR_DEVICE_TIMEOUT = -6
ATTN_ERR_DEVICE_BAD_INDEX = -7
ATTN_ERR_BAD_ARG = -8
ATTN_ERR_SCRATCH_TOO_SMALL = -9

ATTN_FP8_E4M3 = 0
ATTN_FP8_E5M2 = 1
FP8_FORMATS = {"e4m3": ATTN_FP8_E4M3, "e5m2": ATTN_FP8_E5M2}

#: every symbol the header declares
EXPORTS = ("attn_fwd", "attn_fwd_hd", "attn_fwd_fp8", "attn_decode_paged", "attn_decode_paged_fp8", "attn_decode_paged_noalloc", "attn_decode_plan",
           "attn_decode_workspace_bytes", "attn_status_string", "attn_get_device_status",
           "attn_set_option", "attn_get_option", "attn_read_counters", "attn_debug_exp2", "attn_debug_watchdog",
           "attn_version")


class AttnError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: {status_string(code)} (status {code})")
        self.code = code


if not os.path.exists(LIB_PATH):
    raise ImportError(f"CUDA attention library not built: {LIB_PATH} is missing "
                      "(run __graft_entry__.build() or python exact_softmax_attention_gb300/build.py)")

lib = ctypes.CDLL(LIB_PATH)
_vp, _i, _f, _d = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_double
lib.attn_fwd.argtypes = [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, _i, _vp, _vp]
lib.attn_fwd.restype = _i
lib.attn_fwd_hd.argtypes = [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _f, _i, _vp, _vp]
lib.attn_fwd_hd.restype = _i
lib.attn_fwd_fp8.argtypes = [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, _i, _vp, _vp, _i, _f, _f, _f]
lib.attn_fwd_fp8.restype = _i
lib.attn_decode_paged.argtypes = [_vp, _vp, _vp, _vp, _vp, _i, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, _i]
lib.attn_decode_paged.restype = _i
lib.attn_decode_paged_fp8.argtypes = [_vp, _vp, _vp, _vp, _vp, _i, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, _i, _i, _f,
                                       _f]
lib.attn_decode_paged_fp8.restype = _i
lib.attn_decode_paged_noalloc.argtypes = [_vp, _vp, _vp, _vp, _vp, _i, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, _i]
lib.attn_decode_paged_noalloc.restype = _i
lib.attn_decode_plan.argtypes = [_i, _i, _i, _i, _i, _i, _i, ctypes.POINTER(_i), ctypes.POINTER(_i)]
lib.attn_decode_plan.restype = _i
lib.attn_decode_workspace_bytes.argtypes = [_i, _i, _i, _i]
lib.attn_decode_workspace_bytes.restype = ctypes.c_size_t
lib.attn_status_string.argtypes = [_i]
lib.attn_status_string.restype = ctypes.c_char_p
lib.attn_get_device_status.argtypes = [_vp]
lib.attn_get_device_status.restype = _i
lib.attn_set_option.argtypes = [ctypes.c_char_p, _d]
lib.attn_set_option.restype = _i
lib.attn_get_option.argtypes = [ctypes.c_char_p, ctypes.POINTER(_d)]
lib.attn_get_option.restype = _i
lib.attn_read_counters.argtypes = [ctypes.POINTER(ctypes.c_ulonglong), _i]
lib.attn_read_counters.restype = _i
lib.attn_debug_exp2.argtypes = [_vp, _vp, ctypes.c_longlong, _i, _vp]
lib.attn_debug_exp2.restype = _i
lib.attn_debug_watchdog.argtypes = [ctypes.c_ulonglong, _vp]
lib.attn_debug_watchdog.restype = _i
lib.attn_version.argtypes = []
lib.attn_version.restype = ctypes.c_char_p


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s):
    if s is None:
        try:
            import torch
            if torch.cuda.is_available() and torch.cuda.is_initialized():
                return torch.cuda.current_stream().cuda_stream
        except ImportError:
            pass
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(code: int, where: str, raise_on_error: bool):
    if raise_on_error and code != ATTN_OK:
        raise AttnError(code, where)
    return code


def status_string(code: int) -> str:
    return lib.attn_status_string(code).decode()


def attn_fwd(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, d, scale, causal, cu_seqlens=None, stream=None,
             raise_on_error=True):
    """Exact attention forward; see ``attn_fwd`` in include/attn.h."""
    rc = lib.attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B), int(Hq), int(Hkv), int(Nq), int(Nk),
                      int(d), float(scale), int(causal), _ptr(cu_seqlens), _stream(stream))
    return _check(rc, "attn_fwd", raise_on_error)


def attn_fwd_hd(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, d, dv, scale, causal, cu_seqlens=None, stream=None,
                raise_on_error=True):
    """Forward with values narrower than queries and keys, (d, dv) = (192, 128); see
    ``attn_fwd_hd`` in include/attn.h."""
    rc = lib.attn_fwd_hd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B), int(Hq), int(Hkv), int(Nq), int(Nk),
                         int(d), int(dv), float(scale), int(causal), _ptr(cu_seqlens), _stream(stream))
    return _check(rc, "attn_fwd_hd", raise_on_error)


def attn_fwd_fp8(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, d, scale, causal, cu_seqlens=None, stream=None,
                 fp8_format="e4m3", q_descale=1.0, k_descale=1.0, v_descale=1.0, raise_on_error=True):
    """Forward on 8-bit floating-point Q/K/V; see ``attn_fwd_fp8`` in include/attn.h."""
    fmt = FP8_FORMATS[fp8_format] if isinstance(fp8_format, str) else int(fp8_format)
    rc = lib.attn_fwd_fp8(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B), int(Hq), int(Hkv), int(Nq), int(Nk),
                          int(d), float(scale), int(causal), _ptr(cu_seqlens), _stream(stream), fmt, float(q_descale),
                          float(k_descale), float(v_descale))
    return _check(rc, "attn_fwd_fp8", raise_on_error)


def attn_decode_paged(q, k_cache, v_cache, page_table, seqlens, page_size, o, lse, stream, B, Hq, Hkv, d,
                      max_pages_per_seq, num_pages, scale, num_splits=0, raise_on_error=True):
    """Paged-KV split decode; see ``attn_decode_paged`` in include/attn.h."""
    rc = lib.attn_decode_paged(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(page_table), _ptr(seqlens),
                               int(page_size), _ptr(o), _ptr(lse), _stream(stream), int(B), int(Hq), int(Hkv), int(d),
                               int(max_pages_per_seq), int(num_pages), float(scale), int(num_splits))
    return _check(rc, "attn_decode_paged", raise_on_error)


def attn_decode_paged_fp8(q, k_cache, v_cache, page_table, seqlens, page_size, o, lse, stream, B, Hq, Hkv, d,
                          max_pages_per_seq, num_pages, scale, num_splits=0, kv_format="e4m3", k_descale=1.0,
                          v_descale=1.0, raise_on_error=True):
    """Paged decode over FP8 key/value caches; see ``attn_decode_paged_fp8`` in include/attn.h.
    ``kv_format`` is "e4m3" or "e5m2" (or the ATTN_FP8_* code)."""
    fmt = FP8_FORMATS[kv_format] if isinstance(kv_format, str) else int(kv_format)
    rc = lib.attn_decode_paged_fp8(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(page_table), _ptr(seqlens),
                                   int(page_size), _ptr(o), _ptr(lse), _stream(stream), int(B), int(Hq), int(Hkv),
                                   int(d), int(max_pages_per_seq), int(num_pages), float(scale), int(num_splits), fmt,
                                   float(k_descale), float(v_descale))
    return _check(rc, "attn_decode_paged_fp8", raise_on_error)


def attn_decode_paged_noalloc(q, k_cache, v_cache, page_table, seqlens, page_size, o, lse, stream, B, Hq, Hkv, d,
                              max_pages_per_seq, num_pages, scale, num_splits=0, raise_on_error=True):
    """attn_decode_paged without allocating: split partials use the library's fixed 32 MiB
    device array (see include/attn.h for the size limit and the sharing rules)."""
    rc = lib.attn_decode_paged_noalloc(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(page_table), _ptr(seqlens),
                                       int(page_size), _ptr(o), _ptr(lse), _stream(stream), int(B), int(Hq), int(Hkv),
                                       int(d), int(max_pages_per_seq), int(num_pages), float(scale), int(num_splits))
    return _check(rc, "attn_decode_paged_noalloc", raise_on_error)


def attn_decode_plan(B, Hq, Hkv, max_pages_per_seq, page_size, num_splits=0, num_sms=0):
    """(chunk tokens per split, splits per sequence) chosen by the library."""
    c, s = _i(), _i()
    rc = lib.attn_decode_plan(int(B), int(Hq), int(Hkv), int(max_pages_per_seq), int(page_size), int(num_splits),
                              int(num_sms), ctypes.byref(c), ctypes.byref(s))
    _check(rc, "attn_decode_plan", True)
    return c.value, s.value


def attn_decode_workspace_bytes(B, Hq, d, max_splits) -> int:
    """Bytes of split-KV workspace attn_decode_paged takes for these sizes."""
    return int(lib.attn_decode_workspace_bytes(int(B), int(Hq), int(d), int(max_splits)))


def attn_get_device_status(stream=None) -> int:
    """Synchronise the stream, read and clear the device status word (returns the status code)."""
    return lib.attn_get_device_status(_stream(stream))


def attn_set_option(name: str, value: float):
    _check(lib.attn_set_option(name.encode(), float(value)), f"attn_set_option({name})", True)


def attn_get_option(name: str) -> float:
    v = _d()
    _check(lib.attn_get_option(name.encode(), ctypes.byref(v)), f"attn_get_option({name})", True)
    return v.value


def attn_read_counters():
    out = (ctypes.c_ulonglong * 6)()
    _check(lib.attn_read_counters(out, 6), "attn_read_counters", True)
    return list(out)


def attn_debug_exp2(x, y, n, mode, stream=None):
    return _check(lib.attn_debug_exp2(_ptr(x), _ptr(y), int(n), int(mode), _stream(stream)), "attn_debug_exp2", True)


def attn_debug_watchdog(limit_ns, stream=None):
    return _check(lib.attn_debug_watchdog(int(limit_ns), _stream(stream)), "attn_debug_watchdog", True)


def attn_version() -> str:
    return lib.attn_version().decode()
