"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle.

This package only draws random numbers and lays them out; it contains no
attention arithmetic. The generator is splitmix64 used as a counter-based
stream, normals come from Box-Muller pairs in double, and values are rounded
fp32 -> bf16 with round-to-nearest-even (see ``synth.c``). The returned bf16
tensors are numpy ``uint16`` arrays of bit patterns: the CUDA path receives
the same bytes that the CPU oracle reads.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_SO = os.path.join(_OUT_DIR, "libsynth.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``synth.c`` into ``_build/libsynth.so`` (gcc, portable flags)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
             _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            u16p = ctypes.POINTER(ctypes.c_uint16)
            i32p = ctypes.POINTER(ctypes.c_int32)
            lib.synth_normal_bf16.argtypes = [u16p, ctypes.c_int64, ctypes.c_uint64, ctypes.c_double, ctypes.c_int]
            lib.synth_normal_bf16.restype = ctypes.c_int
            lib.synth_uniform_int.argtypes = [i32p, ctypes.c_int64, ctypes.c_uint64, ctypes.c_int32, ctypes.c_int32]
            lib.synth_uniform_int.restype = ctypes.c_int
            lib.synth_permutation.argtypes = [i32p, ctypes.c_int64, ctypes.c_uint64]
            lib.synth_permutation.restype = ctypes.c_int
            lib.synth_splitmix64_at.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
            lib.synth_splitmix64_at.restype = ctypes.c_uint64
            lib.synth_f32_to_bf16.argtypes = [ctypes.c_float]
            lib.synth_f32_to_bf16.restype = ctypes.c_uint16
            _lib = lib
    return _lib


def _threads() -> int:
    return max(1, os.cpu_count() or 1)


def splitmix64_at(seed: int, i: int) -> int:
    """Value ``i`` (0-based) of the splitmix64 stream started from state ``seed``."""
    return int(_load().synth_splitmix64_at(seed & (2**64 - 1), i))


def sub_seed(seed: int, tensor_id: int) -> int:
    """Independent stream seed for tensor ``tensor_id`` of a workload seeded with ``seed``."""
    return splitmix64_at(seed, 1_000_003 + tensor_id)


def normal_bf16(shape, seed: int, mult: float = 1.0, out: np.ndarray | None = None) -> np.ndarray:
    """bf16 bit patterns of ``mult * N(0,1)``; element i (flat, C order) is stream value i."""
    n = int(np.prod(shape)) if len(tuple(shape)) else 1
    if out is None:
        out = np.empty(shape, dtype=np.uint16)
    assert out.dtype == np.uint16 and out.flags.c_contiguous and out.size == n
    rc = _load().synth_normal_bf16(out.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16)), n,
                                   seed & (2**64 - 1), float(mult), _threads())
    if rc != 0:
        raise RuntimeError("synth_normal_bf16 failed")
    return out


def uniform_ints(n: int, seed: int, lo: int, hi: int) -> np.ndarray:
    """``n`` integers, each ``lo + (stream value mod (hi-lo+1))`` (inclusive range)."""
    out = np.empty(n, dtype=np.int32)
    if _load().synth_uniform_int(out.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), n, seed & (2**64 - 1), lo, hi):
        raise RuntimeError("synth_uniform_int failed")
    return out


def permutation(n: int, seed: int) -> np.ndarray:
    """Seeded Fisher-Yates permutation of ``0..n-1`` (int32)."""
    out = np.empty(n, dtype=np.int32)
    if _load().synth_permutation(out.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), n, seed & (2**64 - 1)):
        raise RuntimeError("synth_permutation failed")
    return out


def f32_to_bf16(x) -> np.ndarray:
    """Round fp32 values to bf16 bit patterns (RNE), the same rounding the generator uses."""
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    b = a.view(np.uint32).astype(np.uint64)
    nan = (b & 0x7F800000) == 0x7F800000
    nan &= (b & 0x007FFFFF) != 0
    r = ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint16)
    r[nan] = 0x7FC0
    return r


def bf16_to_f32(h: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# ----------------------------------------------------------------------------- FP8 inputs
# The OCP 8-bit floating-point formats, used to lay out 8-bit key/value caches:
#   e4m3: 4 exponent bits (bias 7), 3 mantissa bits, no infinities, S.1111.111 is NaN
#   e5m2: 5 exponent bits (bias 15), 2 mantissa bits, exponent 31 is infinity or NaN
_FP8_FORMATS = {"e4m3": (3, 7), "e5m2": (2, 15)}
FP8_MAX = {"e4m3": 448.0, "e5m2": 57344.0}


def _fp8_finite_values(fmt: str) -> np.ndarray:
    """Values of the non-negative finite codes 0, 1, 2, ... of ``fmt`` (ascending with the code)."""
    m_bits, bias = _FP8_FORMATS[fmt]
    codes = np.arange(128, dtype=np.int64)
    e = codes >> m_bits
    m = (codes & ((1 << m_bits) - 1)).astype(np.float64) / (1 << m_bits)
    val = np.where(e == 0, m * 2.0 ** (1 - bias), (1.0 + m) * np.exp2((e - bias).astype(np.float64)))
    n_finite = 127 if fmt == "e4m3" else 124
    return val[:n_finite]


def fp8_encode(x, fmt: str) -> np.ndarray:
    """Round values to FP8 codes (uint8): nearest, ties to the even code, saturating at the
    largest finite value. Only lays out inputs; nothing reads these values but the kernels
    and the oracle, each through its own decoding."""
    v = _fp8_finite_values(fmt)
    xs = np.asarray(x, dtype=np.float64)
    a = np.abs(xs).ravel()
    i = np.clip(np.searchsorted(v, a), 1, len(v) - 1)  # v[i-1] < a <= v[i] inside the range
    lo, hi = v[i - 1], v[i]
    up = (a - lo > hi - a) | ((a - lo == hi - a) & (i % 2 == 0))
    code = np.where(up, i, i - 1)
    code = np.where(a >= v[-1], len(v) - 1, code)
    sign = np.signbit(xs).ravel().astype(np.uint8) << 7
    return (code.astype(np.uint8) | sign).reshape(xs.shape)
