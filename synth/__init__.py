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
