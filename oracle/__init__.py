"""CPU oracle for exact softmax attention: TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference legs may import this package. The product path never calls it, and
it shares no code with the CUDA library.

Contents
--------
``attn_fwd`` / ``attn_decode_paged``
    The plain definition in float64, three passes per row (``attn_oracle.c``),
    following "FlashAttention: not computing less, moving less", sections 01-02
    (formula and online-softmax equivalence) and section 03 (LSE output); paged
    decode per "Faster, more flexible FA4 for LLM inference" (PR 1999/2104 page
    gathering, PR 1940 split-KV), with the page table resolved first.
``attn_decode_paged_fp8`` / ``fp8_values``
    Paged decode over 8-bit floating-point caches ("Faster, more flexible FA4
    for LLM inference", PR 2109: e4m3 or e5m2 inputs). The codes are decoded
    from the OCP 8-bit floating-point definitions and multiplied by one descale
    factor per tensor (a reading: the pages fix no scaling scheme), then the
    same three-pass definition runs in float64.
``attn_fwd_f64`` / ``attn_fwd_fp8``
    The forward definition on float64 inputs, also with values (and outputs)
    narrower than queries and keys, e.g. head dims (192, 128) ("FlashAttention-4:
    Blackwell algorithm-pipeline co-design", performance section); ``attn_fwd_fp8`` decodes 8-bit
    floating-point Q/K/V codes (PR 2109 of the same page) and applies one descale
    per tensor before it.
``online_attention``
    The streaming recurrence of "FlashAttention: not computing less, moving
    less", section 02 (running max m, sum l, unnormalised accumulator a,
    rescale by exp(m - m')), with the conditional rescale of "FlashAttention-4:
    Blackwell algorithm-pipeline co-design", section "conditional softmax
    rescaling", and "FlashAttention4 精读" section 3.1.4 (threshold, warp-uniform
    decision). Used to show the recurrence reaches the three-pass result.
``exp2_poly`` and friends
    The software exponential of the hybrid-exponential sections
    (``exp2_poly.c``).

Readings of the pages taken here (the pages are silent or garbled):
 * causal masks are bottom-right aligned (key j visible to row i iff
   j <= i + Nk - Nq); a row with no visible key gives o = 0, lse = -inf;
 * LSE is the natural log of the sum of exp of the *scaled* scores;
 * query head h uses key/value head h // (Hq // Hkv);
 * the rescale threshold "256" is a factor on the exponentials, i.e.
   tau = log2(256) = 8 in the base-2 exponent domain;
 * an FP8 cache holds one descale factor per tensor: code c stands for
   descale * fp8(c).

Every function here is pinned by tests against values the pages print, closed
forms, invariants and an independent library routine (see ``tests/test_oracle.py``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRCS = [os.path.join(_HERE, "attn_oracle.c"), os.path.join(_HERE, "exp2_poly.c")]
_OUT_DIR = os.path.join(_HERE, "_build")
_SO = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

LOG2E = 1.4426950408889634


def build(force: bool = False) -> str:
    """Compile the C oracle into ``_build/liboracle.so`` with plain gcc flags."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    newest = max(os.path.getmtime(s) for s in _SRCS)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < newest:
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
                               *_SRCS, "-o", tmp, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            vp = ctypes.c_void_p
            i, i64, d = ctypes.c_int, ctypes.c_int64, ctypes.c_double
            lib.oracle_attn_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, d, i, vp, vp, i64, i]
            lib.oracle_attn_fwd.restype = i
            lib.oracle_attn_decode_paged.argtypes = [vp, vp, vp, vp, vp, i, vp, vp, i, i, i, i, i, d, i]
            lib.oracle_attn_decode_paged.restype = i
            lib.oracle_attn_decode_paged_fp8.argtypes = [vp, vp, vp, i, d, d, vp, vp, i, vp, vp, i, i, i, i, i, d, i]
            lib.oracle_attn_decode_paged_fp8.restype = i
            lib.oracle_attn_fwd_f64.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, d, i, vp, vp, i64, i]
            lib.oracle_attn_fwd_f64.restype = i
            lib.oracle_fp8_values.argtypes = [vp, vp, i64, i]
            lib.oracle_fp8_values.restype = None
            lib.oracle_exp2_poly.argtypes = [ctypes.c_float]
            lib.oracle_exp2_poly.restype = ctypes.c_float
            lib.oracle_floor_magic.argtypes = [ctypes.c_float]
            lib.oracle_floor_magic.restype = ctypes.c_float
            lib.oracle_exp2_cubic.argtypes = [ctypes.c_float]
            lib.oracle_exp2_cubic.restype = ctypes.c_float
            lib.oracle_exp2_poly_batch.argtypes = [vp, vp, i64]
            lib.oracle_exp2_poly_batch.restype = None
            lib.oracle_exp2_cubic_sweep.argtypes = [i, i, ctypes.POINTER(d), ctypes.POINTER(d),
                                                    ctypes.POINTER(ctypes.c_float)]
            lib.oracle_exp2_cubic_sweep.restype = i
            _lib = lib
    return _lib


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def _u16(a, name):
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError(f"{name}: expected bf16 bit patterns as uint16, got {a.dtype}")
    return a


def attn_fwd(q, k, v, B, Hq, Hkv, Nq, Nk, d, scale, causal, cu_seqlens=None, rows=None, n_threads=None):
    """Exact attention forward in float64.

    q: uint16 [T, Hq, d]; k, v: uint16 [Tk, Hkv, d] (bf16 bits). ``cu_seqlens``
    (int32 [B+1], host) selects packed variable-length sequences. ``rows`` is an
    optional int64 list of ``token * Hq + head`` rows to compute; then o is
    ``[len(rows), d]`` and lse ``[len(rows)]``, else o is ``[T, Hq, d]``, lse ``[T, Hq]``.
    """
    q, k, v = _u16(q, "q"), _u16(k, "k"), _u16(v, "v")
    cu = None if cu_seqlens is None else np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    T = int(cu[-1]) if cu is not None else B * Nq
    if rows is None:
        o = np.zeros((T, Hq, d), dtype=np.float64)
        lse = np.zeros((T, Hq), dtype=np.float64)
        rp, nr = None, 0
    else:
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        o = np.zeros((len(rows), d), dtype=np.float64)
        lse = np.zeros((len(rows),), dtype=np.float64)
        rp, nr = rows.ctypes.data, len(rows)
    rc = _load().oracle_attn_fwd(q.ctypes.data, k.ctypes.data, v.ctypes.data, o.ctypes.data, lse.ctypes.data,
                                 B, Hq, Hkv, Nq, Nk, d, float(scale), int(bool(causal)),
                                 None if cu is None else cu.ctypes.data, rp, nr,
                                 n_threads or default_threads())
    if rc != 0:
        raise ValueError(f"oracle_attn_fwd rejected its arguments (rc={rc})")
    return o, lse


def attn_fwd_f64(q, k, v, B, Hq, Hkv, Nq, Nk, d, scale, causal, cu_seqlens=None, rows=None, n_threads=None, dv=None):
    """attn_fwd on float64 inputs (same layouts, masks and ``rows`` as ``attn_fwd``). ``dv``
    (default ``d``) is the value / output width: q, k are d wide, v and o dv wide."""
    dv = d if dv is None else dv
    q, k, v = (np.ascontiguousarray(a, dtype=np.float64) for a in (q, k, v))
    cu = None if cu_seqlens is None else np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    T = int(cu[-1]) if cu is not None else B * Nq
    if rows is None:
        o = np.zeros((T, Hq, dv), dtype=np.float64)
        lse = np.zeros((T, Hq), dtype=np.float64)
        rp, nr = None, 0
    else:
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        o = np.zeros((len(rows), dv), dtype=np.float64)
        lse = np.zeros((len(rows),), dtype=np.float64)
        rp, nr = rows.ctypes.data, len(rows)
    rc = _load().oracle_attn_fwd_f64(q.ctypes.data, k.ctypes.data, v.ctypes.data, o.ctypes.data, lse.ctypes.data,
                                     B, Hq, Hkv, Nq, Nk, d, dv, float(scale), int(bool(causal)),
                                     None if cu is None else cu.ctypes.data, rp, nr, n_threads or default_threads())
    if rc != 0:
        raise ValueError(f"oracle_attn_fwd_f64 rejected its arguments (rc={rc})")
    return o, lse


def attn_fwd_fp8(q, k, v, fmt, q_descale, k_descale, v_descale, B, Hq, Hkv, Nq, Nk, d, scale, causal,
                 cu_seqlens=None, rows=None, n_threads=None):
    """attn_fwd on 8-bit floating-point Q/K/V codes (uint8, OCP e4m3 or e5m2), each tensor
    standing for its descale times the decoded values."""
    qf = q_descale * fp8_values(q, fmt)
    kf = k_descale * fp8_values(k, fmt)
    vf = v_descale * fp8_values(v, fmt)
    return attn_fwd_f64(qf, kf, vf, B, Hq, Hkv, Nq, Nk, d, scale, causal, cu_seqlens, rows, n_threads)


def attn_decode_paged(q, k_cache, v_cache, page_table, seqlens, page_size, B, Hq, Hkv, d, max_pages, scale,
                      n_threads=None):
    """Single-query paged attention in float64: q [B, Hq, d], caches [pages, page_size, Hkv, d]."""
    q, kc, vc = _u16(q, "q"), _u16(k_cache, "k_cache"), _u16(v_cache, "v_cache")
    pt = np.ascontiguousarray(page_table, dtype=np.int32)
    sl = np.ascontiguousarray(seqlens, dtype=np.int32)
    o = np.zeros((B, Hq, d), dtype=np.float64)
    lse = np.zeros((B, Hq), dtype=np.float64)
    rc = _load().oracle_attn_decode_paged(q.ctypes.data, kc.ctypes.data, vc.ctypes.data, pt.ctypes.data,
                                          sl.ctypes.data, page_size, o.ctypes.data, lse.ctypes.data,
                                          B, Hq, Hkv, d, max_pages, float(scale), n_threads or default_threads())
    if rc != 0:
        raise ValueError(f"oracle_attn_decode_paged rejected its arguments (rc={rc})")
    return o, lse


FP8_FORMATS = {"e4m3": 0, "e5m2": 1}


def fp8_values(codes, fmt: str) -> np.ndarray:
    """float64 values of FP8 codes (OCP e4m3 or e5m2), as decoded by the oracle."""
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.empty(c.shape, dtype=np.float64)
    _load().oracle_fp8_values(c.ctypes.data, out.ctypes.data, c.size, FP8_FORMATS[fmt])
    return out


def attn_decode_paged_fp8(q, k_cache, v_cache, fmt, k_descale, v_descale, page_table, seqlens, page_size, B, Hq,
                          Hkv, d, max_pages, scale, n_threads=None):
    """Single-query paged attention in float64 over FP8 caches: q bf16 [B, Hq, d]; caches
    FP8 codes [pages, page_size, Hkv, d] standing for descale * fp8(code)."""
    q = _u16(q, "q")
    kc = np.ascontiguousarray(k_cache, dtype=np.uint8)
    vc = np.ascontiguousarray(v_cache, dtype=np.uint8)
    pt = np.ascontiguousarray(page_table, dtype=np.int32)
    sl = np.ascontiguousarray(seqlens, dtype=np.int32)
    o = np.zeros((B, Hq, d), dtype=np.float64)
    lse = np.zeros((B, Hq), dtype=np.float64)
    rc = _load().oracle_attn_decode_paged_fp8(q.ctypes.data, kc.ctypes.data, vc.ctypes.data, FP8_FORMATS[fmt],
                                              float(k_descale), float(v_descale), pt.ctypes.data, sl.ctypes.data,
                                              page_size, o.ctypes.data, lse.ctypes.data, B, Hq, Hkv, d, max_pages,
                                              float(scale), n_threads or default_threads())
    if rc != 0:
        raise ValueError(f"oracle_attn_decode_paged_fp8 rejected its arguments (rc={rc})")
    return o, lse


# ----------------------------------------------------------------- exp2 model

def exp2_poly(x) -> np.ndarray:
    """Software 2^x (clamp, magic-bias floor, cubic Horner, exponent add) on fp32 inputs."""
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    y = np.empty_like(x)
    _load().oracle_exp2_poly_batch(x.ctypes.data, y.ctypes.data, x.size)
    return y


def floor_magic(x: float) -> float:
    """n = (x + 1.5*2^23) - 1.5*2^23 with the add rounded toward minus infinity."""
    return float(_load().oracle_floor_magic(float(x)))


def exp2_cubic(f: float) -> float:
    """The fp32 Horner cubic approximating 2^f on [0, 1)."""
    return float(_load().oracle_exp2_cubic(float(f)))


def exp2_cubic_sweep(mode: int, n_threads=None):
    """(max, mean, argmax) relative error of the cubic vs exp2 in double.

    mode 0: every fp32 value in [0, 1); mode 1: uniform grid i / 2^24."""
    mx, mean, arg = ctypes.c_double(), ctypes.c_double(), ctypes.c_float()
    _load().oracle_exp2_cubic_sweep(mode, n_threads or default_threads(), ctypes.byref(mx), ctypes.byref(mean),
                                    ctypes.byref(arg))
    return mx.value, mean.value, arg.value


# ------------------------------------------------------ streaming recurrence

def online_attention(s_blocks, v_blocks, tau=0.0, group=1, history=False):
    """Online-softmax recurrence over key blocks, float64.

    s_blocks: list of arrays [R, n_b] of *scaled* scores (-inf = masked);
    v_blocks: list of arrays [n_b, dv]. For every block, per row:
        m_cand = max(m, max_j s_j)
        rescale if m is -inf or (m_cand - m) * log2(e) > tau  (tau in base-2 exponent units);
        rows are taken in groups of ``group``: if any row of a group rescales, all of them do
        m'  = m_cand if rescaling else m
        l'  = exp(m - m') l + sum_j exp(s_j - m')
        a'  = exp(m - m') a + sum_j exp(s_j - m') v_j
    and finally o = a / l, lse = m + ln l (o = 0, lse = -inf for rows with l = 0).
    Returns (o [R, dv], lse [R]) and, with ``history=True``, the per-block (m, l, a) states.
    """
    R = s_blocks[0].shape[0]
    dv = v_blocks[0].shape[1]
    m = np.full(R, -np.inf)
    l = np.zeros(R)
    a = np.zeros((R, dv))
    hist = []
    for s, vb in zip(s_blocks, v_blocks):
        s = np.asarray(s, dtype=np.float64)
        vb = np.asarray(vb, dtype=np.float64)
        m_cand = np.maximum(m, s.max(axis=1) if s.shape[1] else -np.inf)
        with np.errstate(invalid="ignore"):
            need = (m_cand - m) * LOG2E > tau  # NaN (both -inf) compares False
        if group > 1:
            g = need.reshape(-1, group) if R % group == 0 else None
            if g is None:
                raise ValueError("row count must be a multiple of group")
            need = np.repeat(g.any(axis=1), group)
        m_new = np.where(need, m_cand, m)
        with np.errstate(invalid="ignore"):
            alpha = np.where(np.isneginf(m_new), 1.0, np.exp(m - m_new))
            p = np.where(np.isneginf(s), 0.0, np.exp(s - np.where(np.isneginf(m_new), 0.0, m_new)[:, None]))
        l = alpha * l + p.sum(axis=1)
        a = alpha[:, None] * a + p @ vb
        m = m_new
        if history:
            hist.append((m.copy(), l.copy(), a.copy()))
    with np.errstate(invalid="ignore", divide="ignore"):
        o = np.where(l[:, None] > 0, a / np.where(l > 0, l, 1.0)[:, None], 0.0)
        lse = np.where(l > 0, m + np.log(np.where(l > 0, l, 1.0)), -np.inf)
    return (o, lse, hist) if history else (o, lse)


def scores_dense(q, k, scale, causal, Nq, Nk, G):
    """Scaled scores for one sequence: q [Nq, Hq, d], k [Nk, Hkv, d] (float64) -> [Hq, Nq, Nk] with -inf masked."""
    qd = np.asarray(q, dtype=np.float64)
    kd = np.repeat(np.asarray(k, dtype=np.float64), G, axis=1)
    s = np.einsum("ihc,jhc->hij", qd, kd) * scale
    if causal:
        i = np.arange(Nq)[:, None]
        j = np.arange(Nk)[None, :]
        s = np.where(j <= i + (Nk - Nq), s, -np.inf)
    return s
