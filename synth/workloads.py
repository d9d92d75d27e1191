"""Workload recipes: shapes, seeds, lengths and page tables of the attention workloads.

Only layout and random draws live here, plus the algorithmic work counts
(FLOPs and bytes) used for throughput and roofline figures. There is no
attention arithmetic in this module.

Recipes (inputs i.i.d. N(0,1) rounded to bf16 unless stated):
  tiny        B=1, H=2, N=256, d=64, scale 1/8, non-causal
  prefill     B=2, H=16, N=2048, d=128, scale 1/sqrt(128), non-causal and causal
  long_causal B=1, H=32, N=8192, d=128, Q multiplied by 2 before rounding, causal
  varlen_gqa  8 packed sequences, lengths U[512, 4096], Hq=32, Hkv=8, d=128, causal
  decode      B=64, Hq=32, Hkv=8, d=128, lengths U[1024, 32768], page_size=16,
              physical pages placed by a seeded permutation of the pool
  decode_fp8  the decode workload with e4m3 key/value caches: the same N(0,1) draws,
              divided by a per-tensor descale (max |x| / 448) and rounded to e4m3
Seeds are ``20261202 + index`` in that order; each tensor draws from its own sub-stream.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

from . import FP8_MAX, bf16_to_f32, fp8_encode, normal_bf16, permutation, sub_seed, uniform_ints

BASE_SEED = 20261202

# sub-stream ids
_Q, _K, _V, _LEN, _PERM = 0, 1, 2, 3, 4


def _to_fp8(c: np.ndarray, fmt: str):
    """bf16 bit patterns -> (FP8 codes, per-tensor descale): descale = max |x| / largest
    finite FP8 value (float32); codes = round(x / descale). The code of an element depends
    only on its bf16 bit pattern, so all 65536 patterns are encoded once and gathered."""
    mag = c.reshape(-1) & np.uint16(0x7FFF)
    top = int(mag.max()) if mag.size else 0  # |x| orders like its magnitude bits (no NaN inputs)
    amax = float(bf16_to_f32(np.array([top], dtype=np.uint16))[0])
    ds = float(np.float32(amax / FP8_MAX[fmt])) if amax > 0 else 1.0
    with np.errstate(invalid="ignore"):
        vals = bf16_to_f32(np.arange(65536, dtype=np.uint32).astype(np.uint16)).astype(np.float64)
    vals[~np.isfinite(vals)] = 0.0  # NaN / inf patterns: not produced by the generator
    table = fp8_encode(vals / ds, fmt)
    return table[c], ds


@dataclasses.dataclass
class PrefillCase:
    name: str
    B: int
    Hq: int
    Hkv: int
    Nq: int
    Nk: int
    d: int
    scale: float
    causal: bool
    seed: int
    q_mult: float = 1.0
    cu_seqlens: np.ndarray | None = None  # int32 [B+1] for packed sequences
    dv: int | None = None  # value / output width when it differs from d (e.g. d = 192, dv = 128)

    @property
    def d_v(self) -> int:
        return self.d if self.dv is None else self.dv

    @property
    def total_q(self) -> int:
        return int(self.cu_seqlens[-1]) if self.cu_seqlens is not None else self.B * self.Nq

    @property
    def total_k(self) -> int:
        return int(self.cu_seqlens[-1]) if self.cu_seqlens is not None else self.B * self.Nk

    def generate_fp8(self, fmt: str = "e4m3"):
        """(q, k, v as FP8 codes (uint8), q_descale, k_descale, v_descale): the bf16 case's
        draws divided by a per-tensor descale (max |x| / largest finite FP8 value, float32)
        and rounded to FP8."""
        (q8, qd), (k8, kd), (v8, vd) = (_to_fp8(c, fmt) for c in self.generate())
        return q8, k8, v8, qd, kd, vd

    def generate(self):
        """(q [Tq, Hq, d], k [Tk, Hkv, d], v [Tk, Hkv, d]) as bf16 bit patterns (uint16)."""
        q = normal_bf16((self.total_q, self.Hq, self.d), sub_seed(self.seed, _Q), self.q_mult)
        k = normal_bf16((self.total_k, self.Hkv, self.d), sub_seed(self.seed, _K))
        v = normal_bf16((self.total_k, self.Hkv, self.d_v), sub_seed(self.seed, _V))
        return q, k, v

    def seq_lens(self):
        if self.cu_seqlens is not None:
            c = self.cu_seqlens.astype(np.int64)
            return [(int(c[b + 1] - c[b]), int(c[b + 1] - c[b])) for b in range(self.B)]
        return [(self.Nq, self.Nk)] * self.B

    def visible_pairs(self) -> int:
        """Number of (query row, key) pairs that are not masked, summed over sequences (one head)."""
        total = 0
        for nq, nk in self.seq_lens():
            if not self.causal:
                total += nq * nk
            else:
                i = np.arange(nq, dtype=np.int64)
                total += int(np.clip(i + (nk - nq) + 1, 0, nk).sum())
        return total

    def flops(self) -> int:
        """Algorithmic FLOPs per visible pair and query head: 2*d for QK^T and 2*dv for PV."""
        return 2 * (self.d + self.d_v) * self.Hq * self.visible_pairs()

    def bytes(self) -> int:
        """Algorithmic HBM bytes: read q, k, v once and write o (bf16) and lse (fp32) once."""
        return ((self.total_q * self.Hq * (self.d + self.d_v) + self.total_k * self.Hkv * (self.d + self.d_v)) * 2
                + 4 * self.total_q * self.Hq)


@dataclasses.dataclass
class DecodeCase:
    name: str
    B: int
    Hq: int
    Hkv: int
    d: int
    page_size: int
    seqlens: np.ndarray  # int32 [B]
    max_pages: int
    scale: float
    seed: int
    extra_pages: int = 0  # unreferenced pool pages (for canary tests)
    kv_fmt: str = "bf16"  # cache element format: "bf16", or FP8 "e4m3" / "e5m2"

    @property
    def pages_per_seq(self) -> np.ndarray:
        return (self.seqlens.astype(np.int64) + self.page_size - 1) // self.page_size

    @property
    def num_pages(self) -> int:
        return int(self.pages_per_seq.sum()) + self.extra_pages

    def page_table(self) -> np.ndarray:
        """int32 [B, max_pages]; logical page p of sequence b maps to a permuted physical page.

        Entries past a sequence's last page are 0 (never read)."""
        perm = permutation(self.num_pages, sub_seed(self.seed, _PERM))
        pt = np.zeros((self.B, self.max_pages), dtype=np.int32)
        off = 0
        for b, n in enumerate(self.pages_per_seq):
            pt[b, :n] = perm[off:off + n]
            off += int(n)
        return pt

    def generate(self):
        """(q [B, Hq, d], k_cache, v_cache [num_pages, page_size, Hkv, d], page_table, seqlens)."""
        q = normal_bf16((self.B, self.Hq, self.d), sub_seed(self.seed, _Q))
        shape = (self.num_pages, self.page_size, self.Hkv, self.d)
        kc = normal_bf16(shape, sub_seed(self.seed, _K))
        vc = normal_bf16(shape, sub_seed(self.seed, _V))
        return q, kc, vc, self.page_table(), self.seqlens.copy()

    def generate_fp8(self):
        """(q, k_cache, v_cache (uint8 FP8 codes), page_table, seqlens, k_descale, v_descale).

        The cache values are the bf16 case's draws divided by a per-tensor descale
        (max |x| / largest finite FP8 value, as float32) and rounded to FP8, so that the
        cached key with code c stands for k_descale * fp8(c)."""
        q, kc, vc, pt, sl = self.generate()
        (kc8, kds), (vc8, vds) = (_to_fp8(c, self.kv_fmt) for c in (kc, vc))
        return q, kc8, vc8, pt, sl, kds, vds

    def flops(self) -> int:
        return 4 * self.d * self.Hq * int(self.seqlens.astype(np.int64).sum())

    def bytes(self) -> int:
        """Algorithmic HBM bytes: every cached K and V row of every sequence once, q, o, lse,
        the page-table entries in use and seqlens. Split-KV workspace traffic is not counted."""
        L = self.seqlens.astype(np.int64)
        elem = 2 if self.kv_fmt == "bf16" else 1
        kv = int(L.sum()) * self.Hkv * self.d * elem * 2
        qo = 2 * self.B * self.Hq * self.d * 2
        lse = self.B * self.Hq * 4
        pt = int(self.pages_per_seq.sum()) * 4
        return kv + qo + lse + pt + self.B * 4


def _cu(lengths) -> np.ndarray:
    cu = np.zeros(len(lengths) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(np.asarray(lengths, dtype=np.int64))
    return cu


def tiny() -> PrefillCase:
    return PrefillCase("tiny", 1, 2, 2, 256, 256, 64, 1.0 / 8.0, False, BASE_SEED + 0)


def prefill(causal: bool) -> PrefillCase:
    return PrefillCase("prefill_causal" if causal else "prefill", 2, 16, 16, 2048, 2048, 128,
                       1.0 / math.sqrt(128), causal, BASE_SEED + 1)


def long_causal() -> PrefillCase:
    return PrefillCase("long_causal", 1, 32, 32, 8192, 8192, 128, 1.0 / math.sqrt(128), True, BASE_SEED + 2,
                       q_mult=2.0)


def varlen_gqa() -> PrefillCase:
    seed = BASE_SEED + 3
    lens = uniform_ints(8, sub_seed(seed, _LEN), 512, 4096)
    cu = _cu(lens)
    return PrefillCase("varlen_gqa", 8, 32, 8, int(lens.max()), int(lens.max()), 128, 1.0 / math.sqrt(128), True,
                       seed, cu_seqlens=cu)


def decode() -> DecodeCase:
    seed = BASE_SEED + 4
    lens = uniform_ints(64, sub_seed(seed, _LEN), 1024, 32768)
    return DecodeCase("decode", 64, 32, 8, 128, 16, lens, 32768 // 16, 1.0 / math.sqrt(128), seed)


def decode_fp8() -> DecodeCase:
    c = decode()
    return dataclasses.replace(c, name="decode_fp8", kv_fmt="e4m3")


def all_prefill():
    return [tiny(), prefill(False), prefill(True), long_causal(), varlen_gqa()]
