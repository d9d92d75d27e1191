"""attn_fwd_fp8 (Q/K/V as 8-bit floating-point codes with per-tensor descales) on the GPU
against the float64 CPU oracle, which decodes the codes from the OCP FP8 definitions and
applies the descales before the same three-pass definition."""
import math

import numpy as np
import pytest

import oracle
import synth
from helpers import TOL_LSE, TOL_O, compare, ensure_built
from synth import workloads as W

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def A():
    ensure_built()
    import exact_softmax_attention_gb300 as mod
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return mod


def case(name, B, Hq, Hkv, Nq, Nk, causal, seed, q_mult=1.0, lens=None):
    cu = None
    if lens is not None:
        cu = np.zeros(len(lens) + 1, dtype=np.int32)
        cu[1:] = np.cumsum(lens)
        B, Nq, Nk = len(lens), int(cu[-1]), int(cu[-1])
    return W.PrefillCase(name, B, Hq, Hkv, Nq, Nk, 128, 1.0 / math.sqrt(128), causal, seed, q_mult, cu)


def run(A, c, fmt, q8, k8, v8, qs, ks, vs):
    o = torch.full((c.total_q, c.Hq, c.d), float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.full((c.total_q, c.Hq), float("nan"), dtype=torch.float32, device=DEV)
    cu = None if c.cu_seqlens is None else torch.from_numpy(c.cu_seqlens).to(DEV)
    Nq, Nk = (c.Nq, c.Nk) if cu is None else (c.total_q, c.total_k)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    A.attn_fwd_fp8(dev(q8), dev(k8), dev(v8), o, lse, c.B, c.Hq, c.Hkv, Nq, Nk, c.d, c.scale, c.causal, cu, None,
                   fmt, qs, ks, vs)
    st = A.attn_get_device_status()
    assert st == 0, A.status_string(st)
    return o, lse


def check(A, c, fmt, rows=None):
    q8, k8, v8, qs, ks, vs = c.generate_fp8(fmt)
    o, lse = run(A, c, fmt, q8, k8, v8, qs, ks, vs)
    ro, rl = oracle.attn_fwd_fp8(q8, k8, v8, fmt, qs, ks, vs, c.B, c.Hq, c.Hkv, c.Nq, c.Nk, c.d, c.scale, c.causal,
                                 cu_seqlens=c.cu_seqlens, rows=rows)
    if rows is not None:
        sel = torch.from_numpy(rows).to(DEV)
        assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
        o, lse = o.reshape(-1, c.d)[sel], lse.reshape(-1)[sel]
    do, dl = compare(o, lse, ro, rl)
    assert do <= TOL_O and dl <= TOL_LSE, f"{c.name} {fmt}: max|dO|={do:.3e} max|dLSE|={dl:.3e}"


CASES = [
    case("one_tile", 1, 1, 1, 128, 128, False, 41),
    case("ragged_noncausal", 2, 2, 2, 300, 300, False, 42),
    case("ragged_causal_gqa", 2, 4, 1, 333, 333, True, 43),
    case("q_shorter_than_k", 2, 2, 2, 200, 650, True, 44),
    case("no_key_blocks", 1, 2, 2, 600, 100, True, 45),
    case("sharp", 1, 4, 4, 1024, 1024, True, 46, 3.0),
    case("varlen", 0, 4, 2, 0, 0, True, 47, lens=[1, 129, 0, 256, 257, 5, 600]),
    case("gqa16", 1, 32, 2, 300, 300, True, 50),
]


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("c", CASES, ids=[c.name for c in CASES])
def test_fp8_forward_cases(A, c, fmt):
    check(A, c, fmt)


def test_fp8_forward_prefill_workload(A):
    c = W.prefill(True)
    check(A, c, "e4m3")


def test_fp8_forward_long_causal_full(A):
    """The long causal workload (B1 H32 N8192, Q x2) with e4m3 inputs, every row."""
    check(A, W.long_causal(), "e4m3")


def test_fp8_forward_descales(A):
    """Other descales change the GPU result exactly as they change the oracle's."""
    c = case("descale", 1, 2, 2, 256, 256, True, 48)
    q8, k8, v8, _, _, _ = c.generate_fp8("e4m3")
    for qs, ks, vs in ((0.002, 0.01, 0.004), (0.01, 0.004, 5.0)):
        o, lse = run(A, c, "e4m3", q8, k8, v8, qs, ks, vs)
        ro, rl = oracle.attn_fwd_fp8(q8, k8, v8, "e4m3", qs, ks, vs, c.B, c.Hq, c.Hkv, c.Nq, c.Nk, c.d, c.scale,
                                     c.causal)
        do, dl = compare(o, lse, ro, rl)
        tol = TOL_O * max(1.0, float(np.abs(ro).max()))  # bf16 output rounding grows with |O|
        assert do <= tol and dl <= TOL_LSE, f"descales {qs},{ks},{vs}: {do:.3e} {dl:.3e}"


def test_fp8_forward_rejects_bad_arguments(A):
    c = case("bad", 1, 2, 2, 128, 128, False, 49)
    q8, k8, v8, qs, ks, vs = c.generate_fp8("e4m3")
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    o = torch.full((c.total_q, c.Hq, c.d), float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.full((c.total_q, c.Hq), float("nan"), dtype=torch.float32, device=DEV)
    for fmt, d, q_, code in ((2, 128, qs, A.ATTN_ERR_BAD_ARG), (0, 64, qs, A.ATTN_ERR_BAD_SHAPE),
                             (0, 128, float("nan"), A.ATTN_ERR_BAD_ARG)):
        rc = A.attn_fwd_fp8(dev(q8), dev(k8), dev(v8), o, lse, c.B, c.Hq, c.Hkv, c.Nq, c.Nk, d, c.scale, False, None,
                            None, fmt, q_, ks, vs, raise_on_error=False)
        assert rc == code
    torch.cuda.synchronize()
    assert torch.isnan(o.float()).all()
