"""attn_fwd on the GPU against the float64 CPU oracle, element by element.

Small cases span several 128x128 tiles with ragged tails; the full-size workloads
(the same calls the benchmark times) are compared on every row. The bar is
max|dO| <= 1.5e-2 and max|dLSE| <= 2e-3.
"""
import math

import numpy as np
import pytest

import oracle
import synth
from helpers import TOL_LSE, TOL_O, compare, ensure_built, to_dev, tol_o_stress
from synth import workloads as W

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def A():
    ensure_built()
    import exact_softmax_attention_gb300 as mod
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return mod


DEV = "cuda:0"


def run_fwd(A, case, q, k, v):
    Tq, Tk = case.total_q, case.total_k
    o = torch.full((Tq, case.Hq, case.d), float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.full((Tq, case.Hq), float("nan"), dtype=torch.float32, device=DEV)
    cu = None if case.cu_seqlens is None else torch.from_numpy(case.cu_seqlens).to(DEV)
    Nq, Nk = (case.Nq, case.Nk) if cu is None else (Tq, Tk)
    A.attn_fwd(to_dev(q, DEV), to_dev(k, DEV), to_dev(v, DEV), o, lse, case.B, case.Hq, case.Hkv, Nq, Nk, case.d,
               case.scale, case.causal, cu)
    st = A.attn_get_device_status()
    assert st == 0, A.status_string(st)
    return o, lse


def check_full(A, case, stress=False):
    q, k, v = case.generate()
    o, lse = run_fwd(A, case, q, k, v)
    ro, rl = oracle.attn_fwd(q, k, v, case.B, case.Hq, case.Hkv, case.Nq, case.Nk, case.d, case.scale, case.causal,
                             cu_seqlens=case.cu_seqlens)
    do, dl = compare(o, lse, ro, rl)
    tol = tol_o_stress(ro) if stress else TOL_O
    assert do <= tol and dl <= TOL_LSE, f"{case.name}: max|dO|={do:.3e} (bar {tol:.3e}) max|dLSE|={dl:.3e}"
    return do, dl


def case(name, B, Hq, Hkv, Nq, Nk, d, causal, seed, q_mult=1.0, lens=None):
    cu = None
    if lens is not None:
        cu = np.zeros(len(lens) + 1, dtype=np.int32)
        cu[1:] = np.cumsum(lens)
        B = len(lens)
        Nq = Nk = max(max(lens), 1)
    return W.PrefillCase(name, B, Hq, Hkv, Nq, Nk, d, 1.0 / math.sqrt(d), causal, seed, q_mult, cu)


SMALL = [
    case("one_tile", 1, 1, 1, 128, 128, 128, False, 1),
    case("ragged_noncausal", 2, 2, 2, 300, 300, 128, False, 2),
    case("ragged_causal", 2, 2, 1, 333, 333, 128, True, 3),
    case("d64_causal", 1, 4, 2, 700, 700, 64, True, 4),
    case("d64_noncausal", 1, 2, 2, 515, 515, 64, False, 5),
    case("gqa8_causal", 1, 8, 1, 520, 520, 128, True, 6, 2.0),
    case("q_shorter_than_k", 2, 2, 2, 200, 650, 128, True, 7),      # bottom-right: offset 450
    case("q_longer_than_k", 1, 2, 1, 400, 150, 128, True, 8),       # first 250 rows see no key
    case("q_shorter_nc", 1, 2, 2, 77, 1000, 64, False, 9),
    case("single_row", 3, 2, 2, 1, 513, 128, True, 10),
    case("single_key", 1, 2, 2, 257, 1, 128, False, 11),
    case("sharp", 1, 4, 4, 1024, 1024, 128, True, 12, 4.0),         # large scores: many rescales
    # causal with Nq much larger than Nk: whole 256-row blocks see no key at all
    case("no_key_blocks", 1, 2, 2, 600, 100, 128, True, 18),
    case("no_key_blocks_d64", 2, 2, 1, 900, 64, 64, True, 19),
    case("gqa16_causal", 1, 32, 2, 300, 300, 128, True, 20),
    case("mqa32_noncausal", 2, 32, 1, 200, 350, 64, False, 21),
    case("varlen_small", 0, 4, 2, 0, 0, 128, True, 13, lens=[1, 129, 0, 256, 257, 5, 600]),
    case("varlen_d64_nc", 0, 2, 2, 0, 0, 64, False, 14, lens=[300, 17, 128]),
    # more than 32 sequences (several passes of the work-order build), empties and equal lengths
    case("varlen_many_causal", 0, 2, 1, 0, 0, 64, True, 16,
         lens=[int(x) % 7 * 97 for x in synth.uniform_ints(75, 16, 0, 1 << 20)]),
    case("varlen_many_nc", 0, 2, 2, 0, 0, 64, False, 17,
         lens=[int(x) for x in synth.uniform_ints(40, 17, 0, 640)]),
]


@pytest.mark.parametrize("c", SMALL, ids=[c.name for c in SMALL])
def test_small_cases(A, c):
    check_full(A, c, stress=c.q_mult > 2.0)


def test_tiny_workload(A):
    check_full(A, W.tiny())


@pytest.mark.parametrize("causal", [False, True])
def test_prefill_workload(A, causal):
    check_full(A, W.prefill(causal))


def test_long_causal_workload_full(A):
    """The long causal workload (B1 H32 N8192, Q x2) in the call the benchmark times, every row."""
    check_full(A, W.long_causal())


def test_varlen_gqa_workload_full(A):
    """The packed GQA workload (8 sequences U[512, 4096], Hq32 Hkv8), every row."""
    check_full(A, W.varlen_gqa())


def test_varlen_packed_full(A):
    """A shorter packed GQA case compared in full (same recipe, lengths U[100, 700])."""
    lens = synth.uniform_ints(6, 555, 100, 700)
    check_full(A, case("varlen_gqa_reduced", 0, 32, 8, 0, 0, 128, True, 15, lens=list(lens)))


def test_repeatable(A):
    c = case("repeat", 1, 4, 2, 640, 640, 128, True, 16)
    q, k, v = c.generate()
    o1, l1 = run_fwd(A, c, q, k, v)
    o2, l2 = run_fwd(A, c, q, k, v)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("thr", [0.0, 8.0, 20.0])
def test_rescale_threshold_is_exact(A, thr):
    """The threshold only changes when O is rescaled, never the result (beyond rounding)."""
    A.attn_set_option("rescale_threshold", thr)
    try:
        check_full(A, case(f"thr{thr}", 1, 4, 4, 1024, 1024, 128, True, 17, 3.0), stress=True)
    finally:
        A.attn_set_option("rescale_threshold", 8.0)


def test_polynomial_exponentials(A):
    A.attn_set_option("exp_poly", 1)
    try:
        check_full(A, case("poly", 1, 4, 2, 900, 900, 128, True, 18, 2.0))
        check_full(A, case("poly64", 1, 2, 2, 300, 300, 64, False, 19))
    finally:
        A.attn_set_option("exp_poly", 0)


def test_counters_report_skipped_rescales(A):
    c = W.prefill(True)
    q, k, v = c.generate()
    A.attn_set_option("count", 1)
    try:
        A.attn_read_counters()
        run_fwd(A, c, q, k, v)
        dec, res, poly, mufu, dec1, ores = A.attn_read_counters()
        A.attn_set_option("rescale_threshold", 0.0)  # rescale on every increase of a maximum
        run_fwd(A, c, q, k, v)
        _, _, _, _, dec1_0, ores_0 = A.attn_read_counters()
    finally:
        A.attn_set_option("count", 0)
        A.attn_set_option("rescale_threshold", 8.0)
    # one decision per softmax warp and KV tile; first tiles always raise the maximum
    assert dec > 0 and 0 < res < dec
    assert poly == 0 and mufu == dec * 32 * 128
    # every (Q tile, warp) has one first step: 2 tiles x 4 warps per 256-row block
    blocks = c.B * c.Hq * (c.Nq // 256)
    assert dec - dec1 == 8 * blocks and dec1_0 == dec1
    # O rescales are the raised maxima past the first step; the threshold skips most of them
    assert res - ores == 8 * blocks
    assert ores < ores_0 and ores_0 > 0 and ores <= dec1 // 10


@pytest.mark.parametrize("thr", [8.0, 0.0])
@pytest.mark.parametrize("corr,unroll", [(0, 0), (0, 1), (1, 0), (1, 1)])
def test_pipeline_switches_are_exact(A, corr, unroll, thr):
    """The correction role (on or off) and the unroll-KV burst at work-tile boundaries (on or
    off) change only which warp rescales O and when products are issued, never the result
    beyond rounding: each combination matches the oracle, with sharp scores (Q x 4), with
    threshold 0 (a rescale at nearly every step, so the correction warps serve requests from
    both Q tiles all the time), and with many short work tiles per CTA (several 256-row blocks,
    GQA, ragged tails, packed sequences)."""
    A.attn_set_option("correction", corr)
    A.attn_set_option("unroll_kv", unroll)
    A.attn_set_option("rescale_threshold", thr)
    A.attn_set_option("count", 1)
    try:
        A.attn_read_counters()
        tag = f"{corr}{unroll}_{int(thr)}"
        check_full(A, case(f"sw_sharp{tag}", 2, 8, 2, 1300, 1300, 128, True, 40, 4.0), stress=True)
        check_full(A, case(f"sw_nc{tag}", 1, 4, 4, 700, 900, 64, False, 41))
        check_full(A, case(f"sw_varlen{tag}", 0, 4, 1, 0, 0, 128, True, 42, lens=[700, 1, 300, 0, 513, 256]))
        _, _, _, _, dec1, ores = A.attn_read_counters()
        assert ores > 0 and (thr > 0 or ores > dec1 // 4)
    finally:
        A.attn_set_option("correction", 0)
        A.attn_set_option("unroll_kv", 0)
        A.attn_set_option("rescale_threshold", 8.0)
        A.attn_set_option("count", 0)


def test_packed_order_switch_is_exact(A):
    """Sequences in the caller's order (no heaviest-first sort) give the same result."""
    A.attn_set_option("packed_order", 0)
    try:
        check_full(A, W.varlen_gqa())
    finally:
        A.attn_set_option("packed_order", 1)


def test_varlen_more_sequences_than_one_launch(A):
    """1100 packed sequences (lengths 1 .. 64): more than one launch's work-order tables hold, so
    the call runs as two launches (1024 + 76 sequences)."""
    rng = np.random.default_rng(31)
    lens = [int(x) for x in rng.integers(1, 65, size=1100)]
    check_full(A, case("varlen1100", 0, 2, 1, 0, 0, 128, True, 32, lens=lens))
