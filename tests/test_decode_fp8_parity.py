"""attn_decode_paged_fp8 (8-bit floating-point key/value caches) on the GPU against the float64
CPU oracle, which decodes the codes from the OCP FP8 definitions and applies the descales."""
import math

import numpy as np
import pytest

import oracle
import synth
from helpers import TOL_LSE, TOL_O, compare, ensure_built, to_dev
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


def run(A, c, q, kc8, vc8, pt, sl, kds, vds, num_splits=0):
    o = torch.full((c.B, c.Hq, c.d), float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.full((c.B, c.Hq), float("nan"), dtype=torch.float32, device=DEV)
    A.attn_decode_paged_fp8(to_dev(q, DEV), torch.from_numpy(kc8).to(DEV), torch.from_numpy(vc8).to(DEV),
                            torch.from_numpy(pt).to(DEV), torch.from_numpy(sl).to(DEV), c.page_size, o, lse, None,
                            c.B, c.Hq, c.Hkv, c.d, c.max_pages, c.num_pages, c.scale, num_splits, c.kv_fmt, kds, vds)
    assert A.attn_get_device_status() == 0
    return o, lse


def reference(c, q, kc8, vc8, pt, sl, kds, vds, rows=None):
    if rows is None:
        rows = np.arange(c.B)
    return oracle.attn_decode_paged_fp8(q[rows], kc8, vc8, c.kv_fmt, kds, vds, pt[rows], sl[rows], c.page_size,
                                        len(rows), c.Hq, c.Hkv, c.d, c.max_pages, c.scale)


def fcase(name, B, Hq, Hkv, d, page_size, lo, hi, seed, fmt, extra=0, lens=None):
    if lens is None:
        lens = synth.uniform_ints(B, seed, lo, hi)
    lens = np.asarray(lens, dtype=np.int32)
    max_pages = int((max(int(lens.max()), 1) + page_size - 1) // page_size) + 2
    return W.DecodeCase(name, len(lens), Hq, Hkv, d, page_size, lens, max_pages, 1.0 / math.sqrt(d), seed,
                        extra_pages=extra, kv_fmt=fmt)


CASES = [
    (fcase("e4m3_p16_g4", 9, 32, 8, 128, 16, 1, 3000, 21, "e4m3"), 0),
    (fcase("e5m2_p16_g4", 9, 32, 8, 128, 16, 1, 3000, 22, "e5m2"), 0),
    (fcase("e4m3_split3", 5, 8, 2, 128, 16, 500, 2500, 23, "e4m3"), 3),
    (fcase("e4m3_p1", 4, 8, 2, 128, 1, 1, 700, 24, "e4m3"), 0),
    (fcase("e5m2_p7_d64", 6, 12, 3, 64, 7, 1, 1500, 25, "e5m2"), 0),
    (fcase("e4m3_d64_g16", 3, 16, 1, 64, 16, 100, 5000, 26, "e4m3"), 0),
    (fcase("e4m3_mqa_g16", 3, 16, 1, 128, 16, 100, 5000, 27, "e4m3"), 0),
    (fcase("e4m3_g12", 3, 24, 2, 128, 32, 100, 2000, 28, "e4m3"), 2),
    (fcase("e5m2_g1", 4, 4, 4, 64, 16, 1, 900, 29, "e5m2"), 0),
    (fcase("e4m3_edges", 0, 8, 2, 128, 16, 0, 0, 30, "e4m3", lens=[0, 1, 15, 16, 17, 63, 64, 65, 1024, 1025]), 0),
    (fcase("e4m3_g32_mqa", 3, 32, 1, 128, 16, 100, 3000, 31, "e4m3"), 0),   # two groups of 16 heads
    (fcase("e5m2_g20_split2", 2, 40, 2, 64, 16, 1500, 3000, 32, "e5m2"), 2),  # 16 + 4 heads per kv head
    # head width 64 runs 32-token stages: lengths around multiples of 32 and of the page size
    (fcase("e4m3_edges_d64", 0, 8, 2, 64, 16, 0, 0, 33, "e4m3",
           lens=[0, 1, 31, 32, 33, 47, 63, 64, 65, 95, 96, 97, 1023, 1024, 1025]), 0),
    (fcase("e5m2_edges_d64_split3", 0, 8, 2, 64, 5, 0, 0, 34, "e5m2", lens=[1, 33, 95, 130, 1000, 1600]), 3),
    (fcase("e4m3_p3", 5, 8, 2, 128, 3, 1, 2000, 37, "e4m3"), 0),   # page sizes that are not powers of two
    (fcase("e4m3_p100_d64", 4, 8, 1, 64, 100, 1, 5000, 38, "e4m3"), 0),
    (fcase("e5m2_p1000", 3, 8, 2, 128, 1000, 500, 7000, 39, "e5m2"), 2),
]


@pytest.mark.parametrize("c,ns", CASES, ids=[c.name for c, _ in CASES])
def test_fp8_decode_cases(A, c, ns):
    q, kc8, vc8, pt, sl, kds, vds = c.generate_fp8()
    o, lse = run(A, c, q, kc8, vc8, pt, sl, kds, vds, ns)
    ro, rl = reference(c, q, kc8, vc8, pt, sl, kds, vds)
    do, dl = compare(o, lse, ro, rl)
    assert do <= TOL_O and dl <= TOL_LSE, f"{c.name}: max|dO|={do:.3e} max|dLSE|={dl:.3e}"


def test_fp8_descales_are_applied(A):
    """Scaling the descales changes the GPU result exactly as it changes the oracle's."""
    c = fcase("descale", 4, 8, 2, 128, 16, 200, 3000, 31, "e4m3")
    q, kc8, vc8, pt, sl, _, _ = c.generate_fp8()
    for kds, vds in ((0.004, 0.01), (0.02, 3.0)):
        o, lse = run(A, c, q, kc8, vc8, pt, sl, kds, vds)
        ro, rl = reference(c, q, kc8, vc8, pt, sl, kds, vds)
        do, dl = compare(o, lse, ro, rl)
        # the output is stored in bf16: its rounding grows with |O|, so the bound scales with it
        tol = TOL_O * max(1.0, float(np.abs(ro).max()))
        assert do <= tol and dl <= TOL_LSE, f"descales {kds},{vds}: {do:.3e} {dl:.3e}"


def test_fp8_nan_pages_never_read(A):
    c = fcase("canary", 6, 8, 2, 128, 16, 1, 2000, 32, "e4m3", extra=12)
    q, kc8, vc8, pt, sl, kds, vds = c.generate_fp8()
    used = np.zeros(c.num_pages, dtype=bool)
    for b in range(c.B):
        used[pt[b, : int(c.pages_per_seq[b])]] = True
    kc8[~used] = 0x7F  # NaN codes
    vc8[~used] = 0x7F
    o, lse = run(A, c, q, kc8, vc8, pt, sl, kds, vds)
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    ro, rl = reference(c, q, kc8, vc8, pt, sl, kds, vds)
    do, dl = compare(o, lse, ro, rl)
    assert do <= TOL_O and dl <= TOL_LSE


def test_fp8_split_count_does_not_change_result(A):
    c = fcase("splits", 4, 8, 2, 128, 16, 3000, 6000, 33, "e5m2")
    q, kc8, vc8, pt, sl, kds, vds = c.generate_fp8()
    outs = [run(A, c, q, kc8, vc8, pt, sl, kds, vds, ns) for ns in (1, 2, 5, 0)]
    for o, lse in outs[1:]:
        assert (o.float() - outs[0][0].float()).abs().max().item() <= 2e-2
        assert (lse - outs[0][1]).abs().max().item() <= 2e-3


@pytest.mark.parametrize("fmt,d,seed", [("e4m3", 128, 35), ("e5m2", 64, 36)])
def test_fp8_decode_order_switch_is_exact(A, fmt, d, seed):
    """Both split orders give the same bytes (splits move between CTAs, tokens stay in their
    split), and those match the oracle."""
    c = fcase("order_" + fmt, 29, 16, 4, d, 16, 1, 7000, seed, fmt)
    q, kc8, vc8, pt, sl, kds, vds = c.generate_fp8()
    outs = []
    try:
        for order in (0, 1):
            A.attn_set_option("decode_order", order)
            outs.append(run(A, c, q, kc8, vc8, pt, sl, kds, vds))
    finally:
        A.attn_set_option("decode_order", 1)
    (o0, l0), (o1, l1) = outs
    assert torch.equal(o0.view(torch.int16), o1.view(torch.int16)) and torch.equal(l0, l1)
    ro, rl = reference(c, q, kc8, vc8, pt, sl, kds, vds)
    do, dl = compare(o1, l1, ro, rl)
    assert do <= TOL_O and dl <= TOL_LSE, f"max|dO|={do:.3e} max|dLSE|={dl:.3e}"


def test_fp8_decode_workload_full(A):
    """The full e4m3 decode workload (64 sequences, lengths up to 32768), every sequence and head."""
    c = W.decode_fp8()
    q, kc8, vc8, pt, sl, kds, vds = c.generate_fp8()
    o, lse = run(A, c, q, kc8, vc8, pt, sl, kds, vds)
    ro, rl = reference(c, q, kc8, vc8, pt, sl, kds, vds)
    do, dl = compare(o, lse, ro, rl)
    assert do <= TOL_O and dl <= TOL_LSE, f"max|dO|={do:.3e} max|dLSE|={dl:.3e}"


def test_fp8_rejects_unknown_format_and_bad_descales(A):
    c = fcase("bad", 2, 8, 2, 128, 16, 10, 20, 34, "e4m3")
    q, kc8, vc8, pt, sl, kds, vds = c.generate_fp8()
    for fmt, k_, v_ in ((2, kds, vds), (0, float("inf"), vds), (1, kds, float("nan"))):
        o = torch.full((c.B, c.Hq, c.d), float("nan"), dtype=torch.bfloat16, device=DEV)
        lse = torch.full((c.B, c.Hq), float("nan"), dtype=torch.float32, device=DEV)
        rc = A.attn_decode_paged_fp8(to_dev(q, DEV), torch.from_numpy(kc8).to(DEV), torch.from_numpy(vc8).to(DEV),
                                     torch.from_numpy(pt).to(DEV), torch.from_numpy(sl).to(DEV), c.page_size, o, lse,
                                     None, c.B, c.Hq, c.Hkv, c.d, c.max_pages, c.num_pages, c.scale, 0, fmt, k_, v_,
                                     raise_on_error=False)
        assert rc == A.ATTN_ERR_BAD_ARG
        torch.cuda.synchronize()
        assert torch.isnan(o.float()).all()


MAP_CASES = [
    (fcase("maps_p16_g4", 13, 32, 8, 128, 16, 1, 4000, 41, "e4m3"), 0),
    (fcase("maps_p32_g12_split2", 5, 24, 2, 128, 32, 100, 3000, 42, "e5m2"), 2),
    (fcase("maps_p64_g32", 3, 32, 1, 128, 64, 1, 5000, 43, "e4m3"), 0),
    (fcase("maps_p48_edges", 0, 8, 2, 128, 48, 0, 0, 44, "e4m3", lens=[0, 1, 15, 16, 17, 47, 48, 49, 1023, 1025]), 3),
]


@pytest.mark.parametrize("c,ns", MAP_CASES, ids=[c.name for c, _ in MAP_CASES])
def test_fp8_decode_maps_switch_is_exact(A, c, ns):
    """Page sizes that are multiples of 16 load each token group through the caches' tensor maps
    (option decode_maps, default 1; at most 8 or more than 16 query heads per kv head, the 12-head
    case checks that the switch leaves the other shapes alone); the per-row copies (0) must give
    the same bytes, and both the oracle's result."""
    q, kc8, vc8, pt, sl, kds, vds = c.generate_fp8()
    outs = []
    try:
        for maps in (0, 1):
            A.attn_set_option("decode_maps", maps)
            outs.append(run(A, c, q, kc8, vc8, pt, sl, kds, vds, ns))
    finally:
        A.attn_set_option("decode_maps", 1)
    (o0, l0), (o1, l1) = outs
    assert torch.equal(o0.view(torch.int16), o1.view(torch.int16)) and torch.equal(l0, l1)
    ro, rl = reference(c, q, kc8, vc8, pt, sl, kds, vds)
    do, dl = compare(o1, l1, ro, rl)
    assert do <= TOL_O and dl <= TOL_LSE, f"{c.name}: max|dO|={do:.3e} max|dLSE|={dl:.3e}"


@pytest.mark.parametrize("maps", [1, 0])
def test_fp8_nan_codes_past_the_length_never_count(A, maps):
    """NaN codes in the slots of a sequence's last page past its length (a map load brings those
    rows into shared memory with the group's others) and in unreferenced pages leave the result
    finite and equal to the oracle's."""
    c = fcase("tail_canary", 7, 16, 4, 128, 32, 1, 3000, 45, "e4m3", extra=5,
              lens=[1, 17, 31, 33, 100, 1000, 2047])
    q, kc8, vc8, pt, sl, kds, vds = c.generate_fp8()
    used_rows = np.zeros((c.num_pages, c.page_size), dtype=bool)
    for b in range(c.B):
        for t in range(int(sl[b])):
            used_rows[pt[b, t // c.page_size], t % c.page_size] = True
    kc8[~used_rows] = 0x7F  # NaN codes
    vc8[~used_rows] = 0x7F
    try:
        A.attn_set_option("decode_maps", maps)
        o, lse = run(A, c, q, kc8, vc8, pt, sl, kds, vds)
    finally:
        A.attn_set_option("decode_maps", 1)
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    ro, rl = reference(c, q, kc8, vc8, pt, sl, kds, vds)
    do, dl = compare(o, lse, ro, rl)
    assert do <= TOL_O and dl <= TOL_LSE, f"max|dO|={do:.3e} max|dLSE|={dl:.3e}"


@pytest.mark.parametrize("maps", [1, 0])
def test_fp8_bad_page_index_is_reported(A, maps):
    """An out-of-range page-table entry is reported and not read: its rows count as zeros (with
    the map loads and with the per-row copies), and the sequences that do not use it are
    unaffected."""
    c = fcase("badpage8", 2, 8, 2, 128, 16, 40, 60, 46, "e4m3")
    q, kc8, vc8, pt, sl, kds, vds = c.generate_fp8()
    pt = pt.copy()
    pt[1, 1] = c.num_pages + 5
    o = torch.full((c.B, c.Hq, c.d), float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.full((c.B, c.Hq), float("nan"), dtype=torch.float32, device=DEV)
    try:
        A.attn_set_option("decode_maps", maps)
        A.attn_decode_paged_fp8(to_dev(q, DEV), torch.from_numpy(kc8).to(DEV), torch.from_numpy(vc8).to(DEV),
                                torch.from_numpy(pt).to(DEV), torch.from_numpy(sl).to(DEV), c.page_size, o, lse, None,
                                c.B, c.Hq, c.Hkv, c.d, c.max_pages, c.num_pages, c.scale, 0, c.kv_fmt, kds, vds)
    finally:
        A.attn_set_option("decode_maps", 1)
    assert A.attn_get_device_status() == A.ATTN_ERR_DEVICE_BAD_INDEX
    assert A.attn_get_device_status() == 0
    # the oracle with the bad entry pointing at a page of zero codes (+0.0 in both formats)
    zero = np.zeros((1,) + kc8.shape[1:], dtype=kc8.dtype)
    kz, vz = np.concatenate([kc8, zero]), np.concatenate([vc8, zero])
    pz = pt.copy()
    pz[1, 1] = c.num_pages
    ro, rl = oracle.attn_decode_paged_fp8(q, kz, vz, c.kv_fmt, kds, vds, pz, sl, c.page_size, c.B, c.Hq, c.Hkv, c.d,
                                          c.max_pages, c.scale)
    do, dl = compare(o, lse, ro, rl)
    assert do <= TOL_O and dl <= TOL_LSE, f"max|dO|={do:.3e} max|dLSE|={dl:.3e}"
