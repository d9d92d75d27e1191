"""attn_decode_paged on the GPU against the float64 CPU oracle (full comparison)."""
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


def run_decode(A, c, q, kc, vc, pt, sl, num_splits=0):
    o = torch.full((c.B, c.Hq, c.d), float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.full((c.B, c.Hq), float("nan"), dtype=torch.float32, device=DEV)
    A.attn_decode_paged(to_dev(q, DEV), to_dev(kc, DEV), to_dev(vc, DEV), torch.from_numpy(pt).to(DEV),
                        torch.from_numpy(sl).to(DEV), c.page_size, o, lse, None, c.B, c.Hq, c.Hkv, c.d, c.max_pages,
                        c.num_pages, c.scale, num_splits)
    return o, lse


def check(A, c, num_splits=0, canary=False):
    q, kc, vc, pt, sl = c.generate()
    if canary:  # unreferenced pool pages hold NaN: they must never be read
        used = np.zeros(c.num_pages, dtype=bool)
        for b in range(c.B):
            used[pt[b, : int(c.pages_per_seq[b])]] = True
        kc[~used] = 0x7FC0
        vc[~used] = 0x7FC0
    o, lse = run_decode(A, c, q, kc, vc, pt, sl, num_splits)
    st = A.attn_get_device_status()
    assert st == 0, A.status_string(st)
    ro, rl = oracle.attn_decode_paged(q, kc, vc, pt, sl, c.page_size, c.B, c.Hq, c.Hkv, c.d, c.max_pages, c.scale)
    do, dl = compare(o, lse, ro, rl)
    assert do <= TOL_O and dl <= TOL_LSE, f"{c.name}: max|dO|={do:.3e} max|dLSE|={dl:.3e}"


def dcase(name, B, Hq, Hkv, d, page_size, lo, hi, seed, extra=0, lens=None):
    if lens is None:
        lens = synth.uniform_ints(B, seed, lo, hi)
    lens = np.asarray(lens, dtype=np.int32)
    max_pages = int((max(int(lens.max()), 1) + page_size - 1) // page_size) + 2
    return W.DecodeCase(name, len(lens), Hq, Hkv, d, page_size, lens, max_pages, 1.0 / math.sqrt(d), seed,
                        extra_pages=extra)


CASES = [
    (dcase("p16_g4", 9, 32, 8, 128, 16, 1, 3000, 1), 0),
    (dcase("p16_g4_split3", 5, 8, 2, 128, 16, 500, 2500, 2), 3),
    (dcase("p1", 4, 8, 2, 128, 1, 1, 700, 3), 0),
    (dcase("p7_d64", 6, 12, 3, 64, 7, 1, 1500, 4), 0),
    (dcase("mqa_g16", 3, 16, 1, 128, 16, 100, 5000, 5), 0),
    (dcase("g12", 3, 24, 2, 128, 32, 100, 2000, 6), 2),
    (dcase("g1", 4, 4, 4, 64, 16, 1, 900, 7), 0),
    (dcase("edge_lengths", 0, 8, 2, 128, 16, 0, 0, 8, lens=[0, 1, 15, 16, 17, 63, 64, 65, 1024, 1025]), 0),
    (dcase("one_split", 4, 8, 2, 128, 16, 1, 4000, 9), 1),
    (dcase("g32_mqa", 3, 32, 1, 128, 16, 100, 3000, 13), 0),     # two groups of 16 heads
    (dcase("g24_d64", 3, 48, 2, 64, 8, 1, 2500, 14), 0),       # 16 + 8 heads per kv head
    (dcase("g40_split2", 2, 40, 1, 128, 16, 2000, 4000, 15), 2),
    (dcase("b300_unranked", 300, 4, 2, 64, 16, 1, 700, 16), 3),  # over 256 sequences: last splits unsorted
    (dcase("p3", 5, 8, 2, 128, 3, 1, 2000, 20), 0),              # page sizes that are not powers of two
    (dcase("p100_d64", 4, 8, 1, 64, 100, 1, 5000, 21), 0),
    (dcase("p1000", 3, 8, 2, 128, 1000, 500, 7000, 22), 2),
]


@pytest.mark.parametrize("c,ns", CASES, ids=[c.name for c, _ in CASES])
def test_decode_cases(A, c, ns):
    check(A, c, ns)


def test_nan_pages_never_read(A):
    check(A, dcase("canary", 6, 8, 2, 128, 16, 1, 2000, 10, extra=12), canary=True)


def test_split_count_does_not_change_result(A):
    c = dcase("splits", 4, 8, 2, 128, 16, 3000, 6000, 11)
    q, kc, vc, pt, sl = c.generate()
    outs = []
    for ns in (1, 2, 5, 0):
        o, lse = run_decode(A, c, q, kc, vc, pt, sl, ns)
        outs.append((o.float(), lse))
    for o, lse in outs[1:]:
        assert (o - outs[0][0]).abs().max().item() <= 2e-2
        assert (lse - outs[0][1]).abs().max().item() <= 2e-3


def test_decode_workload_full(A):
    check(A, W.decode())


def test_bad_page_index_is_reported(A):
    c = dcase("badpage", 2, 8, 2, 128, 16, 40, 60, 12)
    q, kc, vc, pt, sl = c.generate()
    pt = pt.copy()
    pt[1, 1] = c.num_pages + 5  # out of range: must be skipped and reported, not read
    o, lse = run_decode(A, c, q, kc, vc, pt, sl)
    assert A.attn_get_device_status() == A.ATTN_ERR_DEVICE_BAD_INDEX
    assert A.attn_get_device_status() == 0  # cleared by the read
    # sequence 0 is unaffected
    ro, rl = oracle.attn_decode_paged(q, kc, vc, pt * (pt < c.num_pages), sl, c.page_size, c.B, c.Hq, c.Hkv, c.d,
                                      c.max_pages, c.scale)
    do, dl = compare(o[:1], lse[:1], ro[:1], rl[:1])
    assert do <= TOL_O and dl <= TOL_LSE


@pytest.mark.parametrize("c,ns", [(dcase("order_mix", 37, 16, 4, 128, 16, 1, 6000, 17), 0),
                                  (dcase("order_b300", 300, 8, 2, 64, 8, 1, 900, 18), 4),
                                  (dcase("order_one_split", 5, 8, 2, 128, 16, 1, 900, 19), 1)],
                         ids=["mix", "b300", "one_split"])
def test_decode_order_switch_is_exact(A, c, ns):
    """The work order moves splits between CTAs, not tokens between splits: both orders give
    the same bytes, and those match the oracle."""
    q, kc, vc, pt, sl = c.generate()
    outs = []
    try:
        for order in (0, 1):
            A.attn_set_option("decode_order", order)
            outs.append(run_decode(A, c, q, kc, vc, pt, sl, ns))
    finally:
        A.attn_set_option("decode_order", 1)
    assert A.attn_get_device_status() == 0
    (o0, l0), (o1, l1) = outs
    assert torch.equal(o0.view(torch.int16), o1.view(torch.int16)) and torch.equal(l0, l1)
    ro, rl = oracle.attn_decode_paged(q, kc, vc, pt, sl, c.page_size, c.B, c.Hq, c.Hkv, c.d, c.max_pages, c.scale)
    do, dl = compare(o1, l1, ro, rl)
    assert do <= TOL_O and dl <= TOL_LSE, f"{c.name}: max|dO|={do:.3e} max|dLSE|={dl:.3e}"
