"""Seeded random shapes through the paged decode entry points, compared in full with the float64
oracle: batch size, query heads per kv head (1 to 40), head width, page size (powers of two or
not), lengths (zero, shorter than a page, many splits), forced split counts and both work orders
(last splits after the others, or sequence by sequence), with bf16 or 8-bit caches."""
import math

import numpy as np
import pytest

import oracle
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


def random_case(seed, kv_fmt):
    rng = np.random.default_rng(seed)
    B = int(rng.choice([1, 3, 17, 70]))
    Hkv = int(rng.choice([1, 2, 4]))
    G = int(rng.choice([1, 2, 4, 8, 12, 16, 24, 40]))
    d = int(rng.choice([64, 128]))
    page = int(rng.choice([1, 2, 5, 16, 37, 64]))
    hi = int(rng.choice([40, 700, 5000]))
    lens = rng.integers(0, hi + 1, size=B).astype(np.int32)
    max_pages = int((max(int(lens.max()), 1) + page - 1) // page) + int(rng.integers(0, 3))
    return W.DecodeCase(f"dr{seed}", B, Hkv * G, Hkv, d, page, lens, max_pages, 1.0 / math.sqrt(d), seed,
                        kv_fmt=kv_fmt), int(rng.choice([0, 0, 1, 3])), int(rng.integers(0, 2))


def run(A, c, ns, order):
    A.attn_set_option("decode_order", order)
    try:
        o = torch.full((c.B, c.Hq, c.d), float("nan"), dtype=torch.bfloat16, device=DEV)
        lse = torch.full((c.B, c.Hq), float("nan"), dtype=torch.float32, device=DEV)
        if c.kv_fmt == "bf16":
            q, kc, vc, pt, sl = c.generate()
            A.attn_decode_paged(to_dev(q, DEV), to_dev(kc, DEV), to_dev(vc, DEV), torch.from_numpy(pt).to(DEV),
                                torch.from_numpy(sl).to(DEV), c.page_size, o, lse, None, c.B, c.Hq, c.Hkv, c.d,
                                c.max_pages, c.num_pages, c.scale, ns)
            ro, rl = oracle.attn_decode_paged(q, kc, vc, pt, sl, c.page_size, c.B, c.Hq, c.Hkv, c.d, c.max_pages,
                                              c.scale)
        else:
            q, kc8, vc8, pt, sl, kds, vds = c.generate_fp8()
            A.attn_decode_paged_fp8(to_dev(q, DEV), torch.from_numpy(kc8).to(DEV), torch.from_numpy(vc8).to(DEV),
                                    torch.from_numpy(pt).to(DEV), torch.from_numpy(sl).to(DEV), c.page_size, o, lse,
                                    None, c.B, c.Hq, c.Hkv, c.d, c.max_pages, c.num_pages, c.scale, ns, c.kv_fmt,
                                    kds, vds)
            ro, rl = oracle.attn_decode_paged_fp8(q, kc8, vc8, c.kv_fmt, kds, vds, pt, sl, c.page_size, c.B, c.Hq,
                                                  c.Hkv, c.d, c.max_pages, c.scale)
        st = A.attn_get_device_status()
        assert st == 0, A.status_string(st)
        return compare(o, lse, ro, rl)
    finally:
        A.attn_set_option("decode_order", 1)


@pytest.mark.parametrize("seed", range(12))
@pytest.mark.parametrize("kv_fmt", ["bf16", "e4m3", "e5m2"])
def test_decode_random_shapes(A, seed, kv_fmt):
    c, ns, order = random_case(1000 + 37 * seed + {"bf16": 0, "e4m3": 1, "e5m2": 2}[kv_fmt], kv_fmt)
    do, dl = run(A, c, ns, order)
    assert do <= TOL_O and dl <= TOL_LSE, (f"{c.name} {kv_fmt} B{c.B} Hq{c.Hq} Hkv{c.Hkv} d{c.d} page{c.page_size} "
                                           f"splits{ns} order{order}: max|dO|={do:.3e} max|dLSE|={dl:.3e}")
