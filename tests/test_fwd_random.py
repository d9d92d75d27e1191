"""Seeded random shapes through the forward entry points, compared in full with the float64 oracle:
batch, heads, GQA group, lengths (ragged, Nq != Nk), mask, head dims, dense or packed sequences."""
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


def random_case(seed, d, dv=None, packed=None):
    rng = np.random.default_rng(seed)
    Hkv = int(rng.choice([1, 2, 3]))
    G = int(rng.choice([1, 2, 4, 8]))
    causal = bool(rng.integers(0, 2))
    packed = bool(rng.integers(0, 2)) if packed is None else packed
    if packed:
        lens = [int(x) for x in rng.integers(0, 700, size=int(rng.integers(1, 9)))]
        cu = np.zeros(len(lens) + 1, dtype=np.int32)
        cu[1:] = np.cumsum(lens)
        return W.PrefillCase(f"r{seed}", len(lens), Hkv * G, Hkv, int(cu[-1]), int(cu[-1]), d, 1.0 / math.sqrt(d),
                             causal, seed, 1.0, cu, dv=dv)
    B = int(rng.integers(1, 4))
    Nq = int(rng.integers(1, 900))
    Nk = int(rng.integers(1, 900))
    return W.PrefillCase(f"r{seed}", B, Hkv * G, Hkv, Nq, Nk, d, 1.0 / math.sqrt(d), causal, seed, dv=dv)


def run_and_compare(A, c, fn="attn_fwd"):
    q, k, v = c.generate()
    o = torch.full((c.total_q, c.Hq, c.d_v), float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.full((c.total_q, c.Hq), float("nan"), dtype=torch.float32, device=DEV)
    cu = None if c.cu_seqlens is None else torch.from_numpy(c.cu_seqlens).to(DEV)
    Nq, Nk = (c.Nq, c.Nk) if cu is None else (c.total_q, c.total_k)
    if fn == "attn_fwd":
        A.attn_fwd(to_dev(q, DEV), to_dev(k, DEV), to_dev(v, DEV), o, lse, c.B, c.Hq, c.Hkv, Nq, Nk, c.d, c.scale,
                   c.causal, cu)
        ro, rl = oracle.attn_fwd(q, k, v, c.B, c.Hq, c.Hkv, c.Nq, c.Nk, c.d, c.scale, c.causal,
                                 cu_seqlens=c.cu_seqlens)
    elif fn == "attn_fwd_hd":
        A.attn_fwd_hd(to_dev(q, DEV), to_dev(k, DEV), to_dev(v, DEV), o, lse, c.B, c.Hq, c.Hkv, Nq, Nk, c.d, c.d_v,
                      c.scale, c.causal, cu)
        f = lambda a: synth.bf16_to_f32(a).astype(np.float64)
        ro, rl = oracle.attn_fwd_f64(f(q), f(k), f(v), c.B, c.Hq, c.Hkv, c.Nq, c.Nk, c.d, c.scale, c.causal,
                                     cu_seqlens=c.cu_seqlens, dv=c.d_v)
    else:
        q8, k8, v8, qs, ks, vs = c.generate_fp8("e4m3")
        dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
        A.attn_fwd_fp8(dev(q8), dev(k8), dev(v8), o, lse, c.B, c.Hq, c.Hkv, Nq, Nk, c.d, c.scale, c.causal, cu, None,
                       "e4m3", qs, ks, vs)
        ro, rl = oracle.attn_fwd_fp8(q8, k8, v8, "e4m3", qs, ks, vs, c.B, c.Hq, c.Hkv, c.Nq, c.Nk, c.d, c.scale,
                                     c.causal, cu_seqlens=c.cu_seqlens)
    st = A.attn_get_device_status()
    assert st == 0, A.status_string(st)
    do, dl = compare(o, lse, ro, rl)
    shape = f"B{c.B} Hq{c.Hq} Hkv{c.Hkv} Nq{c.Nq} Nk{c.Nk} d{c.d}/{c.d_v} causal{c.causal} packed{c.cu_seqlens is not None}"
    assert do <= TOL_O and dl <= TOL_LSE, f"{shape}: max|dO|={do:.3e} max|dLSE|={dl:.3e}"


@pytest.mark.parametrize("seed", range(1000, 1012))
@pytest.mark.parametrize("d", [64, 128])
def test_random_shapes(A, seed, d):
    run_and_compare(A, random_case(seed, d))


@pytest.mark.parametrize("seed", range(2000, 2006))
def test_random_shapes_head_dims_192_128(A, seed):
    run_and_compare(A, random_case(seed, 192, dv=128), "attn_fwd_hd")


@pytest.mark.parametrize("seed", range(3000, 3006))
def test_random_shapes_fp8(A, seed):
    run_and_compare(A, random_case(seed, 128), "attn_fwd_fp8")


def test_many_short_packed_sequences(A):
    """1000 packed sequences (the work-order build runs over 32 chunks of sequences), lengths
    0..40 with repeats, causal GQA."""
    lens = [int(x) % 41 for x in synth.uniform_ints(1000, 77, 0, 1 << 20)]
    cu = np.zeros(len(lens) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lens)
    c = W.PrefillCase("many", len(lens), 4, 2, int(cu[-1]), int(cu[-1]), 64, 0.125, True, 78, 1.0, cu)
    run_and_compare(A, c)
