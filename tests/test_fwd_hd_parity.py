"""attn_fwd_hd with head dims (d, dv) = (192, 128) on the GPU against the float64 CPU oracle
(queries and keys 192 wide, values and outputs 128 wide)."""
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


def case(name, B, Hq, Hkv, Nq, Nk, causal, seed, q_mult=1.0, lens=None):
    cu = None
    if lens is not None:
        cu = np.zeros(len(lens) + 1, dtype=np.int32)
        cu[1:] = np.cumsum(lens)
        B, Nq, Nk = len(lens), int(cu[-1]), int(cu[-1])
    return W.PrefillCase(name, B, Hq, Hkv, Nq, Nk, 192, 1.0 / math.sqrt(192), causal, seed, q_mult, cu, dv=128)


def run(A, c, q, k, v):
    o = torch.full((c.total_q, c.Hq, 128), float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.full((c.total_q, c.Hq), float("nan"), dtype=torch.float32, device=DEV)
    cu = None if c.cu_seqlens is None else torch.from_numpy(c.cu_seqlens).to(DEV)
    Nq, Nk = (c.Nq, c.Nk) if cu is None else (c.total_q, c.total_k)
    A.attn_fwd_hd(to_dev(q, DEV), to_dev(k, DEV), to_dev(v, DEV), o, lse, c.B, c.Hq, c.Hkv, Nq, Nk, 192, 128, c.scale,
                  c.causal, cu)
    st = A.attn_get_device_status()
    assert st == 0, A.status_string(st)
    return o, lse


def check(A, c, rows=None):
    q, k, v = c.generate()
    o, lse = run(A, c, q, k, v)
    f = lambda a: synth.bf16_to_f32(a).astype(np.float64)
    ro, rl = oracle.attn_fwd_f64(f(q), f(k), f(v), c.B, c.Hq, c.Hkv, c.Nq, c.Nk, 192, c.scale, c.causal,
                                 cu_seqlens=c.cu_seqlens, rows=rows, dv=128)
    if rows is not None:
        assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
        sel = torch.from_numpy(rows).to(DEV)
        o, lse = o.reshape(-1, 128)[sel], lse.reshape(-1)[sel]
    do, dl = compare(o, lse, ro, rl)
    assert do <= TOL_O and dl <= TOL_LSE, f"{c.name}: max|dO|={do:.3e} max|dLSE|={dl:.3e}"


CASES = [
    case("one_tile", 1, 1, 1, 96, 96, False, 61),
    case("ragged_noncausal", 2, 2, 2, 300, 300, False, 62),
    case("ragged_causal_gqa", 2, 4, 1, 333, 333, True, 63),
    case("q_shorter_than_k", 2, 2, 2, 200, 650, True, 64),
    case("q_longer_than_k", 1, 2, 1, 400, 150, True, 65),
    case("no_key_blocks", 1, 2, 2, 600, 100, True, 66),
    case("sharp", 1, 4, 4, 1024, 1024, True, 67, 2.0),
    case("varlen", 0, 4, 2, 0, 0, True, 68, lens=[1, 129, 0, 256, 257, 5, 600]),
    case("varlen_nc", 0, 2, 2, 0, 0, False, 69, lens=[300, 17, 96, 97]),
    case("mqa16", 1, 16, 1, 257, 257, True, 72),
]


@pytest.mark.parametrize("c", CASES, ids=[c.name for c in CASES])
def test_hd_cases(A, c):
    check(A, c)


def test_hd_long_causal_full(A):
    """The benchmark's (192, 128) leg (B1 H32 N8192 causal, Q x2), every row."""
    check(A, case("hd_long", 1, 32, 32, 8192, 8192, True, W.long_causal().seed, 2.0))


def test_hd_equal_dims_match_attn_fwd(A):
    """(128, 128) through attn_fwd_hd is attn_fwd."""
    c = W.PrefillCase("eq", 1, 2, 2, 300, 300, 128, 1.0 / math.sqrt(128), True, 71)
    q, k, v = c.generate()
    outs = []
    for fn in ("attn_fwd", "attn_fwd_hd"):
        o = torch.empty((c.total_q, c.Hq, 128), dtype=torch.bfloat16, device=DEV)
        lse = torch.empty((c.total_q, c.Hq), dtype=torch.float32, device=DEV)
        args = (to_dev(q, DEV), to_dev(k, DEV), to_dev(v, DEV), o, lse, c.B, c.Hq, c.Hkv, c.Nq, c.Nk)
        if fn == "attn_fwd":
            A.attn_fwd(*args, 128, c.scale, True)
        else:
            A.attn_fwd_hd(*args, 128, 128, c.scale, True)
        outs.append((o, lse))
    torch.cuda.synchronize()
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])


def test_hd_varlen_several_launches(A):
    """300 packed sequences with head dims (192, 128): two launches of at most 256 sequences."""
    rng = np.random.default_rng(73)
    check(A, case("varlen300", 0, 2, 2, 0, 0, True, 74, lens=[int(x) for x in rng.integers(1, 200, size=300)]))
