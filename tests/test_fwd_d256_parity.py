"""attn_fwd with head width d = 256 on the GPU against the float64 CPU oracle. This width runs a
separate kernel (one 128-row query tile at a time, two score buffers, key/value tiles in
128-column halves through a five-slot ring), so the cases cover one, two and three key tiles
per query tile (the ring's start-up and every position of the last score product), ragged
edges, masks that hide whole tiles, packed sequences and long sequences."""
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
D = 256


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
    return W.PrefillCase(name, B, Hq, Hkv, Nq, Nk, D, 1.0 / math.sqrt(D), causal, seed, q_mult, cu)


def run(A, c, q, k, v):
    o = torch.full((c.total_q, c.Hq, D), float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.full((c.total_q, c.Hq), float("nan"), dtype=torch.float32, device=DEV)
    cu = None if c.cu_seqlens is None else torch.from_numpy(c.cu_seqlens).to(DEV)
    Nq, Nk = (c.Nq, c.Nk) if cu is None else (c.total_q, c.total_k)
    A.attn_fwd(to_dev(q, DEV), to_dev(k, DEV), to_dev(v, DEV), o, lse, c.B, c.Hq, c.Hkv, Nq, Nk, D, c.scale, c.causal,
               cu)
    st = A.attn_get_device_status()
    assert st == 0, A.status_string(st)
    return o, lse


def check(A, c, rows=None):
    q, k, v = c.generate()
    o, lse = run(A, c, q, k, v)
    f = lambda a: synth.bf16_to_f32(a).astype(np.float64)
    ro, rl = oracle.attn_fwd_f64(f(q), f(k), f(v), c.B, c.Hq, c.Hkv, c.Nq, c.Nk, D, c.scale, c.causal,
                                 cu_seqlens=c.cu_seqlens, rows=rows)
    if rows is not None:
        assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
        sel = torch.from_numpy(rows).to(DEV)
        o, lse = o.reshape(-1, D)[sel], lse.reshape(-1)[sel]
    do, dl = compare(o, lse, ro, rl)
    assert do <= TOL_O and dl <= TOL_LSE, f"{c.name}: max|dO|={do:.3e} max|dLSE|={dl:.3e}"


CASES = [
    case("one_key_tile", 1, 1, 1, 96, 96, False, 81),
    case("two_key_tiles", 1, 2, 2, 200, 200, False, 82),
    case("three_key_tiles", 1, 2, 1, 300, 300, False, 83),
    case("ragged_causal_gqa", 2, 4, 1, 333, 333, True, 84),
    case("q_shorter_than_k", 2, 2, 2, 200, 650, True, 85),
    case("q_longer_than_k", 1, 2, 1, 400, 150, True, 86),
    case("no_key_blocks", 1, 2, 2, 600, 100, True, 87),
    case("sharp", 1, 4, 4, 1024, 1024, True, 88, 2.0),
    case("noncausal_many_tiles", 2, 3, 3, 777, 900, False, 89),
    case("varlen", 0, 4, 2, 0, 0, True, 90, lens=[1, 129, 0, 256, 257, 5, 600]),
    case("varlen_nc", 0, 2, 2, 0, 0, False, 91, lens=[300, 17, 96, 97]),
    case("mqa8", 1, 8, 1, 257, 257, True, 92),
]


@pytest.mark.parametrize("c", CASES, ids=[c.name for c in CASES])
def test_d256_cases(A, c):
    check(A, c)


def test_d256_varlen_64_sequences(A):
    """The largest packed batch this width takes (64 sequences), lengths 1 .. 300."""
    rng = np.random.default_rng(93)
    check(A, case("varlen64", 0, 2, 1, 0, 0, True, 93, lens=[int(x) for x in rng.integers(1, 301, size=64)]))


def test_d256_long_causal_full(A):
    """The benchmark's head-width-256 leg (B1 H32 N8192 causal, Q x2), every row."""
    check(A, case("d256_long", 1, 32, 32, 8192, 8192, True, W.long_causal().seed, 2.0))


def test_d256_through_attn_fwd_hd(A):
    """(256, 256) through attn_fwd_hd is attn_fwd."""
    c = case("eq", 1, 2, 2, 300, 300, True, 95)
    q, k, v = c.generate()
    outs = []
    for fn in ("attn_fwd", "attn_fwd_hd"):
        o = torch.empty((c.total_q, c.Hq, D), dtype=torch.bfloat16, device=DEV)
        lse = torch.empty((c.total_q, c.Hq), dtype=torch.float32, device=DEV)
        args = (to_dev(q, DEV), to_dev(k, DEV), to_dev(v, DEV), o, lse, c.B, c.Hq, c.Hkv, c.Nq, c.Nk)
        if fn == "attn_fwd":
            A.attn_fwd(*args, D, c.scale, True)
        else:
            A.attn_fwd_hd(*args, D, D, c.scale, True)
        outs.append((o, lse))
    torch.cuda.synchronize()
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])


def test_d256_noncausal_gqa_full(A):
    """A non-causal GQA prefill (B2 Hq8 Hkv2 N4096, d 256), every row."""
    check(A, case("d256_nc", 2, 8, 2, 4096, 4096, False, 96))


def test_d256_varlen_several_launches(A):
    """150 packed sequences at d = 256: three launches of at most 64 sequences."""
    rng = np.random.default_rng(97)
    check(A, case("varlen150", 0, 2, 1, 0, 0, False, 98, lens=[int(x) for x in rng.integers(1, 300, size=150)]))


def test_d256_static_order_matches(A):
    """The static snake order (dynamic_order = 0) and the dynamic unit counter give the same
    result up to rounding on a ragged, masked, GQA and a packed case."""
    A.attn_set_option("dynamic_order", 0)
    try:
        check(A, case("static_ragged", 2, 4, 1, 333, 333, True, 99))
        check(A, case("static_varlen", 0, 4, 2, 0, 0, True, 100, lens=[1, 129, 0, 256, 257, 5, 600]))
    finally:
        A.attn_set_option("dynamic_order", 1)


def test_d256_calls_on_two_streams_at_once(A):
    """Calls running at the same time on two streams each take their own unit counter: both
    results equal the ones of calls made one after the other."""
    cs = [case("s1", 1, 8, 2, 1500, 1500, True, 101), case("s2", 2, 4, 4, 900, 900, False, 102)]
    ins = [[to_dev(a, DEV) for a in c.generate()] for c in cs]
    outs = [(torch.empty((c.total_q, c.Hq, D), dtype=torch.bfloat16, device=DEV),
             torch.empty((c.total_q, c.Hq), dtype=torch.float32, device=DEV)) for c in cs]

    def call(i, stream):
        c = cs[i]
        A.attn_fwd(*ins[i], *outs[i], c.B, c.Hq, c.Hkv, c.Nq, c.Nk, D, c.scale, c.causal, None, stream)

    call(0, None)
    call(1, None)
    torch.cuda.synchronize()
    ref = [(o.clone(), l.clone()) for o, l in outs]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for _ in range(3):
        for o, l in outs:
            o.fill_(float("nan"))
            l.fill_(float("nan"))
        torch.cuda.synchronize()
        for _ in range(4):  # several calls queued on each stream, interleaved
            call(0, streams[0])
            call(1, streams[1])
        torch.cuda.synchronize()
        assert A.attn_get_device_status() == 0
        for (o, l), (ro, rl) in zip(outs, ref):
            assert torch.equal(o, ro) and torch.equal(l, rl)
