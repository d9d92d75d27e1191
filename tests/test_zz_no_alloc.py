"""The allocation-free decode entry point, attn_decode_paged_noalloc.

Some callers cannot allocate device memory at the moment they run decode: an engine that
has already handed nearly all GPU memory to its own KV-cache pool, or code that must not
enter the driver's allocator. This entry point keeps the split partials in a fixed array
built into the library instead. The tests call it through the C ABI and compare it with
attn_decode_paged on the same inputs over calls in a row (each later call finds the array
as the previous call left it), and check that sizes beyond the array are refused before
anything runs.

The file name makes pytest collect it after every other test file.
"""
import ctypes
import json
import math
import os
import subprocess
import sys
import textwrap

import numpy as np
import pytest

import oracle
import synth
from helpers import ROOT, TOL_LSE, TOL_O, compare, ensure_built, to_dev
from synth import workloads as W

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
DEV = "cuda:0"
ATTN_ERR_SCRATCH_TOO_SMALL = -9


@pytest.fixture(scope="module")
def lib():
    path = ensure_built()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    L = ctypes.CDLL(path)
    vp, i = ctypes.c_void_p, ctypes.c_int
    for name in ("attn_decode_paged", "attn_decode_paged_noalloc"):
        f = getattr(L, name)
        f.argtypes = [vp, vp, vp, vp, vp, i, vp, vp, vp, i, i, i, i, i, i, ctypes.c_float, i]
        f.restype = i
    L.attn_get_device_status.argtypes = [vp]
    L.attn_get_device_status.restype = i
    L.attn_decode_plan.argtypes = [i, i, i, i, i, i, i, ctypes.POINTER(i), ctypes.POINTER(i)]
    L.attn_decode_plan.restype = i
    return L


def make_case(seed, B, Hq, Hkv, d, page_size, lo, hi):
    lens = synth.uniform_ints(B, seed, lo, hi)
    max_pages = int((int(lens.max()) + page_size - 1) // page_size) + 1
    return W.DecodeCase(f"noalloc{seed}", B, Hq, Hkv, d, page_size, lens, max_pages, 1.0 / math.sqrt(d), seed)


def splits_of(L, c):
    chunk, splits = ctypes.c_int(), ctypes.c_int()
    assert L.attn_decode_plan(c.B, c.Hq, c.Hkv, c.max_pages, c.page_size, 0, 0, ctypes.byref(chunk),
                              ctypes.byref(splits)) == 0
    return splits.value


def run(L, name, c, inputs):
    q, kc, vc, pt, sl = inputs
    o = torch.full((c.B, c.Hq, c.d), float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.full((c.B, c.Hq), float("nan"), dtype=torch.float32, device=DEV)
    rc = getattr(L, name)(q.data_ptr(), kc.data_ptr(), vc.data_ptr(), pt.data_ptr(), sl.data_ptr(), c.page_size,
                          o.data_ptr(), lse.data_ptr(), None, c.B, c.Hq, c.Hkv, c.d, c.max_pages, c.num_pages, c.scale, 0)
    assert rc == 0, f"{name} returned {rc}"
    assert L.attn_get_device_status(None) == 0  # synchronises the stream
    return o.float(), lse


def test_noalloc_matches_allocating_entry_point_over_calls_in_a_row(lib):
    cases = [make_case(101, 6, 32, 8, 128, 16, 2000, 9000),  # GQA 4, several splits per sequence
             make_case(102, 3, 16, 1, 64, 7, 100, 5000)]     # different sizes: finds the first call's leftovers
    for c in cases:
        assert splits_of(lib, c) > 1, "the case must use the split workspace"
        q, kc, vc, pt, sl = c.generate()
        inputs = (to_dev(q, DEV), to_dev(kc, DEV), to_dev(vc, DEV), torch.from_numpy(pt).to(DEV),
                  torch.from_numpy(sl).to(DEV))
        o_ref, l_ref = run(lib, "attn_decode_paged", c, inputs)
        ro, rl = oracle.attn_decode_paged(q, kc, vc, pt, sl, c.page_size, c.B, c.Hq, c.Hkv, c.d, c.max_pages, c.scale)
        for _ in range(2):  # two calls in a row on the same inputs
            o, l = run(lib, "attn_decode_paged_noalloc", c, inputs)
            assert torch.isfinite(o).all() and torch.isfinite(l).all()
            assert (o - o_ref).abs().max().item() <= TOL_O
            assert (l - l_ref).abs().max().item() <= TOL_LSE
            do, dl = compare(o, l, ro, rl)  # and against the float64 oracle directly
            assert do <= TOL_O and dl <= TOL_LSE, f"max|dO|={do:.3e} max|dLSE|={dl:.3e}"


def test_noalloc_refuses_sizes_beyond_its_array(lib):
    # 64 sequences x 32 heads x 64 splits x (128 + 1) floats = 67.6 MB > the 32 MiB array
    B, Hq, Hkv, d, page_size, max_pages = 64, 32, 8, 128, 16, 2048
    q = torch.zeros((B, Hq, d), dtype=torch.bfloat16, device=DEV)
    cache = torch.zeros((1, page_size, Hkv, d), dtype=torch.bfloat16, device=DEV)
    pt = torch.zeros((B, max_pages), dtype=torch.int32, device=DEV)
    sl = torch.ones((B,), dtype=torch.int32, device=DEV)
    o = torch.full((B, Hq, d), float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.full((B, Hq), float("nan"), dtype=torch.float32, device=DEV)
    rc = lib.attn_decode_paged_noalloc(q.data_ptr(), cache.data_ptr(), cache.data_ptr(), pt.data_ptr(), sl.data_ptr(),
                                       page_size, o.data_ptr(), lse.data_ptr(), None, B, Hq, Hkv, d, max_pages, 1,
                                       0.088, 64)
    assert rc == ATTN_ERR_SCRATCH_TOO_SMALL
    torch.cuda.synchronize()
    assert torch.isnan(o.float()).all() and torch.isnan(lse).all()  # nothing ran


_FRESH = textwrap.dedent("""
    import ctypes, json, math, re, sys
    import numpy as np
    import torch
    sys.path.insert(0, ROOT)
    import oracle
    import synth
    from synth import workloads as W
    L = ctypes.CDLL(LIB)
    vp, i = ctypes.c_void_p, ctypes.c_int
    f = L.attn_decode_paged_noalloc
    f.argtypes = [vp, vp, vp, vp, vp, i, vp, vp, vp, i, i, i, i, i, i, ctypes.c_float, i]
    f.restype = i
    L.attn_get_device_status.argtypes = [vp]
    L.attn_get_device_status.restype = i
    # the CUDA runtime the library uses, for the device's default memory pool
    rt_path = next(l.split()[-1] for l in open("/proc/self/maps") if re.search(r"libcudart\\.so", l))
    rt = ctypes.CDLL(rt_path)

    def pool_high():
        pool, v = ctypes.c_void_p(), ctypes.c_uint64()
        if rt.cudaDeviceGetDefaultMemPool(ctypes.byref(pool), 0) != 0:
            return None
        out = []
        for attr in (6, 8):  # reserved and used high watermarks
            if rt.cudaMemPoolGetAttribute(pool, attr, ctypes.byref(v)) != 0:
                return None
            out.append(v.value)
        return out

    lens = synth.uniform_ints(64, 103, 2000, 9000)
    c = W.DecodeCase("noalloc_fresh", 64, 32, 8, 128, 16, lens, int(lens.max()) // 16 + 2, 1 / math.sqrt(128), 103)
    q, kc, vc, pt, sl = c.generate()
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    bf = lambda a: dev(a.view(np.int16)).view(torch.bfloat16)
    Q, KC, VC, PT, SL = bf(q), bf(kc), bf(vc), dev(pt), dev(sl)
    O = torch.empty((c.B, c.Hq, c.d), dtype=torch.bfloat16, device="cuda")
    LSE = torch.empty((c.B, c.Hq), dtype=torch.float32, device="cuda")

    def call():
        rc = f(Q.data_ptr(), KC.data_ptr(), VC.data_ptr(), PT.data_ptr(), SL.data_ptr(), c.page_size, O.data_ptr(),
               LSE.data_ptr(), None, c.B, c.Hq, c.Hkv, c.d, c.max_pages, c.num_pages, c.scale, 0)
        assert rc == 0, rc
        assert L.attn_get_device_status(None) == 0  # synchronises

    def step(check=True):
        O.fill_(float("nan"))
        LSE.fill_(float("nan"))
        torch.cuda.synchronize()
        mem0 = torch.cuda.mem_get_info()[0]
        call()
        assert not check or torch.cuda.mem_get_info()[0] == mem0
        return O.cpu().float().numpy(), LSE.cpu().numpy()  # converted on the host: no device memory

    # The first step loads every kernel involved (the library's, and PyTorch's fill) and lets
    # the library resolve its array's address; loading a module takes device memory once.
    step(check=False)
    torch.cuda.synchronize()
    before = (torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated(), torch.cuda.memory_reserved(), pool_high())
    res = [step() for _ in range(2)]
    torch.cuda.synchronize()
    after = (torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated(), torch.cuda.memory_reserved(), pool_high())
    ro, rl = oracle.attn_decode_paged(q, kc, vc, pt, sl, c.page_size, c.B, c.Hq, c.Hkv, c.d, c.max_pages, c.scale)
    err = [(float(np.abs(o - ro).max()), float(np.abs(l - rl).max())) for o, l in res]
    print(json.dumps({"before": before, "after": after, "err": err}))
""")


def test_noalloc_in_a_fresh_process_allocates_nothing(lib):
    """In a process that never calls the allocating decode, two calls in a row leave the free
    device memory, PyTorch's allocator and the device's default memory pool exactly as they
    were (a call that took its workspace from a retained pool or leaked it would show there),
    and both match the float64 oracle."""
    path = ensure_built()
    env = dict(os.environ, PYTHONPATH=ROOT)
    code = f"ROOT = {ROOT!r}\nLIB = {path!r}\n" + _FRESH
    out = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-3000:]
    r = json.loads(out.stdout.strip().splitlines()[-1])
    assert r["before"] == r["after"], r
    for do, dl in r["err"]:
        assert do <= TOL_O and dl <= TOL_LSE, r["err"]
