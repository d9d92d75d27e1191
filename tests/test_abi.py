"""The C-ABI library on the CPU: it loads, exports every declared symbol, and rejects bad
arguments on the host before touching the GPU."""
import ctypes
import os
import re

import pytest

from helpers import ROOT, ensure_built

HEADER = os.path.join(ROOT, "include", "attn.h")


@pytest.fixture(scope="module")
def lib():
    return ctypes.CDLL(ensure_built())


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(attn_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert "attn_fwd" in names and "attn_decode_paged" in names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in attn.h but not exported"


def test_python_binding_lists_the_header():
    import exact_softmax_attention_gb300 as A
    assert sorted(A.EXPORTS) == declared_functions()


def _fwd(lib, q=16, k=16, v=16, o=16, lse=16, B=1, Hq=2, Hkv=2, Nq=8, Nk=8, d=64, scale=0.125, causal=0, cu=None):
    f = lib.attn_fwd
    vp = ctypes.c_void_p
    f.argtypes = [vp, vp, vp, vp, vp] + [ctypes.c_int] * 6 + [ctypes.c_float, ctypes.c_int, vp, vp]
    return f(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, d, scale, causal, cu, None)


def test_fwd_host_validation(lib):
    import exact_softmax_attention_gb300 as A
    assert _fwd(lib, q=None) == A.ATTN_ERR_NULL_PTR
    assert _fwd(lib, lse=None) == A.ATTN_ERR_NULL_PTR
    assert _fwd(lib, d=96) == A.ATTN_ERR_BAD_SHAPE
    assert _fwd(lib, Hq=6, Hkv=4) == A.ATTN_ERR_BAD_SHAPE
    assert _fwd(lib, Nq=-1) == A.ATTN_ERR_BAD_SHAPE
    assert _fwd(lib, B=-1) == A.ATTN_ERR_BAD_SHAPE
    assert _fwd(lib, causal=2) == A.ATTN_ERR_BAD_SHAPE
    assert _fwd(lib, scale=float("nan")) == A.ATTN_ERR_BAD_SHAPE
    assert _fwd(lib, q=0x1008) == A.ATTN_ERR_ALIGN
    assert _fwd(lib, lse=0x1002) == A.ATTN_ERR_ALIGN
    assert _fwd(lib, d=192) == A.ATTN_ERR_BAD_SHAPE                 # 192 only with dv = 128 (attn_fwd_hd)
    assert _fwd(lib, d=256, B=0) == A.ATTN_OK
    # nothing to do: returns before any CUDA call
    assert _fwd(lib, B=0) == A.ATTN_OK
    assert _fwd(lib, Nq=0) == A.ATTN_OK


def _dec(lib, q=16, kc=16, vc=16, pt=16, sl=16, ps=16, o=16, lse=16, B=1, Hq=8, Hkv=2, d=128, mp=4, npg=4,
         scale=0.1, ns=0):
    f = lib.attn_decode_paged
    vp = ctypes.c_void_p
    f.argtypes = [vp, vp, vp, vp, vp, ctypes.c_int, vp, vp, vp] + [ctypes.c_int] * 6 + [ctypes.c_float, ctypes.c_int]
    return f(q, kc, vc, pt, sl, ps, o, lse, None, B, Hq, Hkv, d, mp, npg, scale, ns)


def test_decode_host_validation(lib):
    import exact_softmax_attention_gb300 as A
    assert _dec(lib, pt=None) == A.ATTN_ERR_NULL_PTR
    assert _dec(lib, Hq=36, Hkv=5) == A.ATTN_ERR_BAD_SHAPE   # Hq not a multiple of Hkv
    assert _dec(lib, ps=0) == A.ATTN_ERR_BAD_SHAPE
    assert _dec(lib, npg=0) == A.ATTN_ERR_BAD_SHAPE
    assert _dec(lib, ns=-1) == A.ATTN_ERR_BAD_SHAPE
    assert _dec(lib, kc=0x1004) == A.ATTN_ERR_ALIGN
    assert _dec(lib, sl=0x1002) == A.ATTN_ERR_ALIGN
    assert _dec(lib, ps=1 << 16, npg=1 << 15) == A.ATTN_ERR_BAD_SHAPE  # 2^31 cache rows: indices are 32-bit
    assert _dec(lib, B=0) == A.ATTN_OK


def test_decode_workspace_bytes():
    import exact_softmax_attention_gb300 as A
    assert A.attn_decode_workspace_bytes(64, 32, 128, 19) == 64 * 32 * 19 * 129 * 4
    assert A.attn_decode_workspace_bytes(64, 32, 128, 1) == 0  # one split writes o and lse directly
    assert A.attn_decode_workspace_bytes(0, 32, 128, 4) == 0
    _, splits = A.attn_decode_plan(64, 32, 8, 2048, 16, 0, 152)
    assert A.attn_decode_workspace_bytes(64, 32, 128, splits) < 32 << 20  # the decode workload fits the no-alloc array


def test_hd_host_validation(lib):
    import exact_softmax_attention_gb300 as A
    f = lib.attn_fwd_hd
    vp, i = ctypes.c_void_p, ctypes.c_int
    f.argtypes = [vp] * 5 + [i] * 7 + [ctypes.c_float, i, vp, vp]
    call = lambda d, dv, B=1, cu=None: f(16, 16, 16, 16, 16, B, 2, 2, 64, 64, d, dv, 0.1, 1, cu, None)
    assert call(192, 64) == A.ATTN_ERR_BAD_SHAPE
    assert call(128, 192) == A.ATTN_ERR_BAD_SHAPE
    assert call(96, 96) == A.ATTN_ERR_BAD_SHAPE
    assert call(256, 128) == A.ATTN_ERR_BAD_SHAPE
    assert call(192, 128, B=0) == A.ATTN_OK


def _dec8(lib, fmt=0, kds=0.5, vds=2.0, **kw):
    f = lib.attn_decode_paged_fp8
    vp = ctypes.c_void_p
    f.argtypes = ([vp, vp, vp, vp, vp, ctypes.c_int, vp, vp, vp] + [ctypes.c_int] * 6 +
                  [ctypes.c_float, ctypes.c_int, ctypes.c_int, ctypes.c_float, ctypes.c_float])
    a = dict(q=16, kc=16, vc=16, pt=16, sl=16, ps=16, o=16, lse=16, B=1, Hq=8, Hkv=2, d=128, mp=4, npg=4,
             scale=0.1, ns=0)
    a.update(kw)
    return f(a["q"], a["kc"], a["vc"], a["pt"], a["sl"], a["ps"], a["o"], a["lse"], None, a["B"], a["Hq"], a["Hkv"],
             a["d"], a["mp"], a["npg"], a["scale"], a["ns"], fmt, kds, vds)


def test_fp8_decode_host_validation(lib):
    import exact_softmax_attention_gb300 as A
    assert _dec8(lib, fmt=2) == A.ATTN_ERR_BAD_ARG
    assert _dec8(lib, fmt=-1) == A.ATTN_ERR_BAD_ARG
    assert _dec8(lib, kds=float("inf")) == A.ATTN_ERR_BAD_ARG
    assert _dec8(lib, vds=float("nan")) == A.ATTN_ERR_BAD_ARG
    assert _dec8(lib, kds=1e30, scale=1e30) == A.ATTN_ERR_BAD_ARG  # score scale overflows
    assert _dec8(lib, pt=None) == A.ATTN_ERR_NULL_PTR
    assert _dec8(lib, d=96) == A.ATTN_ERR_BAD_SHAPE
    assert _dec8(lib, vc=0x1008) == A.ATTN_ERR_ALIGN
    assert _dec8(lib, ps=3, npg=(1 << 31) // 3 + 1) == A.ATTN_ERR_BAD_SHAPE
    assert _dec8(lib, fmt=1, B=0) == A.ATTN_OK


@pytest.mark.parametrize("B,Hq,Hkv,mp,ps,ns", [(64, 32, 8, 2048, 16, 0), (1, 1, 1, 1, 1, 0), (3, 4, 2, 10, 7, 4),
                                               (64, 32, 8, 2048, 16, 5), (8, 8, 1, 100, 1, 1), (64, 32, 1, 2048, 16, 0)])
def test_decode_plan(B, Hq, Hkv, mp, ps, ns):
    import exact_softmax_attention_gb300 as A
    chunk, splits = A.attn_decode_plan(B, Hq, Hkv, mp, ps, ns, num_sms=152)
    lmax = mp * ps
    assert chunk % 64 == 0 and chunk >= 64
    assert splits * chunk >= lmax and (splits - 1) * chunk < lmax
    if ns > 0:
        assert splits <= ns
    elif lmax >= 128 * (Hq // Hkv):
        assert chunk >= 128 * (Hq // Hkv)  # partials of many query heads per kv head stay small


def test_decode_plan_rejects_bad_heads():
    import exact_softmax_attention_gb300 as A
    for hq, hkv in ((0, 1), (6, 4)):
        with pytest.raises(A.AttnError):
            A.attn_decode_plan(2, hq, hkv, 10, 16, 0, num_sms=152)


def test_options_roundtrip():
    import exact_softmax_attention_gb300 as A
    A.attn_set_option("rescale_threshold", 4.0)
    assert A.attn_get_option("rescale_threshold") == 4.0
    A.attn_set_option("rescale_threshold", 8.0)
    with pytest.raises(A.AttnError):
        A.attn_set_option("no_such_option", 1)
    with pytest.raises(A.AttnError):
        A.attn_set_option("exp_poly", 3)
    # forward pipeline switches: 0 or 1 only
    for name, default in (("correction", 0), ("unroll_kv", 0), ("packed_order", 1), ("dynamic_order", 1),
                          ("decode_order", 1), ("decode_maps", 1)):
        assert A.attn_get_option(name) == default
        A.attn_set_option(name, 1 - default)
        assert A.attn_get_option(name) == 1 - default
        A.attn_set_option(name, default)
        with pytest.raises(A.AttnError):
            A.attn_set_option(name, 2)
    assert "sm_103a" in A.attn_version()
    assert A.status_string(A.ATTN_ERR_DEVICE_TIMEOUT).startswith("a kernel gave up")


def test_page_divisor_scheme():
    """The decode kernels divide token indices by the page size with a multiply and a shift:
    m = ceil(2^(31+k) / page_size), k = ceil(log2 page_size), quotient (tok * m >> 32) >> (k - 1).
    Exact for every 31-bit tok (the bound the launcher relies on), checked here on the edges."""
    import random
    rng = random.Random(5)
    sizes = list(range(2, 2100)) + [2 ** j for j in range(1, 31)] + [2 ** j + 1 for j in range(1, 31)] + \
        [2 ** j - 1 for j in range(2, 32)] + [rng.randrange(2, 2 ** 31) for _ in range(300)]
    for d in sizes:
        k = (d - 1).bit_length()
        m = -(-(1 << (31 + k)) // d)
        assert m < 1 << 32
        top = (1 << 31) - 1
        ns = {0, 1, d - 1, d, d + 1, top, top - top % d, top - top % d - 1} | {rng.randrange(0, 1 << 31) for _ in range(20)}
        for n in ns:
            if 0 <= n <= top:
                assert ((n * m) >> 32) >> (k - 1) == n // d, (d, n)

