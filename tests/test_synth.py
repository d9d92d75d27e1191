"""The seeded input generator: published splitmix64 values, rounding, determinism, recipes."""
import numpy as np
import pytest

import synth
from synth import workloads as W


def test_splitmix64_published_sequence():
    # splitmix64 started from state 0 (the values of its published reference implementation)
    assert synth.splitmix64_at(0, 0) == 0xE220A8397B1DCDAF
    assert synth.splitmix64_at(0, 1) == 0x6E789E6AA1B965F4
    assert synth.splitmix64_at(0, 2) == 0x06C45D188009454F


def test_bf16_round_to_nearest_even():
    one = np.float32(1.0)
    assert synth.f32_to_bf16([one])[0] == 0x3F80
    assert synth.f32_to_bf16([np.float32(1 + 2**-8)])[0] == 0x3F80          # tie -> even
    assert synth.f32_to_bf16([np.float32(1 + 3 * 2**-8)])[0] == 0x3F82      # tie -> even
    assert synth.f32_to_bf16([np.float32(1 + 2**-8 + 2**-20)])[0] == 0x3F81  # above tie
    assert synth.f32_to_bf16([np.float32(np.nan)])[0] == 0x7FC0


def test_normals_deterministic_and_standard():
    a = synth.normal_bf16((1 << 20,), 5)
    b = synth.normal_bf16((1 << 20,), 5)
    np.testing.assert_array_equal(a, b)
    x = synth.bf16_to_f32(a).astype(np.float64)
    assert abs(x.mean()) < 5e-3 and abs(x.std() - 1) < 5e-3
    # element i does not depend on the array length
    np.testing.assert_array_equal(synth.normal_bf16((1000,), 5), a[:1000])
    # the multiplier is applied before rounding
    y = synth.bf16_to_f32(synth.normal_bf16((1000,), 5, 2.0)).astype(np.float64)
    assert np.abs(y - 2 * x[:1000]).max() <= 2 * np.abs(x[:1000]).max() * 2**-8


def test_uniform_ints_and_permutation():
    u = synth.uniform_ints(100000, 3, 512, 4096)
    assert u.min() >= 512 and u.max() <= 4096 and abs(u.mean() - 2304) < 20
    p = synth.permutation(1000, 8)
    assert sorted(p.tolist()) == list(range(1000)) and not np.array_equal(p, np.arange(1000))


def test_workload_recipes():
    v = W.varlen_gqa()
    lens = np.diff(v.cu_seqlens)
    assert len(lens) == 8 and lens.min() >= 512 and lens.max() <= 4096
    d = W.decode()
    assert d.seqlens.min() >= 1024 and d.seqlens.max() <= 32768 and d.B == 64
    pt = d.page_table()
    used = np.concatenate([pt[b, : int(n)] for b, n in enumerate(d.pages_per_seq)])
    assert sorted(used.tolist()) == list(range(d.num_pages))


def test_exact_work_counts():
    assert W.tiny().flops() == 33_554_432
    assert W.prefill(False).flops() == 68_719_476_736
    assert W.prefill(True).flops() == 34_376_515_584
    assert W.long_causal().flops() == 549_822_922_752
    v = W.varlen_gqa()
    lens = np.diff(v.cu_seqlens).astype(np.int64)
    assert v.flops() == 4 * 128 * 32 * int((lens * (lens + 1) // 2).sum())
    assert W.tiny().bytes() == 262_144 + 2_048
    d = W.decode()
    assert d.bytes() == (int(d.seqlens.astype(np.int64).sum()) * 8 * 128 * 4 + 2 * 64 * 32 * 128 * 2
                         + 64 * 32 * 4 + int(d.pages_per_seq.sum()) * 4 + 64 * 4)


def test_fp8_encoder_rounds_like_torch_and_saturates():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(5)
    for fmt, td in (("e4m3", torch.float8_e4m3fn), ("e5m2", torch.float8_e5m2)):
        mx = synth.FP8_MAX[fmt]
        x = np.concatenate([rng.standard_normal(50000) * mx / 8, rng.standard_normal(1000) * 1e-4, [0.0, -0.0, mx, -mx]])
        x = np.clip(x, -mx, mx)
        ours = synth.fp8_encode(x, fmt)
        ref = torch.from_numpy(x).to(td).view(torch.uint8).numpy()
        np.testing.assert_array_equal(ours, ref)
        big = synth.fp8_encode(np.array([10 * mx, -10 * mx]), fmt)  # saturates at the largest finite code
        assert list(big) == ([0x7E, 0xFE] if fmt == "e4m3" else [0x7B, 0xFB])


def test_fp8_decode_workload_halves_the_cache_bytes():
    from synth import workloads as W
    bf, f8 = W.decode(), W.decode_fp8()
    L = int(bf.seqlens.astype(np.int64).sum())
    assert bf.bytes() - f8.bytes() == L * bf.Hkv * bf.d * 2
