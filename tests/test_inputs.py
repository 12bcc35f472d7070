"""Checks of the seeded input generator against its published definitions."""
import numpy as np
import pytest
import torch

from attention_forward_flashattention_gb300 import inputs as I

MASK = (1 << 64) - 1


def _splitmix_scalar(seed, n):
    """SplitMix64 written out on Python ints (reference form of the finaliser)."""
    z = ((seed << 32) + (n + 1) * 0x9E3779B97F4A7C15) & MASK
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK
    return z ^ (z >> 31)


def test_splitmix_seed0_published_first_output():
    # First output of SplitMix64 from state 0 (the widely published value).
    assert int(I.splitmix64(0, 0, 1)[0]) == 0xE220A8397B1DCDAF


def test_splitmix_vectorised_equals_scalar():
    got = I.splitmix64(4007, 123, 64)
    want = [_splitmix_scalar(4007, 123 + i) for i in range(64)]
    assert [int(x) for x in got] == want


def test_normal_slices_are_consistent():
    full = I.normal(77, 1001)
    assert np.array_equal(I.normal(77, 500, 301), full[301:801])
    assert np.array_equal(I.normal(77, 1, 1000), full[1000:])


def test_normal_moments():
    z = I.normal(123, 1 << 20)
    assert abs(z.mean()) < 5.0 / np.sqrt(z.size)
    assert abs(z.var() - 1.0) < 5.0 * np.sqrt(2.0 / z.size)
    assert abs(np.mean(np.abs(z) < 1.0) - 0.6826894921) < 0.003


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.standard_normal(100000) * 10.0 ** rng.integers(-6, 6, 100000),
                        [0.0, -0.0, 1.0, 3.0, 65504.0, 1e-40]])
    want = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(I.to_bf16_bits(x), want)


def test_fp16_rounding_is_nearest():
    # Correct rounding: no other binary16 value is closer to x than the chosen one.
    rng = np.random.default_rng(4)
    x = rng.standard_normal(100000) * 10.0 ** rng.integers(-8, 4, 100000)
    h = I.to_fp16_bits(x).view(np.float16)
    up = np.nextafter(h, np.float16(np.inf)).astype(np.float64)
    dn = np.nextafter(h, np.float16(-np.inf)).astype(np.float64)
    err = np.abs(h.astype(np.float64) - x)
    assert np.all(err <= np.abs(up - x)) and np.all(err <= np.abs(dn - x))


def test_tensor_bits_deterministic_and_chunk_free():
    w = I.WORKLOADS["mha_b1_h2_n256_d64_fp16"]
    a = I.tensor_bits(w, 1)
    b = I.tensor_bits(w, 1, chunk=4096 + 7)
    assert np.array_equal(a, b)
    assert a.shape == (1, 2, 256, 64)
    assert not np.array_equal(I.tensor_bits(w, 0), a)


def test_q_multiplier():
    w = I.custom("t", 1, 1, 64, 64, "bf16", True, 9, q_mult=3.0)
    w1 = I.custom("t", 1, 1, 64, 64, "bf16", True, 9)
    z = I.normal(w.seed * 4 + 0, 64 * 64)
    assert np.array_equal(I.tensor_bits(w, 0).reshape(-1), I.to_bf16_bits(3.0 * z))
    assert np.array_equal(I.tensor_bits(w1, 0).reshape(-1), I.to_bf16_bits(z))


@pytest.mark.parametrize("name", I.WORKLOAD_ORDER)
def test_workload_flops(name):
    w = I.WORKLOADS[name]
    f = 4.0 * w.B * w.H * w.N ** 2 * w.d
    assert w.flops == (f / 2 if w.causal else f)


def test_e4m3_values_match_torch():
    torch = pytest.importorskip("torch")
    want = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = I.e4m3_values()
    assert np.array_equal(np.isnan(got), np.isnan(want))
    assert np.array_equal(got[~np.isnan(got)], want[~np.isnan(want)])


def test_e4m3_rounding_matches_torch_and_saturates():
    torch = pytest.importorskip("torch")
    x = np.random.default_rng(3).standard_normal(200000) * 60.0
    ties = np.array([1.0625, 1.1875, -1.0625, 2.0 ** -10, 3 * 2.0 ** -10, 464.0, 1e6, -1e6])
    # float32 values: torch rounds from float32 (a float64 is first rounded to
    # float32 there), the encoder rounds once from the exact value
    x = np.concatenate([x, ties]).astype(np.float32).astype(np.float64)
    got = I.to_e4m3_bits(x)
    want = torch.from_numpy(np.clip(x, -448.0, 448.0).astype(np.float32)).to(
        torch.float8_e4m3fn).view(torch.uint8)
    assert np.array_equal(got, want.numpy())
    assert list(I.e4m3_values()[I.to_e4m3_bits(np.array([1.0625, 1.1875, 464.0, -1e6]))]) == \
        [1.0, 1.25, 448.0, -448.0]


def test_fp8_inputs_scales_and_layout():
    w = I.custom("fp8in", 1, 2, 300, 128, "e4m3", False, 21)
    f = I.fp8_inputs(w)
    assert f.q.dtype == np.uint8 and f.vt.shape == (1, 2, 128, 304)
    assert f.k_scales.shape == (1, 2, 3) and f.k_scales.dtype == np.float32
    assert np.all(f.vt[..., 300:] == 0)
    vals = I.e4m3_values()
    # every K block's largest code is the largest finite value (scale = amax / 448)
    for t in range(3):
        assert np.abs(vals[f.k[:, :, 128 * t:128 * (t + 1)]]).max() == 448.0
    # decoded Q approximates the normals within half an e4m3 spacing (relative 2^-4)
    zq = I.normal(w.seed * 4, 1 * 2 * 300 * 128).reshape(1, 2, 300, 128)
    approx = vals[f.q] * f.q_scale
    assert np.all(np.abs(approx - zq) <= np.abs(zq) * 2.0 ** -4 + 2.0 ** -10 * f.q_scale + 1e-12)


def test_e4m3_rounding_is_single_rounding_from_float64():
    # just below / above a tie between two e4m3 values: no detour through float32
    below, above = np.nextafter(0.59375, 0.0), np.nextafter(1.5625, 2.0)
    vals = I.e4m3_values()[I.to_e4m3_bits(np.array([below, 0.59375, above, 1.5625]))]
    assert list(vals) == [0.5625, 0.625, 1.625, 1.5]
