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
