"""Parity of the CUDA backward (fa_bwd) with the fp64 backward oracle.

The forward runs first (its O and LSE feed the backward, as in training).
Tolerance per element, from the arithmetic: the kernel rounds P and dS to the
16-bit input format X (relative error 2^-11 for fp16, 2^-8 for bf16 each),
forms D from the 16-bit O, and accumulates in fp32; every term of an output
element therefore carries a relative error of at most about three X roundings,
and the element's error is bounded by 4 eps_X times the sum of the magnitudes
of its terms (the oracle's mag_* arrays), plus half an X spacing of the exact
value (output rounding), plus 1e-6.
"""
import functools

import numpy as np
import pytest

import attention_forward_flashattention_gb300 as fa
from attention_forward_flashattention_gb300 import inputs as I

from parity_util import bits_to_f64, half_ulp, record, to_bits, to_device

pytestmark = pytest.mark.gpu

EPS = {"fp16": 2.0 ** -11, "bf16": 2.0 ** -8}


@pytest.fixture(scope="module", autouse=True)
def _built(oracle_mod):
    import torch
    torch.cuda.init()
    fa.build.build()
    fa.load_library()


def _dout_bits(w):
    return I.dout_bits(w)


def _run(w, q, k, v, dob):
    import torch
    qd, kd, vd, dod = (to_device(x, w.dtype) for x in (q, k, v, dob))
    o, lse = fa.attention_forward(qd, kd, vd, causal=w.causal, scale=w.scale)
    dq, dk, dv = fa.attention_backward(qd, kd, vd, o, lse, dod, causal=w.causal, scale=w.scale)
    torch.cuda.synchronize()
    assert fa.fa_check(0) == fa.FA_OK
    return to_bits(dq), to_bits(dk), to_bits(dv)


def _check(got_bits, ref, mag, dtype, what):
    got = bits_to_f64(got_bits, dtype)
    err = np.abs(got - ref)
    limit = 4 * EPS[dtype] * mag + half_ulp(ref, dtype) + 1e-6
    record(what, {"max_abs": float(err.max()), "mean_abs": float(err.mean()),
                  "max_err_over_limit": float((err / limit).max()), "elements": int(err.size)})
    assert np.all(np.isfinite(got)), what
    bad = err > limit
    assert not bad.any(), (what, int(bad.sum()), float((err - limit).max()), float(err.max()))


SMALL = [
    # B, H, N, d, dtype, causal
    (1, 2, 256, 64, "fp16", False),
    (1, 2, 256, 128, "bf16", True),
    (2, 3, 300, 128, "fp16", True),
    (1, 2, 1000, 64, "bf16", False),
    (1, 1, 1, 128, "fp16", False),
    (1, 4, 17, 64, "fp16", True),
    (1, 1, 640, 128, "fp16", False),
    (1, 300, 100, 64, "bf16", True),
]


@pytest.mark.parametrize("B,H,N,d,dtype,causal", SMALL)
def test_bwd_small_every_element(oracle_mod, B, H, N, d, dtype, causal):
    w = I.custom("bwd", B, H, N, d, dtype, causal, seed_index=500 + N + d)
    q, k, v = I.qkv_bits(w)
    dob = _dout_bits(w)
    dq, dk, dv = _run(w, q, k, v, dob)
    g = oracle_mod.attn_bwd(q, k, v, dob, dtype, causal, w.scale)
    shape = (B * H, N, d)
    for name, got in (("dq", dq), ("dk", dk), ("dv", dv)):
        _check(got.reshape(shape), g[name], g["mag_" + name], dtype, f"{name} B{B} H{H} N{N} d{d}")


@functools.lru_cache(maxsize=1)
def _inputs(name):
    w = I.WORKLOADS[name]
    return I.qkv_bits(w) + (_dout_bits(w),)


@pytest.mark.parametrize("name", ["mha_b4_h16_n4096_d128_fp16", "causal_b4_h16_n4096_d128_bf16",
                                  "mha_b2_h32_n8192_d64_fp16",
                                  "causal_b1_h32_n16384_d128_bf16_q3"])
def test_bwd_full_size_sampled_heads(oracle_mod, name):
    w = I.WORKLOADS[name]
    q, k, v, dob = _inputs(name)
    dq, dk, dv = _run(w, q, k, v, dob)
    # two heads; one at N = 16384 (its fp64 N x N buffers take 6.4 GB of host memory)
    heads = np.array([0, w.B * w.H - 1]) if w.N <= 8192 else np.array([w.B * w.H - 1])
    g = oracle_mod.attn_bwd(q, k, v, dob, w.dtype, w.causal, w.scale, heads=heads)
    shape = (w.B * w.H, w.N, w.d)
    for nm, got in (("dq", dq), ("dk", dk), ("dv", dv)):
        _check(got.reshape(shape)[heads], g[nm], g["mag_" + nm], w.dtype, f"{nm} {name}")


def test_bwd_deterministic():
    w = I.custom("bwddet", 2, 3, 700, 128, "bf16", True, seed_index=91)
    q, k, v = I.qkv_bits(w)
    dob = _dout_bits(w)
    a = _run(w, q, k, v, dob)
    b = _run(w, q, k, v, dob)
    assert all(np.array_equal(x, y) for x, y in zip(a, b))
