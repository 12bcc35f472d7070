"""Seeded random shapes, forward and backward, every element against the fp64
oracle: B, H, N (ragged, 1 to 1100), d, dtype and causality drawn from a fixed
generator, so that tile edges, unit boundaries, short causal units and both
MMA issue layouts of each head dimension are exercised together. The bounds
are those of the dedicated parity tests (forward, N(0, 1) inputs: 1e-2 per
element, 1e-3 mean, 1e-3 on the LSE, through parity_util.compare; backward: 4
unit roundoffs of the term magnitudes plus half a spacing). Each 16-bit case also runs the strided entry
point on randomly chosen storage layouts, which must reproduce the contiguous
result bit for bit; a second set of random shapes covers the e4m3 forward
against the oracle's per-element bound for weights rounded to 8 bits."""
import numpy as np
import pytest

import attention_forward_flashattention_gb300 as fa
from attention_forward_flashattention_gb300 import inputs as I

from parity_util import bits_to_f64, compare, half_ulp, record, to_bits, to_device
from test_gpu_parity import _in_layout

pytestmark = pytest.mark.gpu

EPS = {"fp16": 2.0 ** -11, "bf16": 2.0 ** -8}


def _layouts(k):
    rng = np.random.default_rng(7000 + k)
    return tuple(str(rng.choice(["bhnd", "bnhd", "pad"])) for _ in range(4))


def _cases(n=48, seed=20261202):
    rng = np.random.default_rng(seed)
    out = []
    for k in range(n):
        d = int(rng.choice([64, 128]))
        dtype = str(rng.choice(["fp16", "bf16"]))
        causal = bool(rng.integers(0, 2))
        N = int(rng.integers(1, 1101))
        B = int(rng.integers(1, 3))
        H = int(rng.integers(1, 4))
        out.append((k, B, H, N, d, dtype, causal))
    return out


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    torch.cuda.init()
    fa.build.build()
    fa.load_library()


@pytest.mark.parametrize("k,B,H,N,d,dtype,causal", _cases())
def test_random_shape_forward_and_backward(oracle_mod, k, B, H, N, d, dtype, causal):
    import torch
    w = I.custom(f"rand{k}", B, H, N, d, dtype, causal, seed_index=3000 + k)
    q, kk, v = I.qkv_bits(w)
    dob = I.dout_bits(w)
    qd, kd, vd, dod = (to_device(x, dtype) for x in (q, kk, v, dob))
    o, lse = fa.attention_forward(qd, kd, vd, causal=causal, scale=w.scale)
    dq, dk, dv = fa.attention_backward(qd, kd, vd, o, lse, dod, causal=causal, scale=w.scale)
    torch.cuda.synchronize()
    assert fa.fa_check(0) == fa.FA_OK

    o_ref, l_ref = oracle_mod.attn_fwd(q, kk, v, dtype, causal, w.scale)
    res = compare(to_bits(o), lse.cpu().numpy(), o_ref, l_ref, dtype)
    record(f"random {k} B{B} H{H} N{N} d{d} {dtype} causal={int(causal)}", res)
    assert res["ok"], (k, res)

    # the same problem through strided views: identical bits
    lq, lk, lv, lo = _layouts(k)
    os_ = _in_layout(torch.full_like(o, float("nan")), lo)
    ls_ = torch.full_like(lse, float("nan"))
    fa.attention_forward_into(_in_layout(qd, lq), _in_layout(kd, lk), _in_layout(vd, lv), os_, ls_,
                              causal=causal, scale=w.scale)
    torch.cuda.synchronize()
    assert fa.fa_check(0) == fa.FA_OK
    assert np.array_equal(to_bits(os_.contiguous()), to_bits(o)), (k, (lq, lk, lv, lo))
    assert np.array_equal(ls_.cpu().numpy(), lse.cpu().numpy()), k

    g = oracle_mod.attn_bwd(q, kk, v, dob, dtype, causal, w.scale)
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        ref = g[name]
        got = bits_to_f64(to_bits(t), dtype).reshape(ref.shape)
        limit = 4 * EPS[dtype] * g["mag_" + name] + half_ulp(ref, dtype) + 1e-6
        bad = np.abs(got - ref) > limit
        assert np.all(np.isfinite(got)) and not bad.any(), (k, name, int(bad.sum()))


def _fp8_cases(n=24, seed=20261203):
    rng = np.random.default_rng(seed)
    return [(k, int(rng.integers(1, 3)), int(rng.integers(1, 4)), int(rng.integers(1, 1101)),
             bool(rng.integers(0, 2)), float(rng.choice([0.5, 1.0, 2.0]))) for k in range(n)]


@pytest.mark.parametrize("k,B,H,N,causal,q_mult", _fp8_cases())
def test_random_shape_fp8_forward(oracle_mod, k, B, H, N, causal, q_mult):
    import torch
    w = I.custom(f"rand8_{k}", B, H, N, 128, "e4m3", causal, 5000 + k, q_mult)
    f = I.fp8_inputs(w)
    dev = [torch.from_numpy(np.ascontiguousarray(t, dtype=np.uint8)).to("cuda:0")
           for t in (f.q, f.k, f.vt)]
    ks = torch.from_numpy(np.ascontiguousarray(f.k_scales)).to("cuda:0")
    o = torch.full((B, H, N, 128), float("nan"), dtype=torch.bfloat16, device="cuda:0")
    lse = torch.full((B, H, N), float("nan"), dtype=torch.float32, device="cuda:0")
    fa.attention_forward_fp8_into(*dev, o, lse, f.q_scale, ks, f.v_scale, causal, w.scale)
    torch.cuda.synchronize()
    assert fa.fa_check(0) == fa.FA_OK
    o_ref, l_ref, bound = oracle_mod.attn_fp8(f.q, f.k, f.vt, f.q_scale, f.k_scales, f.v_scale,
                                              causal, w.scale)
    got = bits_to_f64(to_bits(o).reshape(-1, 128), "bf16")
    err = np.abs(got - o_ref)
    assert np.all(np.isfinite(got)), k
    assert np.all(err <= bound + 2e-3 + half_ulp(o_ref, "bf16")), (k, float(err.max()))
    assert float(np.abs(lse.cpu().numpy().reshape(-1).astype(np.float64) - l_ref).max()) <= 1e-3, k
