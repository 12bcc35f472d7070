"""The 8-bit (e4m3) forward on the GPU.

* building blocks: e4m3 tcgen05 products with both operands in shared memory
  and with A in tensor memory, and the kernel's float -> e4m3 packer (byte
  order, ties to even, saturation) against the host encoder;
* parity with the fp64 oracle: every element of small problems, sampled rows
  of the full-size workloads. The bound per element is the oracle's bound for
  weights rounded to e4m3 (see oracle.attn_fp8) plus 2e-3 for fp32
  accumulation, plus half a bf16 spacing of the exact value (output rounding);
  the LSE, computed from unrounded weights, must agree within 1e-3.
"""
import ctypes
import functools

import numpy as np
import pytest

import attention_forward_flashattention_gb300 as fa
from attention_forward_flashattention_gb300 import build as fabuild
from attention_forward_flashattention_gb300 import inputs as I

from parity_util import bits_to_f64, half_ulp, record, to_bits

pytestmark = pytest.mark.gpu

SLACK = 2e-3
LSE_MAX_ABS = 1e-3


@pytest.fixture(scope="module")
def slib():
    import torch
    torch.cuda.init()
    _, path = fabuild.build()
    lib = ctypes.CDLL(path)
    vp, i = ctypes.c_void_p, ctypes.c_int
    lib.fa_selftest_gemm_qk_fp8.argtypes = [vp, vp, vp, vp, vp]
    lib.fa_selftest_gemm_ts_fp8.argtypes = [vp, vp, vp, vp, vp]
    lib.fa_selftest_pack_e4m3.argtypes = [vp, vp, i, vp]
    fa.load_library()
    return lib


def _dev_u8(x):
    import torch
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.uint8)).to("cuda:0")


def _status():
    import torch
    return torch.zeros(4, dtype=torch.int32, device="cuda:0")


def _codes(rng, shape, scale=1.0):
    return I.to_e4m3_bits(rng.standard_normal(shape) * scale)


def test_gemm_qk_fp8_matches_host(slib):
    import torch
    rng = np.random.default_rng(81)
    a, b = _codes(rng, (128, 128), 8.0), _codes(rng, (128, 128), 8.0)
    c = torch.full((128, 128), float("nan"), dtype=torch.float32, device="cuda:0")
    st = _status()
    da, db = _dev_u8(a), _dev_u8(b)
    rc = slib.fa_selftest_gemm_qk_fp8(da.data_ptr(), db.data_ptr(), c.data_ptr(), st.data_ptr(),
                                      None)
    torch.cuda.synchronize()
    assert rc == 0 and int(st[0]) == 0
    vals = I.e4m3_values()
    ref = vals[a] @ vals[b].T
    tol = 1e-6 * (np.abs(vals[a]) @ np.abs(vals[b]).T) + 1e-6
    assert np.all(np.abs(c.cpu().numpy() - ref) <= tol)


def test_gemm_ts_fp8_a_from_tmem(slib):
    import torch
    rng = np.random.default_rng(82)
    p = I.to_e4m3_bits(rng.random((128, 128)) * 4.0)        # P-like weights, row-major
    bt = _codes(rng, (128, 128), 4.0)                        # V^T: [output column][key]
    words = p.reshape(128, 32, 4).copy().view(np.uint32).reshape(128, 32)  # key 4c+i in byte i
    c = torch.full((128, 128), float("nan"), dtype=torch.float32, device="cuda:0")
    st = _status()
    dw = torch.from_numpy(words.view(np.int32)).to("cuda:0")
    db = _dev_u8(bt)
    rc = slib.fa_selftest_gemm_ts_fp8(dw.data_ptr(), db.data_ptr(), c.data_ptr(), st.data_ptr(),
                                      None)
    torch.cuda.synchronize()
    assert rc == 0 and int(st[0]) == 0
    vals = I.e4m3_values()
    ref = vals[p] @ vals[bt].T
    tol = 1e-6 * (np.abs(vals[p]) @ np.abs(vals[bt]).T) + 1e-6
    assert np.all(np.abs(c.cpu().numpy() - ref) <= tol)


def test_pack_e4m3_matches_host_encoder(slib):
    import torch
    rng = np.random.default_rng(83)
    x = np.concatenate([rng.random(4096) * 300.0, rng.random(4096) * 2.0 ** -5,
                        [1.0625, 1.1875, 2.0 ** -10, 3 * 2.0 ** -10, 448.0, 464.0, 1e5, 0.0,
                         256.0, 255.0, 1.0, 0.5]])
    x = np.concatenate([x, np.zeros((-x.size) % 4)]).astype(np.float32)
    out = torch.zeros(x.size // 4, dtype=torch.int32, device="cuda:0")
    dx = torch.from_numpy(x).to("cuda:0")
    rc = slib.fa_selftest_pack_e4m3(dx.data_ptr(), out.data_ptr(), x.size // 4, None)
    torch.cuda.synchronize()
    assert rc == 0
    got = out.cpu().numpy().view(np.uint32).view(np.uint8)   # little endian: element 4i+k in byte k
    assert np.array_equal(got, I.to_e4m3_bits(x.astype(np.float64)))


# ------------------------------------------------------------ forward parity

def _run_fp8(f, w, pair=False):
    """fa_fwd_fp8 (or fa_fwd_fp8_pair) on the inputs; O bits and LSE."""
    import torch
    q8, k8, vt8 = (_dev_u8(t) for t in (f.q, f.k, f.vt))
    ks = torch.from_numpy(np.ascontiguousarray(f.k_scales)).to("cuda:0")
    o = torch.full((w.B, w.H, w.N, w.d), float("nan"), dtype=torch.bfloat16, device="cuda:0")
    lse = torch.full((w.B, w.H, w.N), float("nan"), dtype=torch.float32, device="cuda:0")
    fa.attention_forward_fp8_into(q8, k8, vt8, o, lse, f.q_scale, ks, f.v_scale, w.causal,
                                  w.scale, pair=pair)
    torch.cuda.synchronize()
    assert fa.fa_check(0) == fa.FA_OK
    return to_bits(o), lse.cpu().numpy()


def _check(o_bits, lse, o_ref, l_ref, bound, what):
    o = bits_to_f64(o_bits, "bf16")
    err = np.abs(o - o_ref)
    lerr = np.abs(lse.astype(np.float64) - l_ref)
    limit = bound + SLACK + half_ulp(o_ref, "bf16")
    record(what, {"o_max_abs": float(err.max()), "o_mean_abs": float(err.mean()),
                  "o_max_over_limit": float((err - limit).max()),
                  "bound_mean": float(bound.mean()), "lse_max_abs": float(lerr.max()),
                  "elements": int(err.size)})
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse)), what
    assert np.all(err <= limit), (what, float((err - limit).max()), float(err.max()))
    assert float(lerr.max()) <= LSE_MAX_ABS, (what, float(lerr.max()))
    # the rounded-weight bound is a worst case; typical errors sit far below it
    assert float(err.mean()) <= float(bound.mean()), what


SMALL = [
    # B, H, N, causal, q_mult
    (1, 2, 256, False, 1.0),
    (1, 2, 300, True, 1.0),
    (2, 3, 1000, False, 1.0),
    (1, 1, 1, True, 1.0),
    (1, 4, 17, False, 1.0),
    (1, 2, 1024, True, 3.0),
    (1, 400, 100, False, 1.0),
]


@pytest.mark.parametrize("pair", [False, True], ids=["auto", "cta_pair"])
@pytest.mark.parametrize("B,H,N,causal,q_mult", SMALL)
def test_fp8_small_every_element(slib, oracle_mod, B, H, N, causal, q_mult, pair):
    w = I.custom("fp8small", B, H, N, 128, "e4m3", causal, 400 + N, q_mult)
    f = I.fp8_inputs(w)
    o, lse = _run_fp8(f, w, pair)
    o_ref, l_ref, bound = oracle_mod.attn_fp8(f.q, f.k, f.vt, f.q_scale, f.k_scales, f.v_scale,
                                              causal, w.scale)
    _check(o.reshape(-1, 128), lse.reshape(-1), o_ref, l_ref, bound,
           f"fp8{' pair' if pair else ''} B{B} H{H} N{N}")


# fa_fwd_fp8 runs the one-CTA kernel (the CTA pair measured slower on 8-bit
# inputs): fa_fwd_fp8_pair must reproduce its bits, at both named 8-bit shapes
# among others.
ONE_CTA_SHAPES = [
    # B, H, N, causal, q_mult
    (1, 4, 2048, False, 1.0),
    (2, 3, 1000, False, 1.0),
    (1, 2, 777, False, 3.0),
    (2, 4, 1536, True, 1.0),
    (1, 3, 1000, True, 3.0),
    (4, 16, 4096, True, 1.0),
    (4, 16, 4096, False, 1.0),
]


@pytest.mark.parametrize("B,H,N,causal,q_mult", ONE_CTA_SHAPES)
def test_fp8_pair_matches_one_cta_bitwise(slib, B, H, N, causal, q_mult):
    w = I.custom("fp8pairbits", B, H, N, 128, "e4m3", causal, 500 + N, q_mult)
    f = I.fp8_inputs(w)
    o1, l1 = _run_fp8(f, w)
    o2, l2 = _run_fp8(f, w, pair=True)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2), (B, H, N, causal)


@functools.lru_cache(maxsize=1)
def _named(name):
    return I.fp8_inputs(I.FP8_WORKLOADS[name])


@pytest.mark.parametrize("name", list(I.FP8_WORKLOADS))
def test_fp8_named_workload_every_element(slib, oracle_mod, name):
    w = I.FP8_WORKLOADS[name]
    f = _named(name)
    o, lse = _run_fp8(f, w)
    o_ref, l_ref, bound = oracle_mod.attn_fp8(f.q, f.k, f.vt, f.q_scale, f.k_scales, f.v_scale,
                                              w.causal, w.scale)
    _check(o.reshape(-1, 128), lse.reshape(-1), o_ref, l_ref, bound, name)


def test_fp8_deterministic(slib):
    w = I.custom("fp8det", 2, 4, 700, 128, "e4m3", True, 77)
    f = I.fp8_inputs(w)
    o1, l1 = _run_fp8(f, w)
    o2, l2 = _run_fp8(f, w)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_masked_keys_never_set_the_reference(slib, oracle_mod, causal):
    """Causal: keys 128.. score far above keys 0..127 (masked for rows
    0..127 on a whole KV tile). Non-causal, N = 200: every visible score is
    far below zero while the zero-filled keys past N would score 0. Either
    way a reference taken from a masked score underflows whole rows."""
    N = 384 if causal else 200
    B, H, d = 1, 2, 128
    w = I.custom("fp8mask", B, H, N, d, "e4m3", causal, 900 + N)
    rng = np.random.default_rng(N)
    q = np.zeros((B, H, N, d))
    q[..., 0] = 16.0
    k = np.zeros((B, H, N, d))
    k[..., 0] = np.where(np.arange(N) >= 128, 16.0, 0.0) if causal else -16.0
    nt = (N + 127) // 128
    k_scales = np.full((B, H, nt), 16.0, dtype=np.float32)   # scores 16 * 16 * 16 * scale
    ldv = (N + 15) // 16 * 16
    vt = np.zeros((B, H, d, ldv), dtype=np.uint8)
    vt[:, :, :, :N] = I.to_e4m3_bits(rng.standard_normal((B, H, N, d)) / 4.0).transpose(0, 1, 3, 2)
    f = I.Fp8Inputs(I.to_e4m3_bits(q), I.to_e4m3_bits(k), vt, 1.0, k_scales, 4.0)
    o, lse = _run_fp8(f, w)
    o_ref, l_ref, bound = oracle_mod.attn_fp8(f.q, f.k, f.vt, f.q_scale, f.k_scales, f.v_scale,
                                              causal, w.scale)
    # every weight is 0 or 1 (exact in e4m3), so the rounded-weight bound is
    # ~0: check the per-element limit and the LSE, not the mean against it
    got = bits_to_f64(o.reshape(-1, 128), "bf16")
    assert np.all(np.isfinite(got)) and np.all(np.isfinite(lse)), causal
    assert np.all(np.abs(got - o_ref) <= bound + SLACK + half_ulp(o_ref, "bf16")), causal
    assert float(np.abs(lse.reshape(-1).astype(np.float64) - l_ref).max()) <= LSE_MAX_ABS, causal
