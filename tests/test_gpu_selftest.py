"""GPU unit tests of the kernel's building blocks (TMA + SW128 panels,
tcgen05.mma descriptors, TMEM lane-quarter read-back, bounded waits)."""
import ctypes

import numpy as np
import pytest

from attention_forward_flashattention_gb300 import build as fabuild
from attention_forward_flashattention_gb300 import inputs as I

from parity_util import bits_to_f64, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def slib():
    import torch
    torch.cuda.init()
    _, path = fabuild.build()
    lib = ctypes.CDLL(path)
    vp, i = ctypes.c_void_p, ctypes.c_int
    lib.fa_selftest_gemm_qk.argtypes = [vp, vp, vp, i, i, vp, vp]
    lib.fa_selftest_gemm_pv.argtypes = [vp, vp, vp, i, i, i, vp, vp]
    lib.fa_selftest_gemm_ts.argtypes = [vp, vp, vp, i, i, vp, vp]
    lib.fa_selftest_gemm_qk_pair.argtypes = [vp, vp, vp, i, i, vp, vp]
    lib.fa_selftest_gemm_pv_pair.argtypes = [vp, vp, vp, i, vp, vp]
    lib.fa_selftest_wait_timeout.argtypes = [vp, vp, vp]
    return lib


def _status():
    import torch
    return torch.zeros(4, dtype=torch.int32, device="cuda:0")


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("K", [64, 128])
def test_gemm_qk_matches_host(slib, K, dtype):
    import torch
    rng = np.random.default_rng(K + (dtype == "bf16"))
    a = I.to_bits(rng.standard_normal((128, K)), dtype)
    b = I.to_bits(rng.standard_normal((128, K)), dtype)
    c = torch.full((128, 128), float("nan"), dtype=torch.float32, device="cuda:0")
    st = _status()
    da, db = to_device(a, dtype), to_device(b, dtype)
    rc = slib.fa_selftest_gemm_qk(da.data_ptr(), db.data_ptr(), c.data_ptr(), K,
                                  int(dtype == "bf16"), st.data_ptr(), None)
    torch.cuda.synchronize()
    assert rc == 0 and int(st[0]) == 0
    ref = bits_to_f64(a, dtype) @ bits_to_f64(b, dtype).T
    np.testing.assert_allclose(c.cpu().numpy(), ref, rtol=1e-5, atol=1e-4)


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("N", [64, 128])
def test_gemm_pv_mn_major_b(slib, N, dtype):
    import torch
    rng = np.random.default_rng(N + 7 * (dtype == "bf16"))
    a = I.to_bits(rng.random((128, 128)), dtype)             # P-like, written by threads
    b = I.to_bits(rng.standard_normal((128, N)), dtype)      # V-like, [key][d]
    ref = bits_to_f64(a, dtype) @ bits_to_f64(b, dtype)
    da, db = to_device(a, dtype), to_device(b, dtype)
    results = {}
    for variant in (0, 1):
        c = torch.full((128, N), float("nan"), dtype=torch.float32, device="cuda:0")
        st = _status()
        rc = slib.fa_selftest_gemm_pv(da.data_ptr(), db.data_ptr(), c.data_ptr(), N,
                                      int(dtype == "bf16"), variant, st.data_ptr(), None)
        torch.cuda.synchronize()
        assert rc == 0 and int(st[0]) == 0
        got = c.cpu().numpy()
        results[variant] = bool(np.allclose(got, ref, rtol=1e-5, atol=1e-4))
    assert results[0], f"MN-major B descriptor mismatch (LBO/SBO swapped variant matches: {results[1]})"


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("N", [64, 128])
def test_gemm_ts_a_from_tmem(slib, N, dtype):
    import torch
    rng = np.random.default_rng(3 * N + (dtype == "bf16"))
    a = I.to_bits(rng.random((128, 128)), dtype)             # P-like, stored into TMEM
    b = I.to_bits(rng.standard_normal((128, N)), dtype)      # V-like, [key][d]
    ref = bits_to_f64(a, dtype) @ bits_to_f64(b, dtype)
    da, db = to_device(a, dtype), to_device(b, dtype)
    c = torch.full((128, N), float("nan"), dtype=torch.float32, device="cuda:0")
    st = _status()
    rc = slib.fa_selftest_gemm_ts(da.data_ptr(), db.data_ptr(), c.data_ptr(), N,
                                  int(dtype == "bf16"), st.data_ptr(), None)
    torch.cuda.synchronize()
    assert rc == 0 and int(st[0]) == 0
    np.testing.assert_allclose(c.cpu().numpy(), ref, rtol=1e-5, atol=1e-4)


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_gemm_qk_on_cta_pair(slib, dtype):
    import torch
    rng = np.random.default_rng(11 + (dtype == "bf16"))
    a = I.to_bits(rng.standard_normal((256, 128)), dtype)   # Q-like, 128 rows per CTA
    b = I.to_bits(rng.standard_normal((128, 128)), dtype)   # K-like, 64 keys per CTA
    c = torch.full((256, 128), float("nan"), dtype=torch.float32, device="cuda:0")
    st = _status()
    da, db = to_device(a, dtype), to_device(b, dtype)   # keep both alive across the launch
    rc = slib.fa_selftest_gemm_qk_pair(da.data_ptr(), db.data_ptr(), c.data_ptr(),
                                       int(dtype == "bf16"), 0, st.data_ptr(), None)
    torch.cuda.synchronize()
    assert rc == 0 and int(st[0]) == 0
    ref = bits_to_f64(a, dtype) @ bits_to_f64(b, dtype).T
    np.testing.assert_allclose(c.cpu().numpy(), ref, rtol=1e-5, atol=1e-4)


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_gemm_pv_on_cta_pair(slib, dtype):
    import torch
    rng = np.random.default_rng(21 + (dtype == "bf16"))
    p = I.to_bits(rng.random((256, 128)), dtype)              # P-like, from TMEM
    v = I.to_bits(rng.standard_normal((128, 128)), dtype)     # V-like, 64 columns per CTA
    c = torch.full((256, 128), float("nan"), dtype=torch.float32, device="cuda:0")
    st = _status()
    dp, dv = to_device(p, dtype), to_device(v, dtype)   # keep both alive across the launch
    rc = slib.fa_selftest_gemm_pv_pair(dp.data_ptr(), dv.data_ptr(), c.data_ptr(),
                                       int(dtype == "bf16"), st.data_ptr(), None)
    torch.cuda.synchronize()
    assert rc == 0 and int(st[0]) == 0
    ref = bits_to_f64(p, dtype) @ bits_to_f64(v, dtype)
    np.testing.assert_allclose(c.cpu().numpy(), ref, rtol=1e-5, atol=1e-4)


def test_bounded_wait_gives_up_and_reports(slib):
    import torch
    st = _status()
    out = torch.full((4,), 7, dtype=torch.int32, device="cuda:0")
    assert slib.fa_selftest_wait_timeout(st.data_ptr(), out.data_ptr(), None) == 0
    torch.cuda.synchronize()
    assert int(out[0]) == 0          # the wait did not complete
    assert int(st[0]) & 32           # and recorded its status bit
    # the context is still usable
    x = torch.arange(10, device="cuda:0").sum()
    assert int(x) == 45
