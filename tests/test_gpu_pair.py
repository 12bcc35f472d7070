"""Parity of the CTA-pair forward (fa_fwd_pair: tcgen05.mma cta_group::2,
M = 256 rows shared by two SMs, head dimension 128) with the fp64 oracle,
under the same bounds as the one-CTA kernel (parity_util.compare), and with
the one-CTA kernel bit for bit (the per-tile arithmetic is the same; a pair
product gives the fp32 sums of two one-CTA products; fa_fwd itself runs the
pair kernel for large non-causal head-dimension-128 problems):

* small problems: ragged N (1, 17, 129, 300, 1000), causal and not, fp16 and
  bf16, more units than pairs, a second row block past N; every element;
* the head-dimension-128 named workloads at full size (C2, C3, C5), every
  element;
* Q = 0 closed forms, masked keys far above the visible ones, sharpened scores
  (the lazy-rescale path), determinism, a side stream, and the SM clock record.
"""
import numpy as np
import pytest

import attention_forward_flashattention_gb300 as fa
from attention_forward_flashattention_gb300 import inputs as I

from parity_util import (bits_to_f64, compare, explain_over, half_ulp, record, to_bits,
                         to_device)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    torch.cuda.init()
    fa.build.build()
    fa.load_library()


def run_pair(q_bits, k_bits, v_bits, dtype, causal, scale, stream=None):
    import torch
    q, k, v = (to_device(x, dtype) for x in (q_bits, k_bits, v_bits))
    o = torch.full_like(q, float("nan"))
    lse = torch.full(q.shape[:3], float("nan"), dtype=torch.float32, device=q.device)
    fa.attention_forward_pair_into(q, k, v, o, lse, causal, scale, stream)
    rc = fa.fa_check(0 if stream is None else int(stream.cuda_stream))
    assert rc == fa.FA_OK, fa.status_string(rc)
    torch.cuda.synchronize()
    return to_bits(o), lse.cpu().numpy()


def _check(res, what):
    record("pair " + what, res)
    assert res["ok"], f"{what}: {res}"


SMALL = [
    # B, H, N, dtype, causal
    (1, 2, 256, "fp16", False),
    (1, 2, 256, "fp16", True),
    (1, 1, 1, "bf16", True),
    (1, 1, 1, "fp16", False),
    (1, 4, 17, "fp16", True),
    (1, 2, 129, "bf16", False),
    (1, 1, 300, "fp16", False),
    (1, 3, 1000, "bf16", True),
    (2, 3, 1000, "bf16", False),
    (1, 1, 384, "fp16", True),
    (2, 2, 520, "fp16", True),
    (1, 96, 700, "bf16", True),
    (2, 40, 513, "fp16", False),
    (2, 200, 128, "bf16", True),
    (1, 400, 100, "fp16", False),
]


@pytest.mark.parametrize("B,H,N,dtype,causal", SMALL)
def test_pair_small_every_element(oracle_mod, B, H, N, dtype, causal):
    w = I.custom("pair", B, H, N, 128, dtype, causal, seed_index=700 + N)
    q, k, v = I.qkv_bits(w)
    o, lse = run_pair(q, k, v, dtype, causal, w.scale)
    o_ref, l_ref = oracle_mod.attn_fwd(q, k, v, dtype, causal, w.scale)
    _check(compare(o, lse, o_ref, l_ref, dtype), f"B{B} H{H} N{N} {dtype} causal={causal}")


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_pair_sharpened_scores_rescale_path(oracle_mod, dtype):
    w = I.custom("sharp", 1, 2, 1024, 128, dtype, True, seed_index=7, q_mult=3.0)
    q, k, v = I.qkv_bits(w)
    o, lse = run_pair(q, k, v, dtype, True, w.scale)
    o_ref, l_ref = oracle_mod.attn_fwd(q, k, v, dtype, True, w.scale)
    res = explain_over(compare(o, lse, o_ref, l_ref, dtype), oracle_mod, q, k, v, dtype, True,
                       w.scale, 128)
    _check(res, f"sharp {dtype}")


@pytest.mark.parametrize("causal", [False, True])
def test_pair_q_zero_gives_mean_of_v(causal):
    rng = np.random.default_rng(55)
    N, d = 640, 128
    q = np.zeros((1, 2, N, d), dtype=np.uint16)
    k = I.to_bits(rng.standard_normal((1, 2, N, d)), "fp16")
    v = I.to_bits(rng.standard_normal((1, 2, N, d)), "fp16")
    o, lse = run_pair(q, k, v, "fp16", causal, 1.0 / np.sqrt(d))
    vd = bits_to_f64(v, "fp16")
    cnt = np.arange(1, N + 1, dtype=np.float64)[None, None, :, None]
    want = np.cumsum(vd, axis=2) / cnt if causal else np.broadcast_to(vd.mean(axis=2, keepdims=True), vd.shape)
    want_lse = np.log(cnt[..., 0]) if causal else np.full((1, 2, N), np.log(N))
    got = bits_to_f64(o, "fp16")
    assert np.all(np.abs(got - want) <= 2e-3 + half_ulp(want, "fp16"))
    np.testing.assert_allclose(lse, np.broadcast_to(want_lse, lse.shape), rtol=0, atol=1e-4)
    if causal:
        assert np.array_equal(o[:, :, 0, :], v[:, :, 0, :])


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_pair_causal_masked_keys_far_above_visible_ones(oracle_mod, dtype):
    """Keys 128.. score ~4096 * scale, keys 0..127 score 0: rows 0..127 (the
    even CTA's tile) meet a KV tile whose scores they may not see, far above
    everything they do see, in both softmax halves."""
    N, d = 384, 128
    rng = np.random.default_rng(N + d)
    q = np.zeros((1, 2, N, d))
    q[..., 0] = 64.0
    k = np.zeros((1, 2, N, d))
    k[..., 0] = np.where(np.arange(N) >= 128, 64.0, 0.0)[None, None, :]
    v = rng.standard_normal((1, 2, N, d))
    qb, kb, vb = (I.to_bits(x, dtype) for x in (q, k, v))
    scale = 1.0 / np.sqrt(d)
    o, lse = run_pair(qb, kb, vb, dtype, True, scale)
    o_ref, l_ref = oracle_mod.attn_fwd(qb, kb, vb, dtype, True, scale)
    _check(compare(o, lse, o_ref, l_ref, dtype), f"masked-high {dtype}")


@pytest.mark.parametrize("name", [n for n in I.WORKLOAD_ORDER if I.WORKLOADS[n].d == 128])
def test_pair_named_workload(oracle_named, name):
    w = I.WORKLOADS[name]
    q, k, v, o_ref, l_ref = oracle_named(name)
    o, lse = run_pair(q, k, v, w.dtype, w.causal, w.scale)
    res = compare(o, lse, o_ref, l_ref, w.dtype)
    if w.q_mult != 1.0:
        import oracle
        res = explain_over(res, oracle, q, k, v, w.dtype, w.causal, w.scale, w.d)
    _check(res, name)


@pytest.mark.parametrize("B,H,N,dtype,causal", [
    (2, 4, 1500, "bf16", True), (1, 3, 700, "fp16", False), (2, 200, 128, "bf16", True),
    (4, 16, 4096, "bf16", True), (4, 16, 4096, "fp16", False), (1, 32, 16384, "bf16", True),
])
def test_pair_bitwise_equal_to_one_cta_kernel(B, H, N, dtype, causal):
    import torch
    w = I.custom("pairbits", B, H, N, 128, dtype, causal, seed_index=88 + N)
    q, k, v = I.qkv_bits(w)
    o1, l1 = run_pair(q, k, v, w.dtype, causal, w.scale)
    o2, l2 = run_pair(q, k, v, w.dtype, causal, w.scale)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)          # deterministic
    # the one-CTA kernel (fa_fwd_noalloc always runs it; fa_fwd may pick the pair)
    qd, kd, vd = (to_device(x, w.dtype) for x in (q, k, v))
    o = torch.full_like(qd, float("nan"))
    lse = torch.full((B, H, N), float("nan"), dtype=torch.float32, device="cuda:0")
    code = fa.FA_DTYPE_BF16 if dtype == "bf16" else fa.FA_DTYPE_FP16
    assert fa.fa_fwd_noalloc(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(),
                             lse.data_ptr(), B, H, N, 128, causal, w.scale, code,
                             int(torch.cuda.current_stream().cuda_stream)) == fa.FA_OK
    torch.cuda.synchronize()
    assert fa.fa_check(0) == fa.FA_OK
    assert np.array_equal(to_bits(o), o1)
    assert np.array_equal(lse.cpu().numpy().view(np.uint32), l1.view(np.uint32))


def test_pair_side_stream_and_clock_record(oracle_mod):
    import torch
    w = I.custom("pairstream", 1, 3, 300, 128, "fp16", False, seed_index=31)
    q, k, v = I.qkv_bits(w)
    s = torch.cuda.Stream()
    fa.fa_sm_clock_read(0)
    o, lse = run_pair(q, k, v, "fp16", False, w.scale, stream=s)
    mhz, ctas = fa.fa_sm_clock_read(int(s.cuda_stream))
    assert ctas >= 2 and ctas % 2 == 0 and 300.0 < mhz < 2200.0
    o_ref, l_ref = oracle_mod.attn_fwd(q, k, v, "fp16", False, w.scale)
    _check(compare(o, lse, o_ref, l_ref, "fp16"), "side stream")
