"""Pins for the fp64 oracle: closed forms, invariances and library routines.

None of these re-types the oracle's formula. Each check comes from a fact the
mathematics fixes independently of the oracle's code:
  * exhaustive decode of every 16-bit pattern against numpy / the IEEE layout;
  * Q = 0 makes every score 0, so O is the (prefix) mean of V and
    LSE = ln(#keys) (closed form);
  * one-hot scores select a single V row with a computable residual weight;
  * V = const gives O = const (rows of P sum to 1);
  * O is linear in V; non-causal O is invariant under a joint permutation of
    K and V rows; adding a constant vector u to every key shifts each score
    of row i by scale * q_i . u, so O is unchanged and LSE shifts by it;
  * agreement with an explicit-softmax formulation built from numpy's matmul
    and scipy.special.softmax / logsumexp on small problems.
A mistake such as a dropped max-subtraction, a wrong mask index, a transposed
operand, a missing scale or a wrong log base fails at least one of them.
"""
import numpy as np
import pytest
import scipy.special as sps

from attention_forward_flashattention_gb300 import inputs as I


def _rand_bits(rng, shape, dtype, mult=1.0):
    return I.to_bits(rng.standard_normal(shape) * mult, dtype)


# ---------------------------------------------------------------- decoding

def test_decode_fp16_exhaustive(oracle_mod):
    bits = np.arange(65536, dtype=np.uint16)
    got = oracle_mod.decode(bits, "fp16")
    want = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])


def test_decode_bf16_exhaustive(oracle_mod):
    bits = np.arange(65536, dtype=np.uint16)
    got = oracle_mod.decode(bits, "bf16")
    with np.errstate(invalid="ignore"):
        want = (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])


# ---------------------------------------------------------------- closed forms

@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("N,d", [(1, 64), (37, 64), (128, 128)])
def test_q_zero_gives_column_mean(oracle_mod, dtype, N, d):
    rng = np.random.default_rng(11)
    q = np.zeros((1, 2, N, d), dtype=np.uint16)          # +0.0 in both formats
    k = _rand_bits(rng, (1, 2, N, d), dtype)
    v = _rand_bits(rng, (1, 2, N, d), dtype)
    o, lse = oracle_mod.attn_fwd(q, k, v, dtype, False, 0.125)
    vd = oracle_mod.decode(v, dtype)
    mean = vd.mean(axis=2, keepdims=True)
    np.testing.assert_allclose(o, np.broadcast_to(mean, o.shape), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, np.full(lse.shape, np.log(N)), rtol=0, atol=1e-12)


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_q_zero_causal_gives_prefix_mean(oracle_mod, dtype):
    rng = np.random.default_rng(12)
    N, d = 200, 64
    q = np.zeros((2, 1, N, d), dtype=np.uint16)
    k = _rand_bits(rng, (2, 1, N, d), dtype)
    v = _rand_bits(rng, (2, 1, N, d), dtype)
    o, lse = oracle_mod.attn_fwd(q, k, v, dtype, True, 0.3)
    vd = oracle_mod.decode(v, dtype)
    counts = np.arange(1, N + 1, dtype=np.float64)[None, None, :, None]
    prefix = np.cumsum(vd, axis=2) / counts
    np.testing.assert_allclose(o, prefix, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, np.broadcast_to(np.log(counts[..., 0]), lse.shape), rtol=0, atol=1e-12)
    # row 0 sees key 0 only: O_0 = v_0 exactly
    assert np.array_equal(o[:, :, 0, :], vd[:, :, 0, :])


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_one_hot_scores_select_one_row(oracle_mod, dtype):
    # k_j = e_j, q_i = 16 e_{pi(i)}, scale 1: s_ij = 16 [j == pi(i)].
    N, d = 48, 64
    rng = np.random.default_rng(13)
    perm = rng.permutation(N)
    qf = np.zeros((1, 1, N, d))
    qf[0, 0, np.arange(N), perm] = 16.0
    kf = np.zeros((1, 1, N, d))
    kf[0, 0, np.arange(N), np.arange(N)] = 1.0
    v = _rand_bits(rng, (1, 1, N, d), dtype)
    o, lse = oracle_mod.attn_fwd(I.to_bits(qf, dtype), I.to_bits(kf, dtype), v, dtype, False, 1.0)
    vd = oracle_mod.decode(v, dtype)[0, 0]
    e16 = np.exp(16.0)
    want = (e16 * vd[perm] + (vd.sum(axis=0)[None, :] - vd[perm])) / (e16 + N - 1)
    np.testing.assert_allclose(o[0, 0], want, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse[0, 0], np.full(N, np.log(e16 + N - 1)), rtol=0, atol=1e-12)
    # and the selected row dominates: |O_i - v_pi(i)| <= (N-1) e^-16 max|v| * 2
    assert np.max(np.abs(o[0, 0] - vd[perm])) <= 2 * (N - 1) * np.exp(-16.0) * np.max(np.abs(vd)) + 1e-15


@pytest.mark.parametrize("causal", [False, True])
def test_constant_v_rows_sum_to_one(oracle_mod, causal):
    rng = np.random.default_rng(14)
    N, d = 96, 64
    q = _rand_bits(rng, (1, 2, N, d), "fp16", 2.0)
    k = _rand_bits(rng, (1, 2, N, d), "fp16")
    cols = rng.standard_normal(d)
    v = I.to_bits(np.broadcast_to(cols, (1, 2, N, d)), "fp16")
    o, _ = oracle_mod.attn_fwd(q, k, v, "fp16", causal, 0.125)
    c = oracle_mod.decode(v, "fp16")[0, 0, 0]
    np.testing.assert_allclose(o, np.broadcast_to(c, o.shape), rtol=0, atol=1e-13)


# ---------------------------------------------------------------- invariances

def test_linear_in_v(oracle_mod):
    rng = np.random.default_rng(15)
    N, d = 80, 128
    q = _rand_bits(rng, (1, 1, N, d), "fp16")
    k = _rand_bits(rng, (1, 1, N, d), "fp16")
    vf = oracle_mod.decode(_rand_bits(rng, (1, 1, N, d), "fp16"), "fp16")
    o1, l1 = oracle_mod.attn_fwd(q, k, I.to_bits(vf, "fp16"), "fp16", True, 0.09)
    o2, l2 = oracle_mod.attn_fwd(q, k, I.to_bits(4.0 * vf, "fp16"), "fp16", True, 0.09)
    np.testing.assert_allclose(o2, 4.0 * o1, rtol=1e-14, atol=1e-14)
    assert np.array_equal(l1, l2)


def test_joint_permutation_of_keys(oracle_mod):
    rng = np.random.default_rng(16)
    N, d = 70, 64
    q = _rand_bits(rng, (1, 1, N, d), "bf16")
    k = _rand_bits(rng, (1, 1, N, d), "bf16")
    v = _rand_bits(rng, (1, 1, N, d), "bf16")
    perm = rng.permutation(N)
    o1, l1 = oracle_mod.attn_fwd(q, k, v, "bf16", False, 0.125)
    o2, l2 = oracle_mod.attn_fwd(q, k[:, :, perm], v[:, :, perm], "bf16", False, 0.125)
    np.testing.assert_allclose(o2, o1, rtol=0, atol=1e-13)
    np.testing.assert_allclose(l2, l1, rtol=0, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_key_shift_moves_lse_only(oracle_mod, causal):
    # Small integers keep K + u exact in fp16; then s'_ij = s_ij + scale q_i.u.
    rng = np.random.default_rng(17)
    N, d = 64, 64
    qf = rng.integers(-3, 4, size=(1, 1, N, d)).astype(np.float64) * 0.25
    kf = rng.integers(-3, 4, size=(1, 1, N, d)).astype(np.float64)
    u = rng.integers(-2, 3, size=d).astype(np.float64)
    vf = rng.standard_normal((1, 1, N, d))
    scale = 0.125
    q, k, k2, v = (I.to_bits(x, "fp16") for x in (qf, kf, kf + u, vf))
    o1, l1 = oracle_mod.attn_fwd(q, k, v, "fp16", causal, scale)
    o2, l2 = oracle_mod.attn_fwd(q, k2, v, "fp16", causal, scale)
    np.testing.assert_allclose(o2, o1, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l2, l1 + scale * (qf[0, 0] @ u)[None, None, :], rtol=0, atol=1e-12)


# ---------------------------------------------------------------- library formulation

def _explicit(qd, kd, vd, causal, scale):
    """Materialised scores -> scipy softmax -> P @ V, and scipy logsumexp."""
    s = scale * np.matmul(qd, np.swapaxes(kd, -1, -2))
    if causal:
        n = s.shape[-1]
        s = np.where(np.tril(np.ones((n, n), dtype=bool)), s, -np.inf)
    p = sps.softmax(s, axis=-1)
    return np.matmul(p, vd), sps.logsumexp(s, axis=-1)


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,N,d", [(1, 1, 1, 64), (1, 2, 7, 64), (2, 1, 33, 128), (1, 2, 64, 128)])
def test_matches_explicit_softmax(oracle_mod, dtype, causal, B, H, N, d):
    rng = np.random.default_rng(N * 131 + d)
    q = _rand_bits(rng, (B, H, N, d), dtype, 3.0)
    k = _rand_bits(rng, (B, H, N, d), dtype)
    v = _rand_bits(rng, (B, H, N, d), dtype)
    scale = float(np.float32(1.0 / np.sqrt(d)))
    o, lse = oracle_mod.attn_fwd(q, k, v, dtype, causal, scale)
    want_o, want_lse = _explicit(*(oracle_mod.decode(x, dtype) for x in (q, k, v)), causal, scale)
    np.testing.assert_allclose(o, want_o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, want_lse, rtol=0, atol=1e-12)


def test_scale_is_taken_as_float32(oracle_mod):
    rng = np.random.default_rng(18)
    q = _rand_bits(rng, (1, 1, 16, 64), "fp16", 4.0)
    k = _rand_bits(rng, (1, 1, 16, 64), "fp16")
    v = _rand_bits(rng, (1, 1, 16, 64), "fp16")
    _, lse = oracle_mod.attn_fwd(q, k, v, "fp16", False, 0.1)
    qd, kd, vd = (oracle_mod.decode(x, "fp16") for x in (q, k, v))
    _, l32 = _explicit(qd, kd, vd, False, float(np.float32(0.1)))
    np.testing.assert_allclose(lse, l32, rtol=0, atol=1e-12)


# ---------------------------------------------------------------- row sampler

@pytest.mark.parametrize("causal", [False, True])
def test_rows_equal_full(oracle_mod, causal):
    rng = np.random.default_rng(19)
    B, H, N, d = 2, 3, 96, 64
    q = _rand_bits(rng, (B, H, N, d), "bf16")
    k = _rand_bits(rng, (B, H, N, d), "bf16")
    v = _rand_bits(rng, (B, H, N, d), "bf16")
    o, lse = oracle_mod.attn_fwd(q, k, v, "bf16", causal, 0.125, nthreads=3)
    rows = np.sort(rng.choice(B * H * N, size=50, replace=False))
    ro, rl = oracle_mod.attn_rows(q, k, v, "bf16", causal, 0.125, rows, nthreads=4)
    assert np.array_equal(ro, o.reshape(-1, d)[rows])
    assert np.array_equal(rl, lse.reshape(-1)[rows])


def test_rejects_bad_arguments(oracle_mod):
    q = np.zeros((1, 1, 4, 64), dtype=np.uint16)
    with pytest.raises(ValueError):
        oracle_mod.attn_rows(q, q, q, "fp16", False, 1.0, np.array([4]))


# ---------------------------------------------------------------- 8-bit (e4m3) oracle

def test_decode_e4m3_exhaustive_against_torch(oracle_mod):
    torch = pytest.importorskip("torch")
    codes = np.arange(256, dtype=np.uint8)
    got = oracle_mod.decode_e4m3(codes)
    want = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan) and nan.sum() == 2   # S.1111.111 only
    assert np.array_equal(got[~nan], want[~nan])


def test_decode_e4m3_format_constants(oracle_mod):
    # OCP FP8 E4M3: 1.0 = 0x38, largest 448 = 0x7E, smallest normal 2^-6 = 0x08,
    # smallest subnormal 2^-9 = 0x01, sign in bit 7
    got = oracle_mod.decode_e4m3(np.array([0x38, 0x7E, 0x08, 0x01, 0xB8, 0x00, 0x80], np.uint8))
    assert list(got) == [1.0, 448.0, 2.0 ** -6, 2.0 ** -9, -1.0, 0.0, -0.0]


def _fp8_problem(seed, B, H, N, d=128, q_mult=1.0):
    w = I.custom("fp8pin", B, H, N, d, "e4m3", False, seed, q_mult)
    return w, I.fp8_inputs(w)


def _decoded(oracle_mod, f):
    B, H, N, d = f.q.shape
    q = oracle_mod.decode_e4m3(f.q) * np.float64(f.q_scale)
    ks = np.repeat(f.k_scales.astype(np.float64), 128, axis=2)[:, :, :N, None]
    k = oracle_mod.decode_e4m3(f.k) * ks
    v = oracle_mod.decode_e4m3(f.vt[..., :N]).transpose(0, 1, 3, 2) * np.float64(f.v_scale)
    return q, k, v


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_oracle_matches_explicit_softmax(oracle_mod, causal):
    w, f = _fp8_problem(11, 1, 2, 300)
    o, lse, _ = oracle_mod.attn_fp8(f.q, f.k, f.vt, f.q_scale, f.k_scales, f.v_scale, causal,
                                    w.scale)
    q, k, v = _decoded(oracle_mod, f)
    s = np.einsum("bhid,bhjd->bhij", q, k) * np.float64(np.float32(w.scale))
    if causal:
        s = np.where(np.tril(np.ones((w.N, w.N), bool)), s, -np.inf)
    p = sps.softmax(s, axis=-1)
    want_o = np.einsum("bhij,bhjd->bhid", p, v).reshape(-1, w.d)
    want_l = sps.logsumexp(s, axis=-1).reshape(-1)
    np.testing.assert_allclose(o, want_o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, want_l, rtol=0, atol=1e-12)


def test_fp8_oracle_rows_equal_full(oracle_mod):
    w, f = _fp8_problem(12, 2, 1, 200)
    o, lse, b = oracle_mod.attn_fp8(f.q, f.k, f.vt, f.q_scale, f.k_scales, f.v_scale, True,
                                    w.scale)
    rows = np.array([0, 5, 199, 200, 333, 399])
    o2, l2, b2 = oracle_mod.attn_fp8(f.q, f.k, f.vt, f.q_scale, f.k_scales, f.v_scale, True,
                                     w.scale, rows=rows)
    assert np.array_equal(o[rows], o2) and np.array_equal(lse[rows], l2)
    assert np.array_equal(b[rows], b2)


@pytest.mark.parametrize("shift", [0.0, 2.5, 8.0])
@pytest.mark.parametrize("q_mult", [1.0, 3.0])
def test_fp8_bound_covers_rounded_weights(oracle_mod, shift, q_mult):
    # Simulate what the bound is about: weights on a scale whose largest value
    # is 2^shift (shift in [0, 8]), each rounded to the nearest e4m3 value,
    # O normalised by the unrounded sum. The bound must hold for every element
    # and be far from vacuous.
    w, f = _fp8_problem(13, 1, 2, 256, q_mult=q_mult)
    o, lse, bound = oracle_mod.attn_fp8(f.q, f.k, f.vt, f.q_scale, f.k_scales, f.v_scale,
                                        False, w.scale)
    q, k, v = _decoded(oracle_mod, f)
    s = np.einsum("bhid,bhjd->bhij", q, k) * np.float64(np.float32(w.scale))
    p = np.exp(s - s.max(axis=-1, keepdims=True)) * 2.0 ** shift
    p_rounded = oracle_mod.decode_e4m3(I.to_e4m3_bits(p))
    o_q = np.einsum("bhij,bhjd->bhid", p_rounded, v) / p.sum(axis=-1)[..., None]
    err = np.abs(o_q.reshape(-1, w.d) - o)
    assert np.all(err <= bound + 1e-12)
    assert float(bound.max()) < 0.5 and float(err.max()) > 0.0


# ---------------------------------------------------------------- weighted deviation of V

def test_dev_uniform_weights_is_mean_absolute_deviation(oracle_mod):
    """Q = 0: every weight is 1/N, so dev_t = mean_j |v_jt - mean(v_t)|."""
    rng = np.random.default_rng(21)
    N, d = 57, 64
    q = np.zeros((1, 2, N, d), dtype=np.uint16)
    k = _rand_bits(rng, (1, 2, N, d), "bf16")
    v = _rand_bits(rng, (1, 2, N, d), "bf16")
    rows = np.array([0, 5, N - 1, N + 3, 2 * N - 1])
    o, lse, dev = oracle_mod.attn_rows_dev(q, k, v, "bf16", False, 0.125, rows)
    vd = oracle_mod.decode(v, "bf16").reshape(2, N, d)
    for r, row in enumerate(rows):
        vh = vd[row // N]
        want = np.abs(vh - vh.mean(axis=0)).mean(axis=0)
        np.testing.assert_allclose(dev[r], want, rtol=0, atol=1e-13)


def test_dev_two_keys_closed_form(oracle_mod):
    """Two keys with scores a, b: O = p1 v1 + p2 v2 and dev = 2 p1 p2 |v1 - v2|
    (|v1 - O| = p2 |v1 - v2|, |v2 - O| = p1 |v1 - v2|)."""
    N, d = 2, 64
    qf = np.zeros((1, 1, N, d))
    qf[..., 0] = 1.0
    kf = np.zeros((1, 1, N, d))
    kf[0, 0, :, 0] = [1.5, -0.25]                     # scores 1.5 and -0.25 (scale 1)
    rng = np.random.default_rng(22)
    v = _rand_bits(rng, (1, 1, N, d), "fp16")
    o, lse, dev = oracle_mod.attn_rows_dev(I.to_bits(qf, "fp16"), I.to_bits(kf, "fp16"), v, "fp16",
                                           False, 1.0, np.array([0, 1]))
    vd = oracle_mod.decode(v, "fp16")[0, 0]
    p1 = 1.0 / (1.0 + np.exp(-1.75))
    p2 = 1.0 - p1
    want = 2 * p1 * p2 * np.abs(vd[0] - vd[1])
    for r in range(2):
        np.testing.assert_allclose(o[r], p1 * vd[0] + p2 * vd[1], rtol=0, atol=1e-13)
        np.testing.assert_allclose(dev[r], want, rtol=0, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_dev_zero_for_constant_v_and_single_key(oracle_mod, causal):
    rng = np.random.default_rng(23)
    N, d = 70, 128
    q = _rand_bits(rng, (1, 1, N, d), "bf16", 2.0)
    k = _rand_bits(rng, (1, 1, N, d), "bf16")
    cols = rng.standard_normal(d)
    vc = I.to_bits(np.broadcast_to(cols, (1, 1, N, d)), "bf16")
    rows = np.arange(N)
    _, _, dev = oracle_mod.attn_rows_dev(q, k, vc, "bf16", causal, 0.1, rows)
    assert np.max(np.abs(dev)) <= 1e-13
    v = _rand_bits(rng, (1, 1, N, d), "bf16")
    o, lse, dev = oracle_mod.attn_rows_dev(q, k, v, "bf16", causal, 0.1, rows)
    o2, l2 = oracle_mod.attn_rows(q, k, v, "bf16", causal, 0.1, rows)
    assert np.array_equal(o, o2) and np.array_equal(lse, l2)
    if causal:   # row 0 sees key 0 alone: no deviation
        assert np.all(dev[0] == 0.0)


def test_dev_bounds_rounded_weights(oracle_mod):
    """The bound it exists for: O recomputed from bf16-rounded weights (and
    their sum) lies within u / (1 - u) dev of O, u = 2^-8 (bf16's unit
    roundoff: 8 significant bits), on random rows."""
    rng = np.random.default_rng(24)
    N, d = 300, 64
    q = _rand_bits(rng, (1, 1, N, d), "bf16", 3.0)
    k = _rand_bits(rng, (1, 1, N, d), "bf16")
    v = _rand_bits(rng, (1, 1, N, d), "bf16")
    rows = np.arange(N)
    o, _, dev = oracle_mod.attn_rows_dev(q, k, v, "bf16", True, 0.125, rows)
    qd, kd, vd = (oracle_mod.decode(x, "bf16")[0, 0] for x in (q, k, v))
    u = 2.0 ** -8
    for i in rows:
        s = np.float64(np.float32(0.125)) * (kd[:i + 1] @ qd[i])
        p = np.exp(s - s.max())
        m, e = np.frexp(p)
        r = np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)   # bf16 rounding of the weights
        o_r = (r @ vd[:i + 1]) / r.sum()
        assert np.all(np.abs(o_r - o[i]) <= u / (1 - u) * dev[i] + 1e-13)
