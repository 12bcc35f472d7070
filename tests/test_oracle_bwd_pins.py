"""Pins for the fp64 backward oracle (oracle.attn_bwd).

Each check comes from a fact independent of the oracle's code:
  * central finite differences of the loss L = sum(dO * O), with O computed by
    an explicit-softmax forward built from numpy / scipy routines;
  * Q = 0 (uniform softmax) gives closed forms: dV_j = mean_i dO_i,
    dK = 0, dQ_i = scale / N * sum_j (dO_i . v_j) (k_j - mean k);
  * translation invariance of the softmax in the keys: sum_j dK_j = 0;
  * the magnitude sums bound the gradients.
A mistake such as a missing D_i term, a transposed dS, a wrong scale or a
causal mask applied on the wrong side fails at least one of them.
"""
import numpy as np
import pytest
import scipy.special as sps

from attention_forward_flashattention_gb300 import inputs as I


def _problem(seed, B, H, N, d, dtype="fp16"):
    rng = np.random.default_rng(seed)
    return tuple(I.to_bits(rng.standard_normal((B, H, N, d)), dtype) for _ in range(4))


def _forward_np(q, k, v, scale, causal):
    s = np.einsum("bhid,bhjd->bhij", q, k) * scale
    if causal:
        n = s.shape[-1]
        s = np.where(np.tril(np.ones((n, n), bool)), s, -np.inf)
    return np.einsum("bhij,bhjd->bhid", sps.softmax(s, axis=-1), v)


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_matches_finite_differences(oracle_mod, causal):
    B, H, N, d = 1, 2, 6, 4
    bits = _problem(5 + causal, B, H, N, d)
    q, k, v, do = (oracle_mod.decode(x, "fp16") for x in bits)
    scale = float(np.float32(0.7))
    g = oracle_mod.attn_bwd(*bits, "fp16", causal, scale)
    h = 1e-5

    def loss(qq, kk, vv):
        return float(np.sum(do * _forward_np(qq, kk, vv, scale, causal)))

    for name, idx in (("dq", 0), ("dk", 1), ("dv", 2)):
        fd = np.zeros((B, H, N, d))
        base = [q, k, v]
        for pos in np.ndindex(B, H, N, d):
            plus = [x.copy() for x in base]
            minus = [x.copy() for x in base]
            plus[idx][pos] += h
            minus[idx][pos] -= h
            fd[pos] = (loss(*plus) - loss(*minus)) / (2 * h)
        np.testing.assert_allclose(g[name].reshape(B, H, N, d), fd, rtol=0, atol=1e-7,
                                   err_msg=name)


def test_bwd_q_zero_closed_forms(oracle_mod):
    B, H, N, d = 1, 1, 40, 16
    _, kb, vb, dob = _problem(9, B, H, N, d)
    qb = np.zeros_like(kb)
    scale = float(np.float32(0.25))
    g = oracle_mod.attn_bwd(qb, kb, vb, dob, "fp16", False, scale)
    k, v, do = (oracle_mod.decode(x, "fp16")[0, 0] for x in (kb, vb, dob))
    np.testing.assert_allclose(g["dv"][0], np.broadcast_to(do.mean(axis=0), (N, d)), atol=1e-13)
    assert np.all(g["dk"][0] == 0.0)
    want_dq = scale / N * (do @ v.T) @ (k - k.mean(axis=0))
    np.testing.assert_allclose(g["dq"][0], want_dq, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_key_gradients_sum_to_zero(oracle_mod, causal):
    bits = _problem(13, 2, 2, 50, 8, "bf16")
    g = oracle_mod.attn_bwd(*bits, "bf16", causal, float(np.float32(0.35)))
    np.testing.assert_allclose(g["dk"].sum(axis=1), 0.0, atol=1e-11)


def test_bwd_magnitudes_bound_gradients_and_heads_select(oracle_mod):
    bits = _problem(17, 2, 3, 33, 8)
    scale = float(np.float32(0.3))
    full = oracle_mod.attn_bwd(*bits, "fp16", True, scale)
    for n in ("dq", "dk", "dv"):
        assert np.all(np.abs(full[n]) <= full["mag_" + n] + 1e-15)
    part = oracle_mod.attn_bwd(*bits, "fp16", True, scale, heads=[4, 1])
    for n in full:
        assert np.array_equal(part[n], full[n][[4, 1]])
