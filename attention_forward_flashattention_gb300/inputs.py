"""Seeded synthetic inputs and the named attention workloads.

This module holds none of the attention arithmetic. It is the one piece the
CUDA path and the CPU oracle share: both consume the 16-bit values it emits.

Generator (counter based, so any slice can be produced independently):
  * SplitMix64 (Steele, Lea, Flood, "Fast splittable pseudorandom number
    generators", OOPSLA 2014): the n-th output of stream ``seed`` is
    mix64(seed * 2^32 + (n + 1) * 0x9E3779B97F4A7C15 mod 2^64), where mix64 is
    SplitMix64's finaliser (xor-shift 30 / multiply / xor-shift 27 / multiply /
    xor-shift 31).
  * Box-Muller (1958): two outputs u1, u2 -> 53-bit uniforms in [0, 1);
    z0 = sqrt(-2 ln(1 - u1)) cos(2 pi u2), z1 = sqrt(-2 ln(1 - u1)) sin(2 pi u2).
  * Rounding to storage: binary16 by numpy's float64 -> float16 cast
    (round-to-nearest-even); bfloat16 by float64 -> float32 (RNE) and then
    float32 -> bfloat16 (RNE on the bit pattern).

Streams: tensor t in {Q: 0, K: 1, V: 2} of a workload with seed index c uses
seed (1000 + c) * 4 + t.

8-bit (e4m3) inputs for the FP8 forward: the same normals, divided by a
float32 scale (the largest magnitude / 448: per tensor for Q and V, per
128-key block of each head for K) and rounded to the nearest e4m3 value (ties
to an even code, magnitudes above 448 saturating). V is stored transposed,
[B][H][d][ldv] with ldv = N rounded up to 16 and zero padding. Format: OCP
8-bit floating point, E4M3 "fn" variant (bias 7, 3 fraction bits, no
infinities, S.1111.111 = NaN, largest finite 448).
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


@dataclass(frozen=True)
class Workload:
    """One attention forward problem: Q, K, V are [B, H, N, d] in ``dtype``."""
    name: str
    B: int
    H: int
    N: int
    d: int
    dtype: str            # "fp16" or "bf16"
    causal: bool
    seed_index: int
    q_mult: float = 1.0   # Q = round(q_mult * z), z ~ N(0, 1)

    @property
    def scale(self) -> float:
        return float(np.float32(1.0 / np.sqrt(self.d)))

    @property
    def flops(self) -> float:
        """Metric FLOPs: 4 B H N^2 d, halved when causal."""
        f = 4.0 * self.B * self.H * self.N * self.N * self.d
        return f / 2.0 if self.causal else f

    @property
    def seed(self) -> int:
        return 1000 + self.seed_index


# The five workloads the library is measured and checked on.
WORKLOADS = {
    w.name: w for w in [
        Workload("mha_b1_h2_n256_d64_fp16", 1, 2, 256, 64, "fp16", False, 1),
        Workload("mha_b4_h16_n4096_d128_fp16", 4, 16, 4096, 128, "fp16", False, 2),
        Workload("causal_b4_h16_n4096_d128_bf16", 4, 16, 4096, 128, "bf16", True, 3),
        Workload("mha_b2_h32_n8192_d64_fp16", 2, 32, 8192, 64, "fp16", False, 4),
        Workload("causal_b1_h32_n16384_d128_bf16_q3", 1, 32, 16384, 128, "bf16", True, 5, 3.0),
    ]
}
WORKLOAD_ORDER = list(WORKLOADS)


def _mix64(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def splitmix64(seed: int, start: int, count: int) -> np.ndarray:
    """Outputs start .. start+count-1 of SplitMix64 stream ``seed``."""
    n = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        state = np.uint64((seed << 32) & 0xFFFFFFFFFFFFFFFF) + n * _GOLDEN
        return _mix64(state)


def normal(seed: int, count: int, start: int = 0) -> np.ndarray:
    """Standard normals ``start .. start+count-1`` of stream ``seed`` (float64).

    Normal 2p and 2p+1 come from SplitMix64 outputs 2p and 2p+1.
    """
    p0 = start // 2
    p1 = (start + count + 1) // 2
    bits = splitmix64(seed, 2 * p0, 2 * (p1 - p0)).reshape(-1, 2)
    u1 = (bits[:, 0] >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)
    u2 = (bits[:, 1] >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)
    r = np.sqrt(-2.0 * np.log1p(-u1))
    t = 2.0 * np.pi * u2
    z = np.empty(2 * (p1 - p0), dtype=np.float64)
    z[0::2] = r * np.cos(t)
    z[1::2] = r * np.sin(t)
    off = start - 2 * p0
    return z[off:off + count]


def to_fp16_bits(x: np.ndarray) -> np.ndarray:
    """float64 -> binary16 bit patterns (round to nearest even)."""
    with np.errstate(over="ignore"):
        return np.asarray(x, dtype=np.float64).astype(np.float16).view(np.uint16)


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float64 -> float32 (RNE) -> bfloat16 bit patterns (RNE)."""
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float64).astype(np.float32)).view(np.uint32)
    bias = np.uint32(0x7FFF) + ((f >> np.uint32(16)) & np.uint32(1))
    return ((f + bias) >> np.uint32(16)).astype(np.uint16)


def to_bits(x: np.ndarray, dtype: str) -> np.ndarray:
    return to_fp16_bits(x) if dtype == "fp16" else to_bf16_bits(x)


def tensor_bits(w: Workload, which: int, chunk: int = 1 << 22) -> np.ndarray:
    """Stored 16-bit values of Q (0), K (1), V (2) or the output gradient dO
    (3) of workload ``w``: [B, H, N, d]."""
    n = w.B * w.H * w.N * w.d
    out = np.empty(n, dtype=np.uint16)
    seed = w.seed * 4 + which
    mult = w.q_mult if which == 0 else 1.0
    for s in range(0, n, chunk):
        c = min(chunk, n - s)
        z = normal(seed, c, s)
        if mult != 1.0:
            z = z * mult
        out[s:s + c] = to_bits(z, w.dtype)
    return out.reshape(w.B, w.H, w.N, w.d)


def qkv_bits(w: Workload):
    """(Q, K, V) stored 16-bit values of workload ``w``."""
    return tensor_bits(w, 0), tensor_bits(w, 1), tensor_bits(w, 2)


def dout_bits(w: Workload) -> np.ndarray:
    """Stored 16-bit values of a seeded output gradient dO for the backward."""
    return tensor_bits(w, 3)


def custom(name: str, B: int, H: int, N: int, d: int, dtype: str, causal: bool,
           seed_index: int, q_mult: float = 1.0) -> Workload:
    """A workload outside the five named ones (edge cases in tests)."""
    return Workload(name, B, H, N, d, dtype, causal, seed_index, q_mult)


# ------------------------------------------------------------ 8-bit (e4m3) inputs

E4M3_MAX = 448.0


def e4m3_values() -> np.ndarray:
    """Value of each of the 256 e4m3 codes (float64; NaN for S.1111.111)."""
    c = np.arange(256)
    e, m = (c >> 3) & 0xF, c & 7
    v = np.where(e == 0, m * 2.0 ** -9, (8 + m) * np.exp2(e - 10.0))
    v = np.where(c & 0x80, -v, v)
    v[(e == 15) & (m == 7)] = np.nan
    return v


def to_e4m3_bits(x: np.ndarray) -> np.ndarray:
    """float64 -> e4m3 codes: nearest value, ties to the even code, |x| > 448 -> 448;
    the sign bit follows x (a negative value that rounds to zero gives -0)."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), E4M3_MAX)
    # spacing of e4m3 values around a: 2^(e - 3) in the binade [2^e, 2^(e+1)),
    # 2^-9 below 2^-6 (subnormals); numpy's round is round-half-to-even, and
    # a / spacing is exact, so r is the correctly rounded value
    _, ex = np.frexp(a)                       # a = f 2^ex, f in [0.5, 1)
    e = np.maximum(ex - 1, -6)
    r = np.minimum(np.round(np.ldexp(a, 3 - e)), 16.0)   # 8..16 (normal) or 0..8 (subnormal)
    # r == 16 carried into the next binade; below 2^-6 r counts 2^-9 steps
    e = np.where(r == 16.0, e + 1, e)
    r = np.where(r == 16.0, 8.0, r)
    normal = r >= 8.0
    code = np.where(normal, ((e + 7) << 3) + (r.astype(np.int64) - 8), r.astype(np.int64))
    code = np.minimum(code, 0x7E).astype(np.uint8)
    return np.where(np.signbit(x), code | np.uint8(0x80), code).astype(np.uint8)


@dataclass(frozen=True)
class Fp8Inputs:
    """e4m3 codes and scales of one workload (values = scale * code value)."""
    q: np.ndarray         # uint8 [B, H, N, d]
    k: np.ndarray         # uint8 [B, H, N, d]
    vt: np.ndarray        # uint8 [B, H, d, ldv], V transposed, zero padded
    q_scale: float        # float32 value
    k_scales: np.ndarray  # float32 [B, H, ceil(N / 128)]
    v_scale: float        # float32 value

    @property
    def ldv(self) -> int:
        return int(self.vt.shape[-1])


def _scale_for(amax: float) -> float:
    return float(np.float32(amax / E4M3_MAX)) if amax > 0 else 1.0


def fp8_inputs(w: Workload) -> Fp8Inputs:
    """e4m3 inputs of ``w`` from the same normals as its 16-bit inputs."""
    B, H, N, d = w.B, w.H, w.N, w.d
    n = B * H * N * d
    zq = normal(w.seed * 4 + 0, n).reshape(B, H, N, d) * w.q_mult
    zk = normal(w.seed * 4 + 1, n).reshape(B, H, N, d)
    zv = normal(w.seed * 4 + 2, n).reshape(B, H, N, d)
    q_scale = _scale_for(float(np.abs(zq).max()))
    v_scale = _scale_for(float(np.abs(zv).max()))
    q8 = to_e4m3_bits(zq / q_scale)
    nt = (N + 127) // 128
    k_scales = np.empty((B, H, nt), dtype=np.float32)
    k8 = np.empty((B, H, N, d), dtype=np.uint8)
    for t in range(nt):
        blk = zk[:, :, 128 * t:128 * (t + 1), :]
        sc = np.array([[_scale_for(float(np.abs(blk[b, h]).max())) for h in range(H)]
                       for b in range(B)], dtype=np.float32)
        k_scales[:, :, t] = sc
        k8[:, :, 128 * t:128 * (t + 1), :] = to_e4m3_bits(blk / sc[:, :, None, None].astype(np.float64))
    ldv = (N + 15) // 16 * 16
    vt = np.zeros((B, H, d, ldv), dtype=np.uint8)
    vt[:, :, :, :N] = to_e4m3_bits(zv / v_scale).transpose(0, 1, 3, 2)
    return Fp8Inputs(q8, k8, vt, q_scale, k_scales, v_scale)


# 8-bit workloads (e4m3 Q, K, V; bf16 O): the shape of the headline 16-bit one.
FP8_WORKLOADS = {
    w.name: w for w in [
        Workload("mha_b4_h16_n4096_d128_e4m3", 4, 16, 4096, 128, "e4m3", False, 2),
        Workload("causal_b4_h16_n4096_d128_e4m3", 4, 16, 4096, 128, "e4m3", True, 3),
    ]
}
