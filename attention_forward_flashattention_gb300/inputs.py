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
    """Stored 16-bit values of Q (0), K (1) or V (2) of workload ``w``: [B, H, N, d]."""
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


def custom(name: str, B: int, H: int, N: int, d: int, dtype: str, causal: bool,
           seed_index: int, q_mult: float = 1.0) -> Workload:
    """A workload outside the five named ones (edge cases in tests)."""
    return Workload(name, B, H, N, d, dtype, causal, seed_index, q_mult)
