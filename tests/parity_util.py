"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI,
decode its outputs, and compare them with the fp64 oracle.

Tolerances (the stated bounds of the library's specification):
  * O: mean |O_gpu - O_ref| <= 1e-3, and every element
    |O_gpu - O_ref| <= 1e-2 + half_ulp_X(O_ref). The second term is the
    rounding of the exact result to the 16-bit output format X, which no
    X-output kernel can avoid (for bf16 it reaches 0.0156 at |O| >= 4).
    The plain max |O_gpu - O_ref| is reported alongside.
  * LSE: max |LSE_gpu - LSE_ref| <= 1e-3.
"""
from __future__ import annotations

import numpy as np

O_MAX_ABS = 1e-2
O_MEAN_ABS = 1e-3
LSE_MAX_ABS = 1e-3

_PRECISION = {"fp16": 11, "bf16": 8}  # significant bits


def bits_to_f64(bits: np.ndarray, dtype: str) -> np.ndarray:
    bits = np.asarray(bits, dtype=np.uint16)
    if dtype == "fp16":
        return bits.view(np.float16).astype(np.float64)
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def half_ulp(x: np.ndarray, dtype: str) -> np.ndarray:
    """Half the spacing of format `dtype` at |x| (normal range; subnormal floor)."""
    p = _PRECISION[dtype]
    min_exp = -14 if dtype == "fp16" else -126
    _, e = np.frexp(np.abs(x))            # |x| = m 2^e, m in [0.5, 1)
    e = np.where(x == 0, min_exp, np.maximum(e - 1, min_exp))  # floor(log2 |x|), clamped
    return np.ldexp(1.0, (e - (p - 1) - 1).astype(np.int64))


def compare(o_bits: np.ndarray, lse: np.ndarray, o_ref: np.ndarray, lse_ref: np.ndarray,
            dtype: str) -> dict:
    o = bits_to_f64(o_bits, dtype)
    err = np.abs(o - o_ref)
    lerr = np.abs(np.asarray(lse, dtype=np.float64) - lse_ref)
    excess = err - half_ulp(o_ref, dtype)
    res = {
        "o_max_abs": float(err.max()) if err.size else 0.0,
        "o_mean_abs": float(err.mean()) if err.size else 0.0,
        "o_max_excess_over_rounding": float(excess.max()) if err.size else 0.0,
        "lse_max_abs": float(lerr.max()) if lerr.size else 0.0,
        "finite": bool(np.all(np.isfinite(o)) and np.all(np.isfinite(lse))),
    }
    res["ok"] = (res["finite"] and res["o_mean_abs"] <= O_MEAN_ABS
                 and res["o_max_excess_over_rounding"] <= O_MAX_ABS
                 and res["lse_max_abs"] <= LSE_MAX_ABS)
    return res


def torch_dtype(dtype: str):
    import torch
    return torch.float16 if dtype == "fp16" else torch.bfloat16


def to_device(bits: np.ndarray, dtype: str, device="cuda:0"):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(torch_dtype(dtype)).to(device)


def to_bits(t) -> np.ndarray:
    import torch
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)


def run_fa(q_bits, k_bits, v_bits, dtype: str, causal: bool, scale: float, device="cuda:0",
           stream=None):
    """Runs fa_fwd through the C ABI; returns (O bits [B,H,N,d], LSE float32 [B,H,N])."""
    import torch
    import attention_forward_flashattention_gb300 as fa
    q, k, v = (to_device(x, dtype, device) for x in (q_bits, k_bits, v_bits))
    o = torch.full_like(q, float("nan"))
    lse = torch.full(q.shape[:3], float("nan"), dtype=torch.float32, device=device)
    fa.attention_forward_into(q, k, v, o, lse, causal, scale, stream)
    rc = fa.fa_check(0 if stream is None else int(stream.cuda_stream))
    assert rc == fa.FA_OK, fa.status_string(rc)
    torch.cuda.synchronize()
    return to_bits(o), lse.cpu().numpy()


def sample_rows(B: int, H: int, N: int, n: int, seed: int) -> np.ndarray:
    """Flat rows bh * N + i: tile edges of the first, middle and last heads,
    plus random rows; grouped by head."""
    rng = np.random.default_rng(seed)
    BH = B * H
    heads = sorted({0, BH // 2, BH - 1})
    edge = [0, 1, 127, 128, 129, 255, 256, N // 2, N - 129, N - 128, N - 2, N - 1]
    rows = {h * N + i for h in heads for i in edge if 0 <= i < N}
    while len(rows) < n:
        rows.add(int(rng.integers(0, BH)) * N + int(rng.integers(0, N)))
    return np.array(sorted(rows), dtype=np.int64)
