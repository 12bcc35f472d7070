"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI,
decode its outputs, and compare them with the fp64 oracle.

Tolerances (the stated bounds of the library's specification, for N(0, 1)
inputs), asserted as stated:
  * O: every element |O_gpu - O_ref| <= 1e-2 and mean |O_gpu - O_ref| <= 1e-3;
  * LSE: max |LSE_gpu - LSE_ref| <= 1e-3.
One case is set apart rather than passed: an element whose exact value lies
more than 1e-2 from every value of the 16-bit output format X (the rounding
floor |round_X(O_ref) - O_ref| > 1e-2, possible for bf16 at |O| >= 4, where
the spacing is 2^-5) cannot meet the bound in any X-output kernel. Such
elements are counted as "unattainable" in the result and must lie within
1e-2 + half an X spacing of O_ref; every other element must meet 1e-2.

Inputs that are not N(0, 1) (Q scaled x 3 to sharpen the softmax) fall
outside the stated bound. There an element above 1e-2 must lie within the
bound derived from the two roundings the method prescribes (explain_over):
half an X spacing of O_ref (the output) plus u / (1 - u) times the weighted
mean absolute deviation of V under the row's softmax weights (every weight
rounded to X, unit roundoff u, before the P V product), plus 2e-5 of fp32
arithmetic. The count of such elements is reported.
The rounding floor's maximum over all elements is reported alongside.
"""
from __future__ import annotations

import json
import os

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


def round_to(x: np.ndarray, dtype: str) -> np.ndarray:
    """x rounded to the nearest value of format `dtype` (ties to even), as float64."""
    x = np.asarray(x, dtype=np.float64)
    if dtype == "fp16":
        return x.astype(np.float16).astype(np.float64)
    # bf16: float64 -> float32 is exact only to 24 bits, so round the float64
    # value directly to 8 significant bits (ties to even on the scaled value)
    m, e = np.frexp(x)                    # x = m 2^e, |m| in [0.5, 1)
    return np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)


def compare(o_bits: np.ndarray, lse: np.ndarray, o_ref: np.ndarray, lse_ref: np.ndarray,
            dtype: str) -> dict:
    o = bits_to_f64(o_bits, dtype)
    o_ref = np.asarray(o_ref, dtype=np.float64)
    err = np.abs(o - o_ref)
    lerr = np.abs(np.asarray(lse, dtype=np.float64) - lse_ref)
    floor = np.abs(round_to(o_ref, dtype) - o_ref)
    over = err > O_MAX_ABS
    unattainable = over & (floor > O_MAX_ABS)
    attainable_over = over & ~unattainable
    relaxed_bad = unattainable & (err > O_MAX_ABS + half_ulp(o_ref, dtype))
    res = {
        "o_max_abs": float(err.max()) if err.size else 0.0,
        "o_mean_abs": float(err.mean()) if err.size else 0.0,
        "o_rounding_floor_max": float(floor.max()) if err.size else 0.0,
        "o_over_bound": int(attainable_over.sum()),
        "o_unattainable": int(unattainable.sum()),
        "lse_max_abs": float(lerr.max()) if lerr.size else 0.0,
        "elements": int(err.size),
        "finite": bool(np.all(np.isfinite(o)) and np.all(np.isfinite(lse))),
    }
    if over.any():  # the largest errors above the bound, for the record
        idx = np.flatnonzero(over.reshape(-1))
        res["_over_flat"] = idx
        res["_over_err"] = err.reshape(-1)[idx]
        top = idx[np.argsort(-res["_over_err"])][:32]
        res["over_elements"] = [
            {"flat": int(i), "o_gpu": float(o.reshape(-1)[i]), "o_ref": float(o_ref.reshape(-1)[i]),
             "floor": float(floor.reshape(-1)[i])} for i in top]
    res["ok"] = (res["finite"] and res["o_mean_abs"] <= O_MEAN_ABS
                 and res["o_over_bound"] == 0 and not relaxed_bad.any()
                 and res["lse_max_abs"] <= LSE_MAX_ABS)
    return res


# unit roundoff 2^-p of a p-significant-bit format: the largest relative error
# of round-to-nearest (half the spacing 2^(e + 1 - p) over the smallest value
# 2^e of a binade)
UNIT_ROUNDOFF = {"fp16": 2.0 ** -11, "bf16": 2.0 ** -8}


def explain_over(res: dict, oracle, q, k, v, dtype: str, causal: bool, scale: float,
                 d: int) -> dict:
    """For inputs outside the stated bound's N(0, 1) clause: checks every
    element above 1e-2 against the bound derived from the method's two
    roundings (16-bit P, 16-bit O) and sets res["ok"] accordingly. Adds
    o_over_bound_within_rounding_bound (count) and the largest ratio of error
    to that bound."""
    idx = res.get("_over_flat")
    if idx is None or idx.size == 0:
        res["o_over_bound_within_rounding_bound"] = 0
        return res
    rows, cols = idx // d, idx % d
    urows, inv = np.unique(rows, return_inverse=True)
    o_ref, _, dev = oracle.attn_rows_dev(q, k, v, dtype, causal, scale, urows)
    ref = o_ref[inv, cols]
    u = UNIT_ROUNDOFF[dtype]
    allowed = half_ulp(ref, dtype) + u / (1.0 - u) * dev[inv, cols] + 2e-5
    ratio = res["_over_err"] / allowed
    res["o_over_bound_within_rounding_bound"] = int((ratio <= 1.0).sum())
    res["o_over_bound_max_ratio_to_rounding_bound"] = float(ratio.max())
    res["ok"] = (res["finite"] and res["o_mean_abs"] <= O_MEAN_ABS
                 and bool(np.all(ratio <= 1.0)) and res["lse_max_abs"] <= LSE_MAX_ABS)
    return res


def record(name: str, res: dict, **extra) -> None:
    """Appends one JSON line (a parity result) to the file named by the
    FA_PARITY_RECORD environment variable, if it is set."""
    path = os.environ.get("FA_PARITY_RECORD")
    if path:
        keep = {k: v for k, v in res.items() if not k.startswith("_")}
        with open(path, "a") as f:
            f.write(json.dumps({"case": name, **keep, **extra}) + "\n")


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
