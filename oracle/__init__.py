"""fp64 CPU oracle for the attention forward (16-bit and e4m3) and backward
passes (TEST INFRASTRUCTURE ONLY).

Only the test suite, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU
baseline / reference arm may import this package. The CUDA library never
imports, links or calls it, and it shares no code with the CUDA path: the two
meet only through the seeded input generator, which holds none of the
method's arithmetic.

The arithmetic lives in ``attn_ref.cpp`` (plain C++17, fp64, std::thread).
This module compiles it with g++ and wraps it with ctypes.

Parity pins: every function here is checked in ``tests/test_oracle_pins.py``
against closed forms, invariances, exhaustive decoder checks and an
explicit-softmax formulation built from scipy routines.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_ref.cpp")
_LIB = os.path.join(_HERE, "_build", "liboracle.so")
_lock = threading.Lock()
_lib = None

DTYPE_CODES = {"fp16": 0, "bf16": 1}


def build(force: bool = False) -> str:
    """Compiles attn_ref.cpp into a shared library (g++, -O2, no fast-math)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["g++", "-std=c++17", "-O2", "-fno-fast-math", "-ffp-contract=off",
           "-fPIC", "-shared", "-pthread", _SRC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            u16p = ctypes.POINTER(ctypes.c_uint16)
            f64p = ctypes.POINTER(ctypes.c_double)
            i64 = ctypes.c_int64
            lib.oracle_threads.argtypes = [ctypes.c_int]
            lib.oracle_threads.restype = ctypes.c_int
            lib.oracle_decode.argtypes = [u16p, ctypes.c_int, i64, f64p]
            lib.oracle_decode.restype = None
            lib.oracle_attn_fwd.argtypes = [u16p, u16p, u16p, ctypes.c_int, i64, i64, i64, i64,
                                            ctypes.c_int, ctypes.c_float, f64p, f64p, ctypes.c_int]
            lib.oracle_attn_fwd.restype = ctypes.c_int
            lib.oracle_attn_rows.argtypes = [u16p, u16p, u16p, ctypes.c_int, i64, i64, i64, i64,
                                             ctypes.c_int, ctypes.c_float, ctypes.POINTER(i64), i64,
                                             f64p, f64p, ctypes.c_int]
            lib.oracle_attn_rows.restype = ctypes.c_int
            lib.oracle_attn_rows_dev.argtypes = [u16p, u16p, u16p, ctypes.c_int, i64, i64, i64,
                                                 i64, ctypes.c_int, ctypes.c_float,
                                                 ctypes.POINTER(i64), i64, f64p, f64p, f64p,
                                                 ctypes.c_int]
            lib.oracle_attn_rows_dev.restype = ctypes.c_int
            u8p = ctypes.POINTER(ctypes.c_uint8)
            f32p = ctypes.POINTER(ctypes.c_float)
            lib.oracle_attn_fp8.argtypes = [u8p, u8p, u8p, i64, i64, i64, i64, i64, ctypes.c_float,
                                            f32p, ctypes.c_float, ctypes.c_int, ctypes.c_float,
                                            ctypes.POINTER(i64), i64, f64p, f64p, f64p,
                                            ctypes.c_int]
            lib.oracle_attn_fp8.restype = ctypes.c_int
            lib.oracle_attn_bwd.argtypes = [u16p, u16p, u16p, u16p, ctypes.c_int, i64, i64, i64,
                                            i64, ctypes.c_int, ctypes.c_float,
                                            ctypes.POINTER(i64), i64] + [f64p] * 6 + [ctypes.c_int]
            lib.oracle_attn_bwd.restype = ctypes.c_int
            lib.oracle_decode_e4m3.argtypes = [u8p, i64, f64p]
            lib.oracle_decode_e4m3.restype = None
            _lib = lib
    return _lib


def _u16(a: np.ndarray):
    a = np.ascontiguousarray(a, dtype=np.uint16)
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16))


def threads(requested: int = 0) -> int:
    """Worker threads the oracle uses for ``requested`` (0 = every core)."""
    return _load().oracle_threads(requested)


def decode(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Exact decode of stored 16-bit values (``fp16`` or ``bf16``) to float64."""
    bits, p = _u16(bits)
    out = np.empty(bits.shape, dtype=np.float64)
    _load().oracle_decode(p, DTYPE_CODES[dtype], bits.size,
                          out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)))
    return out


def attn_fwd(q: np.ndarray, k: np.ndarray, v: np.ndarray, dtype: str, causal: bool,
             scale: float, nthreads: int = 0):
    """Full forward on [B, H, N, d] stored 16-bit inputs.

    Returns (O float64 [B, H, N, d], LSE float64 [B, H, N]). ``scale`` is taken
    as the float32 value the CUDA library receives.
    """
    assert q.shape == k.shape == v.shape and q.ndim == 4
    B, H, N, d = q.shape
    q, qp = _u16(q)
    k, kp = _u16(k)
    v, vp = _u16(v)
    o = np.empty((B, H, N, d), dtype=np.float64)
    lse = np.empty((B, H, N), dtype=np.float64)
    rc = _load().oracle_attn_fwd(qp, kp, vp, DTYPE_CODES[dtype], B, H, N, d, int(bool(causal)),
                                 float(np.float32(scale)),
                                 o.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
                                 lse.ctypes.data_as(ctypes.POINTER(ctypes.c_double)), nthreads)
    if rc != 0:
        raise ValueError("oracle_attn_fwd rejected its arguments")
    return o, lse


def attn_rows(q: np.ndarray, k: np.ndarray, v: np.ndarray, dtype: str, causal: bool,
              scale: float, rows: np.ndarray, nthreads: int = 0):
    """Selected rows of the forward. ``rows`` are flat indices bh * N + i.

    Returns (O float64 [R, d], LSE float64 [R]).
    """
    assert q.shape == k.shape == v.shape and q.ndim == 4
    B, H, N, d = q.shape
    q, qp = _u16(q)
    k, kp = _u16(k)
    v, vp = _u16(v)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    o = np.empty((rows.size, d), dtype=np.float64)
    lse = np.empty((rows.size,), dtype=np.float64)
    rc = _load().oracle_attn_rows(qp, kp, vp, DTYPE_CODES[dtype], B, H, N, d, int(bool(causal)),
                                  float(np.float32(scale)),
                                  rows.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), rows.size,
                                  o.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
                                  lse.ctypes.data_as(ctypes.POINTER(ctypes.c_double)), nthreads)
    if rc != 0:
        raise ValueError("oracle_attn_rows rejected its arguments")
    return o, lse


def attn_rows_dev(q: np.ndarray, k: np.ndarray, v: np.ndarray, dtype: str, causal: bool,
                  scale: float, rows: np.ndarray, nthreads: int = 0):
    """Selected rows of the forward (as attn_rows) and, per element, the
    weighted mean absolute deviation of V under the row's softmax weights,
    dev_t = sum_j p_j |v_jt - O_t| / sum_j p_j: rounding every weight with
    relative error at most u moves O_t by at most u / (1 - u) * dev_t.

    Returns (O float64 [R, d], LSE float64 [R], dev float64 [R, d]).
    """
    assert q.shape == k.shape == v.shape and q.ndim == 4
    B, H, N, d = q.shape
    q, qp = _u16(q)
    k, kp = _u16(k)
    v, vp = _u16(v)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    o = np.empty((rows.size, d), dtype=np.float64)
    lse = np.empty((rows.size,), dtype=np.float64)
    dev = np.empty((rows.size, d), dtype=np.float64)
    f64 = ctypes.POINTER(ctypes.c_double)
    rc = _load().oracle_attn_rows_dev(qp, kp, vp, DTYPE_CODES[dtype], B, H, N, d,
                                      int(bool(causal)), float(np.float32(scale)),
                                      rows.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
                                      rows.size, o.ctypes.data_as(f64), lse.ctypes.data_as(f64),
                                      dev.ctypes.data_as(f64), nthreads)
    if rc != 0:
        raise ValueError("oracle_attn_rows_dev rejected its arguments")
    return o, lse, dev


def _u8(a: np.ndarray):
    a = np.ascontiguousarray(a, dtype=np.uint8)
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8))


def decode_e4m3(codes: np.ndarray) -> np.ndarray:
    """Exact decode of e4m3 codes (OCP FP8 E4M3, "fn" variant) to float64."""
    codes, p = _u8(codes)
    out = np.empty(codes.shape, dtype=np.float64)
    _load().oracle_decode_e4m3(p, codes.size, out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)))
    return out


def attn_fp8(q8: np.ndarray, k8: np.ndarray, vt8: np.ndarray, q_scale: float,
             k_scales: np.ndarray, v_scale: float, causal: bool, scale: float,
             rows: np.ndarray | None = None, nthreads: int = 0):
    """8-bit forward on e4m3 codes: q8, k8 [B, H, N, d], vt8 [B, H, d, ldv] (V
    transposed), k_scales float32 [B, H, ceil(N / 128)] (one per 128-key block).

    Returns (O float64 [R, d], LSE float64 [R], bound float64 [R, d]) for the
    flat rows ``rows`` (bh * N + i), or every row in order when ``rows`` is None;
    ``bound`` bounds |O' - O| for any kernel that rounds the softmax weights to
    e4m3 before the P V product (see attend_row_bound in attn_ref.cpp).
    """
    B, H, N, d = q8.shape
    ldv = vt8.shape[-1]
    assert k8.shape == q8.shape and vt8.shape == (B, H, d, ldv)
    assert k_scales.shape == (B, H, (N + 127) // 128)
    q8, qp = _u8(q8)
    k8, kp = _u8(k8)
    vt8, vp = _u8(vt8)
    ks = np.ascontiguousarray(k_scales, dtype=np.float32)
    if rows is None:
        nr, rp = B * H * N, None
    else:
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        nr, rp = rows.size, rows.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))
    o = np.empty((nr, d), dtype=np.float64)
    lse = np.empty((nr,), dtype=np.float64)
    bound = np.empty((nr, d), dtype=np.float64)
    f64 = ctypes.POINTER(ctypes.c_double)
    rc = _load().oracle_attn_fp8(qp, kp, vp, B, H, N, d, ldv, float(np.float32(q_scale)),
                                 ks.ctypes.data_as(ctypes.POINTER(ctypes.c_float)),
                                 float(np.float32(v_scale)), int(bool(causal)),
                                 float(np.float32(scale)), rp, nr, o.ctypes.data_as(f64),
                                 lse.ctypes.data_as(f64), bound.ctypes.data_as(f64), nthreads)
    if rc != 0:
        raise ValueError("oracle_attn_fp8 rejected its arguments")
    return o, lse, bound


def attn_bwd(q: np.ndarray, k: np.ndarray, v: np.ndarray, dout: np.ndarray, dtype: str,
             causal: bool, scale: float, heads=None, nthreads: int = 0):
    """Backward of the forward on [B, H, N, d] stored 16-bit inputs, for the
    flat heads ``heads`` (bh indices; all heads when None), from the
    definition (see bwd_head in attn_ref.cpp).

    Returns a dict of float64 [nheads, N, d] arrays: dq, dk, dv and the
    magnitude sums mag_dq, mag_dk, mag_dv.
    """
    assert q.shape == k.shape == v.shape == dout.shape and q.ndim == 4
    B, H, N, d = q.shape
    heads = np.arange(B * H) if heads is None else np.asarray(heads)
    heads = np.ascontiguousarray(heads, dtype=np.int64)
    q, qp = _u16(q)
    k, kp = _u16(k)
    v, vp = _u16(v)
    dout, dp = _u16(dout)
    names = ("dq", "dk", "dv", "mag_dq", "mag_dk", "mag_dv")
    out = {n: np.empty((heads.size, N, d), dtype=np.float64) for n in names}
    f64 = ctypes.POINTER(ctypes.c_double)
    rc = _load().oracle_attn_bwd(qp, kp, vp, dp, DTYPE_CODES[dtype], B, H, N, d,
                                 int(bool(causal)), float(np.float32(scale)),
                                 heads.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), heads.size,
                                 *[out[n].ctypes.data_as(f64) for n in names], nthreads)
    if rc != 0:
        raise ValueError("oracle_attn_bwd rejected its arguments")
    return out
