"""The C ABI library builds, loads and exports what include/fa.h declares, and
rejects bad arguments before touching a GPU (runs without one)."""
import ctypes

import numpy as np
import pytest

import attention_forward_flashattention_gb300 as fa
from attention_forward_flashattention_gb300 import build as fabuild

GOOD = 0x100000  # 16-byte aligned stand-in pointer: never dereferenced by the checks


@pytest.fixture(scope="module")
def lib():
    fabuild.build()
    return fa.load_library()


def test_header_declares_expected_entry_points():
    names = fa.header_functions()
    assert names == ["fa_fwd", "fa_fwd_pair", "fa_fwd_strided", "fa_fwd_fp8", "fa_fwd_fp8_pair",
                     "fa_bwd", "fa_bwd_workspace_size",
                     "fa_fwd_noalloc", "fa_fwd_host", "fa_fwd_host_workspace_size", "fa_check",
                     "fa_sm_clock_read", "fa_query_launch",
                     "fa_sm_clock_probe", "fa_status_string", "fa_version"]


def test_library_exports_every_declared_symbol(lib):
    for name in fa.header_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_selftest_library_exports():
    _, st = fabuild.build()
    slib = ctypes.CDLL(st)
    for name in ("fa_selftest_gemm_qk", "fa_selftest_gemm_pv", "fa_selftest_gemm_ts",
                 "fa_selftest_gemm_qk_pair", "fa_selftest_gemm_pv_pair", "fa_selftest_wait_timeout",
                 "fa_selftest_gemm_qk_fp8", "fa_selftest_gemm_ts_fp8", "fa_selftest_pack_e4m3"):
        assert hasattr(slib, name)


def test_status_strings(lib):
    assert fa.status_string(fa.FA_OK) == "FA_OK"
    assert fa.status_string(fa.FA_ERR_TIMEOUT) == "FA_ERR_TIMEOUT"
    assert fa.status_string(99) == "FA_ERR_UNKNOWN"
    assert fa.fa_version() == 100


def _call(q=GOOD, k=GOOD, v=GOOD, o=GOOD, lse=GOOD, B=1, H=1, N=128, d=128, causal=0,
          scale=0.125, dtype=fa.FA_DTYPE_FP16):
    return fa.fa_fwd(q, k, v, o, lse, B, H, N, d, causal, scale, dtype, 0)


@pytest.mark.parametrize("kw", [dict(q=0), dict(k=0), dict(v=0), dict(o=0), dict(lse=0)])
def test_null_pointers_rejected(lib, kw):
    assert _call(**kw) == fa.FA_ERR_INVALID_ARG


@pytest.mark.parametrize("kw", [dict(q=GOOD + 2), dict(v=GOOD + 8), dict(o=GOOD + 4),
                                dict(lse=GOOD + 4)])
def test_misaligned_pointers_rejected(lib, kw):
    assert _call(**kw) == fa.FA_ERR_INVALID_ARG


@pytest.mark.parametrize("scale", [0.0, -0.125, float("nan"), float("inf")])
def test_bad_scale_rejected(lib, scale):
    assert _call(scale=scale) == fa.FA_ERR_INVALID_ARG


@pytest.mark.parametrize("kw", [dict(B=0), dict(H=0), dict(N=0), dict(N=-5), dict(dtype=2),
                                dict(dtype=-1)])
def test_bad_sizes_and_dtype_rejected(lib, kw):
    assert _call(**kw) == fa.FA_ERR_INVALID_ARG


@pytest.mark.parametrize("kw", [dict(d=96), dict(d=256), dict(d=32), dict(N=(1 << 30) + 1),
                                dict(B=1 << 16, H=1 << 16)])
def test_unsupported_shapes(lib, kw):
    assert _call(**kw) == fa.FA_ERR_UNSUPPORTED


def test_no_device_is_an_error_not_a_fallback(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    # valid arguments on a machine without a GPU must fail, never compute on the CPU
    assert _call() in (fa.FA_ERR_CUDA, fa.FA_ERR_ARCH)


def test_missing_library_raises(tmp_path):
    with pytest.raises(RuntimeError):
        fa.load_library(str(tmp_path / "libfa_sm103.so"))


def _strided(strides, d=128, N=128, **kw):
    args = dict(q=GOOD, k=GOOD, v=GOOD, o=GOOD, lse=GOOD, B=1, H=2, N=N, d=d)
    args.update(kw)
    return fa.fa_fwd_strided(args["q"], args["k"], args["v"], args["o"], args["lse"], args["B"],
                             args["H"], args["N"], args["d"], strides, 0, 0.125,
                             fa.FA_DTYPE_FP16, 0)


CONTIG = (2 * 128 * 128, 128 * 128, 128)   # [B][H][N][d], H=2, N=128, d=128
BNHD = (128 * 2 * 128, 128, 2 * 128)       # [B][N][H][d]


def test_strided_null_strides_rejected(lib):
    assert _strided(None) == fa.FA_ERR_INVALID_ARG


@pytest.mark.parametrize("bad", [(CONTIG[0], CONTIG[1], 130), (CONTIG[0], 4, 128),
                                 (0, CONTIG[1], 128), (CONTIG[0], -128, 128),
                                 (CONTIG[0], CONTIG[1], 64)])
@pytest.mark.parametrize("which", [0, 1, 2, 3])
def test_strided_bad_strides_rejected(lib, bad, which):
    s = [CONTIG] * 4
    s[which] = bad
    assert _strided(s) == fa.FA_ERR_INVALID_ARG


def test_strided_huge_strides_unsupported(lib):
    assert _strided([CONTIG, CONTIG, (1 << 38, CONTIG[1], 128), CONTIG]) == fa.FA_ERR_UNSUPPORTED


def test_strided_checks_sizes_and_pointers_first(lib):
    assert _strided([BNHD] * 4, d=96) == fa.FA_ERR_UNSUPPORTED
    assert _strided([BNHD] * 4, q=0) == fa.FA_ERR_INVALID_ARG
    assert _strided([BNHD] * 4, o=GOOD + 8) == fa.FA_ERR_INVALID_ARG


def test_strided_valid_layouts_reach_the_device(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    # valid strides pass every check; without a GPU the call must then fail, never fall back
    assert _strided([BNHD, CONTIG, (2 * 136 * 128, 136 * 128, 136), BNHD]) in (fa.FA_ERR_CUDA,
                                                                           fa.FA_ERR_ARCH)


FP8_ENTRIES = ["fa_fwd_fp8", "fa_fwd_fp8_pair"]


def _fp8(fn="fa_fwd_fp8", **kw):
    a = dict(q=GOOD, k=GOOD, vt=GOOD, o=GOOD, lse=GOOD, B=1, H=2, N=300, d=128, ldv=304,
             q_scale=0.01, k_scales=GOOD, v_scale=0.01, causal=0, scale=0.088)
    a.update(kw)
    return getattr(fa, fn)(a["q"], a["k"], a["vt"], a["o"], a["lse"], a["B"], a["H"], a["N"],
                           a["d"], a["ldv"], a["q_scale"], a["k_scales"], a["v_scale"],
                           a["causal"], a["scale"], 0)


@pytest.mark.parametrize("fn", FP8_ENTRIES)
@pytest.mark.parametrize("kw", [dict(q=0), dict(vt=0), dict(k_scales=0), dict(vt=GOOD + 8),
                                dict(k_scales=GOOD + 2), dict(ldv=296), dict(ldv=300),
                                dict(q_scale=0.0), dict(v_scale=float("nan")),
                                dict(scale=-1.0), dict(N=0)])
def test_fp8_bad_arguments_rejected(lib, kw, fn):
    assert _fp8(fn, **kw) == fa.FA_ERR_INVALID_ARG


@pytest.mark.parametrize("fn", FP8_ENTRIES)
@pytest.mark.parametrize("kw", [dict(d=64), dict(d=96)])
def test_fp8_head_dim_must_be_128(lib, kw, fn):
    assert _fp8(fn, **kw) == fa.FA_ERR_UNSUPPORTED


@pytest.mark.parametrize("fn", FP8_ENTRIES)
def test_fp8_valid_arguments_reach_the_device(lib, fn):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert _fp8(fn) in (fa.FA_ERR_CUDA, fa.FA_ERR_ARCH)


def _bwd(**kw):
    a = dict(q=GOOD, k=GOOD, v=GOOD, o=GOOD, dout=GOOD, lse=GOOD, dq=GOOD, dk=GOOD, dv=GOOD,
             ws=GOOD, B=1, H=2, N=300, d=128, causal=0, scale=0.088, dtype=fa.FA_DTYPE_FP16)
    a.update(kw)
    return fa.fa_bwd(a["q"], a["k"], a["v"], a["o"], a["dout"], a["lse"], a["dq"], a["dk"],
                     a["dv"], a["ws"], a["B"], a["H"], a["N"], a["d"], a["causal"], a["scale"],
                     a["dtype"], 0)


@pytest.mark.parametrize("kw", [dict(o=0), dict(dout=0), dict(lse=0), dict(dk=0), dict(ws=0),
                                dict(dq=GOOD + 8), dict(ws=GOOD + 4), dict(scale=0.0),
                                dict(dtype=3), dict(N=0)])
def test_bwd_bad_arguments_rejected(lib, kw):
    assert _bwd(**kw) == fa.FA_ERR_INVALID_ARG


def test_bwd_unsupported_and_workspace_size(lib):
    assert _bwd(d=96) == fa.FA_ERR_UNSUPPORTED
    # 2^30 units of 256 rows pass the forward's limit; 2^31 tiles of 128 rows do not
    assert _bwd(B=1, H=1 << 14, N=1 << 24) == fa.FA_ERR_UNSUPPORTED
    assert fa.fa_bwd_workspace_size(2, 3, 300, 64) == 2 * 2 * 3 * 3 * 128 * 4
    with pytest.raises(fa.FaError):
        fa.fa_bwd_workspace_size(1, 1, 128, 96)


def test_bwd_valid_arguments_reach_the_device(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert _bwd() in (fa.FA_ERR_CUDA, fa.FA_ERR_ARCH)


def _host(**kw):
    a = dict(q=GOOD, k=GOOD, v=GOOD, o=GOOD, lse=GOOD, B=2, H=3, N=300, d=128, causal=0,
             scale=0.088, dtype=fa.FA_DTYPE_FP16, ws=GOOD, wsz=None)
    a.update(kw)
    if a["wsz"] is None:
        a["wsz"] = 4 * a["B"] * a["H"] * a["N"] * 128 * 2 + a["B"] * a["H"] * a["N"] * 4 + 144
    return fa.fa_fwd_host(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["N"],
                          a["d"], a["causal"], a["scale"], a["dtype"], a["ws"], a["wsz"], 0)


@pytest.mark.parametrize("kw", [dict(q=0), dict(v=0), dict(o=0), dict(lse=0), dict(ws=0),
                                dict(ws=GOOD + 8), dict(wsz=1000), dict(scale=0.0),
                                dict(scale=float("inf")), dict(dtype=2), dict(N=0), dict(H=-1)])
def test_host_bad_arguments_rejected(lib, kw):
    assert _host(**kw) == fa.FA_ERR_INVALID_ARG


def test_host_unsupported_and_workspace_size(lib):
    assert _host(d=96) == fa.FA_ERR_UNSUPPORTED
    # Q, K, V, O (2 bytes each), LSE (4 bytes), 16 bytes of alignment padding
    # for each of up to 9 chunks
    assert fa.fa_fwd_host_workspace_size(2, 3, 300, 64) == 4 * 2 * 3 * 300 * 64 * 2 + \
        2 * 3 * 300 * 4 + 144
    with pytest.raises(fa.FaError):
        fa.fa_fwd_host_workspace_size(1, 1, 128, 96)


def test_host_valid_arguments_reach_the_device(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert _host() in (fa.FA_ERR_CUDA, fa.FA_ERR_ARCH)


C_PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "fa.h"

int main(void) {
  /* every entry point is a plain C function */
  typedef void (*fn_t)(void);
  fn_t fns[] = {(fn_t)fa_fwd, (fn_t)fa_fwd_pair, (fn_t)fa_fwd_strided, (fn_t)fa_fwd_fp8,
                (fn_t)fa_fwd_fp8_pair, (fn_t)fa_bwd,
                (fn_t)fa_bwd_workspace_size, (fn_t)fa_fwd_noalloc, (fn_t)fa_fwd_host,
                (fn_t)fa_fwd_host_workspace_size, (fn_t)fa_check, (fn_t)fa_sm_clock_read,
                (fn_t)fa_query_launch,
                (fn_t)fa_sm_clock_probe, (fn_t)fa_status_string, (fn_t)fa_version};
  size_t i;
  size_t ws = 0;
  for (i = 0; i < sizeof(fns) / sizeof(fns[0]); ++i)
    if (!fns[i]) return 1;
  if (strcmp(fa_status_string(FA_OK), "FA_OK") != 0) return 2;
  if (fa_version() <= 0) return 3;
  /* argument checks run before any device call */
  if (fa_fwd(NULL, NULL, NULL, NULL, NULL, 1, 1, 128, 128, 0, 0.125f, FA_DTYPE_FP16, NULL) !=
      FA_ERR_INVALID_ARG)
    return 4;
  if (fa_bwd_workspace_size(1, 1, 128, 96, &ws) != FA_ERR_UNSUPPORTED) return 5;
  printf("ok %d\n", fa_version());
  return 0;
}
"""


def test_header_is_plain_c_and_links(tmp_path):
    """include/fa.h compiles as strict C99 and a C program links against the
    library and runs its host-side checks (no GPU needed)."""
    import os
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    lib_path, _ = fabuild.build()
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    src = tmp_path / "use_fa.c"
    src.write_text(C_PROGRAM)
    exe = tmp_path / "use_fa"
    lib_dir = os.path.dirname(lib_path)
    lib_name = os.path.basename(lib_path)
    subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
                    "-I", os.path.join(root, "include"), str(src), "-o", str(exe),
                    os.path.join(lib_dir, lib_name), f"-Wl,-rpath,{lib_dir}"],
                   check=True, capture_output=True, text=True)
    env = dict(os.environ)
    nvcc = shutil.which("nvcc")
    if nvcc:  # the library's CUDA runtime
        cuda_lib = os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(nvcc))), "lib64")
        env["LD_LIBRARY_PATH"] = cuda_lib + os.pathsep + env.get("LD_LIBRARY_PATH", "")
    out = subprocess.run([str(exe)], capture_output=True, text=True, env=env, timeout=60)
    assert out.returncode == 0 and out.stdout.startswith("ok"), (out.returncode, out.stderr)


def _pair(q=GOOD, k=GOOD, v=GOOD, o=GOOD, lse=GOOD, B=1, H=1, N=128, d=128, causal=0,
          scale=0.125, dtype=fa.FA_DTYPE_FP16):
    return fa.fa_fwd_pair(q, k, v, o, lse, B, H, N, d, causal, scale, dtype, 0)


@pytest.mark.parametrize("kw,want", [
    (dict(q=0), fa.FA_ERR_INVALID_ARG), (dict(lse=GOOD + 4), fa.FA_ERR_INVALID_ARG),
    (dict(scale=0.0), fa.FA_ERR_INVALID_ARG), (dict(B=0), fa.FA_ERR_INVALID_ARG),
    (dict(dtype=2), fa.FA_ERR_INVALID_ARG), (dict(d=64), fa.FA_ERR_UNSUPPORTED),
    (dict(d=96), fa.FA_ERR_UNSUPPORTED), (dict(N=(1 << 30) + 1), fa.FA_ERR_UNSUPPORTED),
])
def test_pair_bad_arguments_rejected(lib, kw, want):
    """fa_fwd_pair checks its arguments like fa_fwd, and takes head dimension 128 only."""
    assert _pair(**kw) == want


def test_pair_no_device_is_an_error(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert _pair() in (fa.FA_ERR_CUDA, fa.FA_ERR_ARCH)
