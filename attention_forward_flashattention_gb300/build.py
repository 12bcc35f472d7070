"""Builds the CUDA libraries in-tree with nvcc for sm_103a.

  _build/libfa_sm103.so    the product: C ABI of include/fa.h
  _build/libfa_selftest.so GPU unit tests of the PTX building blocks

Translation units are compiled in parallel (one nvcc process each), then
linked. ptxas resource usage (registers, spills, shared memory) of every
kernel is kept in _build/ptxas_<unit>.log.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OUT = os.path.join(PKG, "_build")
INCLUDE = os.path.join(ROOT, "include")

LIB_NAME = "libfa_sm103.so"
SELFTEST_NAME = "libfa_selftest.so"
LIB_UNITS = ["fa_host.cu", "fa_fwd_d64.cu", "fa_fwd_d128.cu", "fa_fwd_fp8.cu", "fa_fwd_pair.cu",
             "fa_bwd_d64.cu", "fa_bwd_d128.cu", "fa_noalloc.cu", "fa_pipeline.cu"]
SELFTEST_UNITS = ["selftest.cu"]
HEADERS = ["ptx.cuh", "fa_common.cuh", "fa_kernel.cuh", "fa_launch.cuh", "fa_pair.cuh", "fa_bwd.cuh",
           "fa_bwd_launch.cuh", "fa_dispatch.h"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found (set NVCC or put the CUDA toolkit on PATH)")


def _cuda_home(nvcc: str) -> str:
    return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))


def _flags() -> list[str]:
    return ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                   "-Xptxas", "-v", "-I", INCLUDE, "-I", CSRC]


def lib_path() -> str:
    return os.path.join(OUT, LIB_NAME)


def selftest_path() -> str:
    return os.path.join(OUT, SELFTEST_NAME)


def _stale(target: str, sources: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    deps = [os.path.join(CSRC, s) for s in sources + HEADERS] + [os.path.join(INCLUDE, "fa.h")]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> tuple[str, str]:
    """Compiles both libraries if any source is newer; returns their paths."""
    nvcc = nvcc_path()
    os.makedirs(OUT, exist_ok=True)
    jobs = []
    for units, name in ((LIB_UNITS, LIB_NAME), (SELFTEST_UNITS, SELFTEST_NAME)):
        if force or _stale(os.path.join(OUT, name), units):
            jobs.append((units, name))
    if not jobs:
        return lib_path(), selftest_path()
    procs = []
    for units, _ in jobs:
        for u in units:
            obj = os.path.join(OUT, u.replace(".cu", ".o"))
            log = open(os.path.join(OUT, "ptxas_" + u.replace(".cu", ".log")), "w")
            cmd = [nvcc] + _flags() + ["-c", os.path.join(CSRC, u), "-o", obj]
            if verbose:
                print(" ".join(cmd), file=sys.stderr)
            procs.append((u, subprocess.Popen(cmd, stdout=log, stderr=subprocess.STDOUT), log))
    failed = []
    for u, p, log in procs:
        p.wait()
        log.close()
        if p.returncode != 0:
            failed.append(u)
    if failed:
        msgs = []
        for u in failed:
            with open(os.path.join(OUT, "ptxas_" + u.replace(".cu", ".log"))) as f:
                msgs.append(f"--- {u}\n" + f.read()[-6000:])
        raise RuntimeError("nvcc failed:\n" + "\n".join(msgs))
    libdir = os.path.join(_cuda_home(nvcc), "lib64")
    for units, name in jobs:
        objs = [os.path.join(OUT, u.replace(".cu", ".o")) for u in units]
        tmp = os.path.join(OUT, name + f".tmp{os.getpid()}")
        cmd = [nvcc] + ARCH + ["-shared", "-cudart", "shared", "-o", tmp] + objs + [
            "-Xlinker", "-rpath", "-Xlinker", libdir]
        subprocess.run(cmd, check=True)
        os.replace(tmp, os.path.join(OUT, name))
    return lib_path(), selftest_path()


if __name__ == "__main__":
    paths = build(force="--force" in sys.argv, verbose=True)
    print("\n".join(paths))
