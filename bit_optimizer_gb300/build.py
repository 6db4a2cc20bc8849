"""Builds libfp8opt.so in-tree (bit_optimizer_gb300/_build) with nvcc for
sm_103a: one object per .cu file, compiled in parallel, then linked.

Flags that matter for results: ``-fmad=false`` (no multiply-add contraction
in device code, so each product and sum is rounded on its own) and
``-ffp-contract=off`` for the host compiler (the per-call scalars).  Division
and square root keep nvcc's IEEE defaults (``-prec-div=true
-prec-sqrt=true``), and denormals are kept (``-ftz=false``).
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libfp8opt.so")
SOURCES = ["api.cu", "cast_kernels.cu", "step_kernels.cu", "fused_kernels.cu",
           "noalloc.cu", "reduce_kernels.cu", "norm_kernels.cu"]
DEPS = ["fp8opt_internal.cuh", os.path.join("..", "..", "include", "fp8opt.h")]

NVCC = os.environ.get("NVCC", "nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-fmad=false", "-ftz=false",
         "-prec-div=true", "-prec-sqrt=true", "-Xcompiler",
         "-fPIC,-ffp-contract=off,-fvisibility=hidden", "-Xptxas",
         "-warn-spills"]


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    paths = [os.path.join(CSRC, s) for s in SOURCES + DEPS] + [__file__]
    return any(os.path.getmtime(p) > t for p in paths)


def _compile(src: str, verbose: bool) -> str:
    obj = os.path.join(OUT_DIR, os.path.splitext(src)[0] + ".o")
    cmd = [NVCC, *ARCH, *FLAGS, "-c", os.path.join(CSRC, src), "-o", obj]
    if verbose:
        cmd += ["-Xptxas", "-v"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    if verbose and (r.stdout or r.stderr):
        sys.stderr.write(r.stdout + r.stderr)
    return obj


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile and link libfp8opt.so if a source is newer; return its path."""
    if not force and not _stale():
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    with cf.ThreadPoolExecutor(len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose), SOURCES))
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [NVCC, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
