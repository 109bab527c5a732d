"""Build libqmm.so in-tree with nvcc for sm_103a (GB300).

Each translation unit is compiled in parallel into ``_build/`` and linked into
``block_quantized_matmul_q4_gb300/libqmm.so``. nvcc cross-compiles without a
GPU, so this runs on any machine with the CUDA 13 toolkit.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libqmm.so")

SOURCES = ["api.cu", "quantize.cu", "repack.cu", "gemv.cu", "debug.cu", "static_scratch.cu", "tmap.cu",
           "w4a16.cu", "gemm_f16.cu", "gemv_mma.cu", "gemv_mma6.cu", "streamk.cu", "peaks.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE,
                 "-I", CSRC, "--expt-relaxed-constexpr"]
# Translation units whose integer results are decided by fp32 arithmetic:
# no contraction, IEEE division and square root.
EXACT = {"quantize.cu": ["-fmad=false", "-prec-div=true", "-prec-sqrt=true"]}


def nvcc() -> str:
    for c in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libqmm")


def _deps():
    hdrs = [os.path.join(INCLUDE, "qmm.h")] + [os.path.join(CSRC, f) for f in os.listdir(CSRC)
                                               if f.endswith(".cuh")]
    return hdrs


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src: str) -> str:
    obj = os.path.join(BUILD, src.replace(".cu", ".o"))
    deps = [os.path.join(CSRC, src)] + _deps() + [__file__]
    if _stale(obj, deps):
        cmd = [nvcc(), "-c", os.path.join(CSRC, src), "-o", obj] + COMMON + EXACT.get(src, [])
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    return obj


def build(verbose: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=min(len(SOURCES), os.cpu_count() or 1)) as ex:
        objs = list(ex.map(_compile, SOURCES))
    if _stale(LIB, objs):
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = [nvcc(), "-shared", "-o", tmp] + objs + ARCH
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, LIB)
    if verbose:
        print(LIB)
    return LIB


if __name__ == "__main__":
    build(verbose=True)
    sys.exit(0)
