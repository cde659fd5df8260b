"""Builds libfp8q.so in-tree with nvcc for sm_103a.

    python -m fp8_fine_grained_25_b300.build [--verbose]

The library is a plain shared object with a C ABI (include/fp8q.h); the
CUDA runtime is linked statically and the driver's tensor-map encoder is
reached through the runtime's driver entry point, so the library needs no
libcuda at link time.
"""
from __future__ import annotations

import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libfp8q.so")
SOURCES = ["api.cu", "quant.cu", "gemm.cu", "gemm_pair.cu", "gemm_bs.cu"]
HEADERS = ["ptx.cuh", "gemm.cuh", "gemm_kernel.cuh", "quant.cuh"]
# ptxas options per source: the block-scaled dense GEMM's pair-tile kernels
# measured faster at -O1 (see gemm_pair.cu); everything else uses the default
PTXAS = {"gemm_pair.cu": ["-Xptxas", "-O1"]}
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.sep not in cand or os.path.exists(cand)):
            return cand
    raise RuntimeError("nvcc not found")


def _inputs():
    files = [os.path.join(CSRC, s) for s in SOURCES + HEADERS]
    files.append(os.path.join(INCLUDE, "fp8q.h"))
    files.append(os.path.abspath(__file__))
    return files


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and up_to_date():
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    common = [*ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-fvisibility=hidden",
              "-I", INCLUDE, "-I", CSRC]
    objs = []
    try:
        for src in SOURCES:
            obj = f"{tmp}.{src}.o"
            cmd = [nvcc(), *common, *PTXAS.get(src, []), "-c", os.path.join(CSRC, src), "-o", obj]
            if verbose:
                cmd.insert(1, "-Xptxas=-v")
            res = subprocess.run(cmd, capture_output=True, text=True)
            if res.returncode != 0:
                raise RuntimeError(f"nvcc failed on {src}:\n" + res.stdout + res.stderr)
            if verbose:
                sys.stderr.write(res.stdout + res.stderr)
            objs.append(obj)
        res = subprocess.run([nvcc(), *ARCH, "-shared", "-o", tmp, *objs], capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError("nvcc link failed:\n" + res.stdout + res.stderr)
    finally:
        for obj in objs:
            if os.path.exists(obj):
                os.remove(obj)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose="--verbose" in sys.argv))
