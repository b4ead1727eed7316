"""Build libsampler.so in-tree with nvcc for sm_103a (GB300).

The library has five translation units (the C ABI's host code, the slice
kernel and its variant with the extensions, the fork-group kernel, the LM-head
GEMM); they compile in parallel and link into one shared object.
"""
from __future__ import annotations

import glob
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libsampler.so")
OBJ_DIR = os.path.join(PKG, "_build")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = [*ARCH, "-lineinfo", "-O3", "-std=c++17", "-Xcompiler", "-fPIC"]
UNITS = ("sampler_api.cu", "slice_kernel.cu", "slice_kernel_ext.cu", "group_kernel.cu", "lm_head_kernel.cu")


def sources() -> list:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cuh"))
                  + glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(INCLUDE, "*.h")))


def is_stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(s) > t for s in sources())


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.isabs(cand) and os.path.exists(cand) or not os.path.isabs(cand)):
            return cand
    return "nvcc"


def _compile(unit: str, verbose: bool) -> str:
    obj = os.path.join(OBJ_DIR, unit.replace(".cu", f".{os.getpid()}.o"))
    cmd = [nvcc(), *NVCC_FLAGS, f"-I{INCLUDE}", "-c", "-o", obj, os.path.join(CSRC, unit)]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    subprocess.run(cmd, check=True)
    return obj


def build_library(force: bool = False, verbose: bool = False) -> str:
    """Compile the CUDA sources into libsampler.so next to this file (if stale)."""
    if not force and not is_stale():
        return LIB
    os.makedirs(OBJ_DIR, exist_ok=True)
    with ThreadPoolExecutor(len(UNITS)) as ex:
        objs = list(ex.map(lambda u: _compile(u, verbose), UNITS))
    tmp = LIB + f".tmp{os.getpid()}"
    try:
        subprocess.run([nvcc(), *ARCH, "-shared", "-o", tmp, *objs], check=True)
        os.replace(tmp, LIB)
    finally:
        for o in objs:
            if os.path.exists(o):
                os.remove(o)
    return LIB


if __name__ == "__main__":
    print(build_library(force=True, verbose=True))
