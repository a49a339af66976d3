"""Build libsvdq.so in-tree: the host pack (g++/OpenMP) and the sm_103a kernels (nvcc).

    python -m w4a4_rank_corrected_e2m1_b300.build [--force] [-v]

nvcc cross-compiles for sm_103a without a GPU.  The CUDA runtime is linked
statically, so the library only needs the NVIDIA driver at run time.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
ROOT = os.path.dirname(PKG)
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libsvdq.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xptxas", "-v",
                     "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")]
CXX_FLAGS = ["-O3", "-std=c++17", "-fPIC", "-fopenmp", "-ffp-contract=off", "-I", os.path.join(ROOT, "include")]

CU_SOURCES = ["api.cu", "k1_actquant.cu", "k2_fp4gemm.cu", "awq_gemv.cu", "int4_path.cu", "int4_api.cu"]
CXX_SOURCES = ["pack_host.cpp", "awq_host.cpp"]
HEADERS = ["svdq_internal.h", "ptx.cuh", "abi_util.cuh", "nvfp4_block.cuh"]


def _nvcc() -> str:
    for c in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found")


def _stale(out: str, deps) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(d) > t for d in deps)


def _run(cmd, verbose):
    r = subprocess.run(cmd, capture_output=True, text=True)
    if verbose or r.returncode != 0:
        sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
    if r.returncode != 0:
        raise RuntimeError(f"build step failed: {' '.join(cmd[:3])} ...")
    return r.stdout + r.stderr


def build(force: bool = False, verbose: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    hdrs = [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(ROOT, "include", "svdq.h")]
    jobs = []
    objs = []
    for s in CU_SOURCES:
        src, obj = os.path.join(CSRC, s), os.path.join(BUILD, s + ".o")
        objs.append(obj)
        if force or _stale(obj, [src] + hdrs):
            jobs.append([_nvcc()] + NVCC_FLAGS + ["-c", src, "-o", obj])
    for s in CXX_SOURCES:
        src, obj = os.path.join(CSRC, s), os.path.join(BUILD, s + ".o")
        objs.append(obj)
        if force or _stale(obj, [src] + hdrs):
            jobs.append(["g++"] + CXX_FLAGS + ["-c", src, "-o", obj])
    logs = []
    with cf.ThreadPoolExecutor(max_workers=4) as ex:
        for out in ex.map(lambda c: _run(c, verbose), jobs):
            logs.append(out)
    if force or jobs or _stale(LIB, objs):
        _run([_nvcc()] + ARCH + ["-shared", "-cudart", "static", "-o", LIB] + objs + ["-Xcompiler", "-fopenmp"],
             verbose)
    with open(os.path.join(BUILD, "ptxas.log"), "a") as f:
        f.write("\n".join(logs))
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="-v" in sys.argv)
    print(LIB)
