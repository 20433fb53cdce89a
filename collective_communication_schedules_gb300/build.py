"""Builds libhoc.so in place: the CUDA kernels and the C++ runtime for sm_103a.

Run ``python -m collective_communication_schedules_gb300.build`` (or call
``build()``).  Objects go to ``_build/`` next to this file; the shared library
to ``libhoc.so`` in the package directory.  The CUDA runtime is linked
statically, so the library loads (and reports HOC_ERR_NO_DEVICE) on machines
without a GPU.
"""
from __future__ import annotations

import os
import platform
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libhoc.so")
STAMP = LIB + ".stamp"  # the machine the library was built for: a copy from another machine is rebuilt

SOURCES = ["reduce.cu", "reduce_tma.cu", "tma_copy.cu", "workload.cu", "plan.cpp", "hoc.cpp", "topo_sched.cpp", "proxy.cpp", "ep.cu", "host_ar.cpp"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I" + INCLUDE, "-I" + CSRC]
# IEEE arithmetic in the reduce kernels: no flush to zero, no fast math.
CUDA_ONLY = ["-ftz=false", "-prec-div=true", "-prec-sqrt=true"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libhoc.so")


def _inputs() -> list[str]:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cu", ".cpp", ".h", ".cuh"))]
    files += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    return files + [os.path.abspath(__file__)]


def _machine() -> str:
    return platform.machine()


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    try:
        with open(STAMP) as f:
            if f.read().strip() != _machine():
                return False
    except OSError:
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def _compile(src: str) -> str:
    obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc()] + ARCH + COMMON
    if src.endswith(".cu"):
        cmd += CUDA_ONLY
    else:
        cmd += ["-x", "c++"]
    cmd += ["-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"compile failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    return obj


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and up_to_date():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(_compile, SOURCES))
    tmp = LIB + ".tmp"
    cmd = [nvcc()] + ARCH + ["-shared", "-cudart", "static", "-o", tmp] + objs + ["-lpthread", "-ldl", "-lrt"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    with open(STAMP, "w") as f:
        f.write(_machine() + "\n")
    if verbose:
        print("built", LIB)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True)
