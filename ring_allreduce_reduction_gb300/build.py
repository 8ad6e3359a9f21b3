"""Build libvrccl.so in-tree for sm_103a (nvcc, no CMake).

Translation units compile in parallel into ``_build/`` at the repository
root and link into ``ring_allreduce_reduction_gb300/libvrccl.so``. A unit
is rebuilt when it or any header is newer than its object.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libvrccl.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", f"-I{INCLUDE}", f"-I{CSRC}",
         "-Xcompiler", "-Wall", "--expt-relaxed-constexpr"]
SOURCES = ["kernels_simple.cu", "kernels_simple_x.cu", "kernels_ll.cu", "kernels_ll128.cu", "kernels_ll128w.cu",
           "kernels_ll128w_x.cu", "kernels_oneshot.cu", "kernels_group_simple.cu",
           "kernels_group_ll.cu", "kernels_group_ll128.cu", "vrccl.cu", "vrccl_noalloc.cu", "tuner.cc", "parse.cc",
           "model.cc"]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found (need the CUDA 13 toolkit)")
    return cand


def _cuda_lib_dir() -> str:
    nvcc = os.path.realpath(_nvcc())
    return os.path.join(os.path.dirname(os.path.dirname(nvcc)), "lib64")


def _newest_header() -> float:
    t = 0.0
    for d in (CSRC, INCLUDE):
        for f in os.listdir(d):
            if f.endswith((".h", ".cuh")):
                t = max(t, os.path.getmtime(os.path.join(d, f)))
    return t


def _compile(src: str, verbose: bool) -> str:
    obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
    srcp = os.path.join(CSRC, src)
    if os.path.exists(obj) and os.path.getmtime(obj) >= max(os.path.getmtime(srcp), _newest_header()):
        return obj
    cmd = [_nvcc(), *ARCH, *FLAGS, "-c", srcp, "-o", obj]
    if src.endswith(".cc"):
        cmd = [_nvcc(), *FLAGS, "-x", "c++", "-c", srcp, "-o", obj]
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"compiling {src} failed:\n{r.stdout}\n{r.stderr}")
    return obj


def build(verbose: bool = False, force: bool = False) -> str:
    """Compile every unit (in parallel) and link the shared library."""
    os.makedirs(BUILD, exist_ok=True)
    if force:
        for f in os.listdir(BUILD):
            if f.endswith(".o"):
                os.remove(os.path.join(BUILD, f))
    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose), SOURCES))
    if os.path.exists(LIB) and os.path.getmtime(LIB) >= max(os.path.getmtime(o) for o in objs):
        return LIB
    tmp = LIB + ".tmp"
    cmd = [_nvcc(), *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs,
           "-Xlinker", f"-rpath,{_cuda_lib_dir()}"]
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"linking libvrccl.so failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv))
