"""Builds ``libkreduce.so`` (and the pipe probe ``libkrprobe.so``) in-tree from
``csrc/`` for sm_103a.

Each translation unit is compiled by its own ``nvcc`` process (in parallel), then
linked into a shared library with the CUDA runtime linked statically, so the
library depends on no particular ``libcudart`` build and loads next to any
PyTorch.  Run ``python -m symbolic_matrix_reductions_gb300.build`` or call
``build()``.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OBJ = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libkreduce.so")
# Debug variant (-DKR_DEBUG): the kernels check every global element index against its
# array's extent and report violations through kr_device_status; built only on request.
OBJ_DEBUG = os.path.join(HERE, "_build_debug")
LIB_DEBUG = os.path.join(HERE, "libkreduce_debug.so")
PROBE_LIB = os.path.join(HERE, "libkrprobe.so")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")

SOURCES = ["kr_api.cpp", "kr_fwd_sum.cu", "kr_fwd_lse.cu", "kr_grad.cu", "kr_knn.cu", "kr_combine.cu", "kr_records.cu",
           "kr_noalloc.cu", "kr_tc.cu", "kr_radial_gauss.cu", "kr_radial_laplace.cu", "kr_radial_cauchy.cu",
           "kr_radial_imq.cu"]
PROBE_SOURCES = ["kr_probe.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-std=c++17", "-O3", "-lineinfo", *ARCH, "-Xcompiler", "-fPIC", "-I", INCLUDE]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libkreduce.so")


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "kreduce.h"))
    files.append(os.path.abspath(__file__))
    return files


def up_to_date() -> bool:
    if not (os.path.exists(LIB) and os.path.exists(PROBE_LIB)):
        return False
    t = min(os.path.getmtime(LIB), os.path.getmtime(PROBE_LIB))
    return all(os.path.getmtime(f) <= t for f in _deps())


def build_debug(force: bool = False) -> str:
    """Compile and link the debug variant libkreduce_debug.so; returns its path."""
    if not force and os.path.exists(LIB_DEBUG) and all(os.path.getmtime(f) <= os.path.getmtime(LIB_DEBUG)
                                                       for f in _deps()):
        return LIB_DEBUG
    nvcc = _nvcc()
    os.makedirs(OBJ_DEBUG, exist_ok=True)

    def compile_one(src):
        obj = os.path.join(OBJ_DEBUG, os.path.splitext(src)[0] + ".o")
        cmd = [nvcc, *NVCC_FLAGS, "-DKR_DEBUG", "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src} (debug):\n{r.stdout}\n{r.stderr}")
        return obj

    with cf.ThreadPoolExecutor(max_workers=min(len(SOURCES), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = LIB_DEBUG + ".tmp"
    r = subprocess.run([nvcc, "-shared", *ARCH, "-cudart", "static", "-o", tmp, *objs], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed (debug):\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB_DEBUG)
    return LIB_DEBUG


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    """Compile and link the libraries; returns the path of libkreduce.so."""
    if not force and up_to_date():
        return LIB
    nvcc = _nvcc()
    os.makedirs(OBJ, exist_ok=True)

    def compile_one(src):
        obj = os.path.join(OBJ, os.path.splitext(src)[0] + ".o")
        cmd = [nvcc, *NVCC_FLAGS, *extra_flags, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            sys.stderr.write(r.stdout + r.stderr)
        return obj

    allsrc = SOURCES + PROBE_SOURCES
    with cf.ThreadPoolExecutor(max_workers=min(len(allsrc), os.cpu_count() or 4)) as ex:
        objs = dict(zip(allsrc, ex.map(compile_one, allsrc)))
    for lib, srcs in ((LIB, SOURCES), (PROBE_LIB, PROBE_SOURCES)):
        tmp = lib + ".tmp"
        cmd = [nvcc, "-shared", *ARCH, "-cudart", "static", "-o", tmp, *[objs[s] for s in srcs]]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
