"""Build the in-tree CUDA library ``_lib/libw12.so`` for sm_103a.

Each translation unit is compiled in parallel with nvcc (host C++ with g++),
then linked into one shared library with the CUDA runtime linked statically.
Nothing is installed; the library lands next to this file.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
BUILD = os.path.join(HERE, "_build")
LIBDIR = os.path.join(HERE, "_lib")
LIB = os.path.join(LIBDIR, "libw12.so")

CU_SOURCES = ("runtime.cu", "gemm_fma.cu", "gemm_tc.cu", "decode.cu", "noalloc.cu", "encode.cu", "reduce.cu", "i8.cu")
CPP_SOURCES = ("host.cpp",)
HEADERS = ("ptx.cuh", "kernels.cuh", "w12_internal.h")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for c in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found: the W12 library needs the CUDA toolkit to build")


def _newest_input() -> float:
    paths = [os.path.join(CSRC, f) for f in CU_SOURCES + CPP_SOURCES + HEADERS]
    paths.append(os.path.join(INCLUDE, "w12.h"))
    paths.append(os.path.abspath(__file__))
    return max(os.path.getmtime(p) for p in paths)


def _run(cmd):
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("build step failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)
    return r.stdout + r.stderr


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    """Compile (if stale) and return the path of libw12.so."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= _newest_input():
        return LIB
    nvcc = _nvcc()
    os.makedirs(BUILD, exist_ok=True)
    os.makedirs(LIBDIR, exist_ok=True)
    common = ["-std=c++17", "-O3", "-Xcompiler", "-fPIC", f"-I{INCLUDE}"]
    cmds = []
    objs = []
    for f in CU_SOURCES:
        o = os.path.join(BUILD, f + ".o")
        extra = ["-Xptxas", "-v"] if ptxas_info else []
        cmds.append([nvcc, *ARCH, "-lineinfo", *common, *extra, "-c", os.path.join(CSRC, f), "-o", o])
        objs.append(o)
    for f in CPP_SOURCES:
        o = os.path.join(BUILD, f + ".o")
        cmds.append([nvcc, *common, "-x", "c++", "-c", os.path.join(CSRC, f), "-o", o])
        objs.append(o)
    with cf.ThreadPoolExecutor(max_workers=len(cmds)) as ex:
        outs = list(ex.map(_run, cmds))
    if verbose or ptxas_info:
        for o in outs:
            if o.strip():
                print(o)
    tmp = LIB + f".tmp{os.getpid()}"
    _run([nvcc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs, "-lpthread"])
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    import sys

    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv))
