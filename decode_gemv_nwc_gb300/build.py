"""Builds the in-tree library decode_gemv_nwc_gb300/_build/libnwc.so for sm_103a.

The CUDA translation unit is compiled with nvcc (-gencode arch=compute_103a,code=sm_103a)
while the host C++ units compile with g++ in parallel; nvcc links the shared library.
"""
from __future__ import annotations

import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OUT = os.path.join(PKG, "_build")
LIB = os.path.join(OUT, "libnwc.so")
INCLUDE = os.path.join(ROOT, "include")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CU = ["kernels.cu", "dequant.cu"]
CPP = ["encoder.cpp", "bind.cpp", "blobfile.cpp"]


def _sources():
    return [os.path.join(CSRC, f) for f in CU + CPP + ["nwc_format.h"]] + [os.path.join(INCLUDE, "nwc.h")]


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(s) > t for s in _sources())


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not _stale():
        return LIB
    os.makedirs(OUT, exist_ok=True)
    jobs = []
    objs = []
    for f in CU:
        o = os.path.join(OUT, f + ".o")
        objs.append(o)
        jobs.append([NVCC, *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                     "-I", INCLUDE, "-c", os.path.join(CSRC, f), "-o", o])
    for f in CPP:
        o = os.path.join(OUT, f + ".o")
        objs.append(o)
        jobs.append(["g++", "-O2", "-std=c++17", "-fPIC", "-I", INCLUDE, "-I", "/usr/local/cuda/include",
                     "-c", os.path.join(CSRC, f), "-o", o])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("build failed: " + " ".join(cmd) + "\n" + r.stdout + r.stderr)
        if verbose:
            print(r.stdout + r.stderr)

    with ThreadPoolExecutor(len(jobs)) as ex:
        list(ex.map(run, jobs))
    run([NVCC, *ARCH, "-shared", "-o", LIB + ".tmp", *objs, "-lpthread"])
    os.replace(LIB + ".tmp", LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose=True))
