"""Build libentropack.so in-tree for B300 (sm_103a).

    python -m dit_weight_compression_02_b300.build [--force]

CUDA sources are compiled with nvcc for ``-gencode arch=compute_103a,code=sm_103a``
(``-lineinfo`` for profiling); the host encoder and validator with g++ and
``-ffp-contract=off`` (the stream format fixes the floating-point operation
order of the encoder, so no multiply-add may be fused).  The CUDA runtime is
linked statically so the library does not depend on which libcudart the
calling process (e.g. PyTorch) loaded.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT = os.path.join(PKG, "libentropack.so")
BUILD_DIR = os.path.join(ROOT, "_build")

CU_SOURCES = ["ep_decode.cu", "ep_linear.cu", "ep_fused.cu", "ep_q4.cu"]
CXX_SOURCES = ["ep_host.cpp", "ep_encode.cpp", "ep_q4.cpp"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libentropack.so")


def _sources():
    files = [os.path.join(CSRC, f) for f in CU_SOURCES + CXX_SOURCES]
    files += [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".hpp", ".cuh", ".h"))]
    files.append(os.path.join(INCLUDE, "entropack.h"))
    return files


def needs_build() -> bool:
    if not os.path.exists(OUT):
        return True
    t = os.path.getmtime(OUT)
    return any(os.path.getmtime(f) > t for f in _sources())


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not needs_build():
        return OUT
    nvcc = _nvcc()
    os.makedirs(BUILD_DIR, exist_ok=True)
    objs = []
    inc = ["-I", INCLUDE, "-I", CSRC]
    for f in CU_SOURCES:
        o = os.path.join(BUILD_DIR, f + ".o")
        cmd = [nvcc, *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xptxas", "-v" if verbose else "-O3",
               *inc, "-c", os.path.join(CSRC, f), "-o", o]
        subprocess.check_call(cmd)
        objs.append(o)
    for f in CXX_SOURCES:
        o = os.path.join(BUILD_DIR, f + ".o")
        cmd = ["g++", "-O3", "-std=c++17", "-fPIC", "-ffp-contract=off", "-pthread", "-Wall", *inc,
               "-I", "/usr/local/cuda/include", "-c", os.path.join(CSRC, f), "-o", o]
        subprocess.check_call(cmd)
        objs.append(o)
    tmp = OUT + f".tmp{os.getpid()}"
    subprocess.check_call([nvcc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs, "-lpthread"])
    os.replace(tmp, OUT)
    return OUT


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
