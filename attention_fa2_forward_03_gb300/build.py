"""Builds the CUDA library in-tree with nvcc (sm_103a only).

    python -m attention_fa2_forward_03_gb300.build
"""
from __future__ import annotations

import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libfa2.so")
# The same sources with FA2_DEBUG: device-side bounds checks that report
# FA2_ERR_BOUNDS instead of touching memory outside the planned extents.
DEBUG_LIB = os.path.join(PKG, "libfa2_debug.so")
SOURCES = [os.path.join(CSRC, "fa2_fwd_sm103.cu")]
DEPENDS = SOURCES + [os.path.join(CSRC, "ptx_sm103.cuh"), os.path.join(CSRC, "fa2_fwd_sm103.cuh"), os.path.join(CSRC, "fa2_bwd_sm103.cuh"), os.path.join(CSRC, "fa2_fwd_fp8_sm103.cuh"),
                     os.path.join(CSRC, "fa2_fwd_d64_sm103.cuh"),
                     os.path.join(INCLUDE, "fa2.h")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def needs_build(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(f) > t for f in DEPENDS)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile libfa2.so and libfa2_debug.so next to this file (in parallel)
    if they are missing or stale; returns the release library's path."""
    jobs = []
    for lib, extra in ((LIB, []), (DEBUG_LIB, ["-DFA2_DEBUG"])):
        if not force and not needs_build(lib):
            continue
        tmp = lib + f".tmp{os.getpid()}"
        cmd = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
               *extra, "-I", INCLUDE, "-o", tmp, *SOURCES]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        jobs.append((subprocess.Popen(cmd), tmp, lib, cmd))
    for proc, tmp, lib, cmd in jobs:
        if proc.wait() != 0:
            raise subprocess.CalledProcessError(proc.returncode, cmd)
        os.replace(tmp, lib)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
