"""Builds the in-tree CUDA library ``libmp_layout.so`` for sm_103a.

The three translation units are compiled in parallel with nvcc and linked
into a shared library next to this file (no torch extension machinery, no
cmake).  Intermediate objects go to ``_build/`` at the repository root.
"""
from __future__ import annotations

import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libmp_layout.so")
UNITS = ["mp_abi", "mp_layout_kernels", "mp_copy_kernels", "mp_noalloc"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xptxas", "-v"]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libmp_layout.so")


def _sources():
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    deps.append(os.path.join(ROOT, "include", "mp_layout.h"))
    return deps


def stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(d) > t for d in _sources())


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not stale():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()
    procs = []
    for u in UNITS:
        obj = os.path.join(BUILD, u + ".o")
        log = open(os.path.join(BUILD, u + ".log"), "w")
        cmd = [cc, *ARCH, *NVCC_FLAGS, "-c", os.path.join(CSRC, u + ".cu"), "-o", obj]
        procs.append((u, subprocess.Popen(cmd, stdout=log, stderr=subprocess.STDOUT), log))
    failed = []
    for u, p, log in procs:
        if p.wait() != 0:
            failed.append(u)
        log.close()
    if failed:
        msgs = "".join(open(os.path.join(BUILD, u + ".log")).read() for u in failed)
        raise RuntimeError("nvcc failed for %s:\n%s" % (failed, msgs))
    tmp = LIB + ".tmp%d" % os.getpid()
    subprocess.check_call([cc, *ARCH, "-shared", "-o", tmp,
                           *[os.path.join(BUILD, u + ".o") for u in UNITS], "-lcudart"])
    os.replace(tmp, LIB)
    if verbose:
        for u in UNITS:
            print(open(os.path.join(BUILD, u + ".log")).read())
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose=True))
