"""Compile libkda.so in-tree with nvcc for sm_103a.

One translation unit per .cu file, compiled in parallel, then linked into a
shared library with the CUDA runtime linked statically (the library needs no
libcuda at load time; driver entry points are looked up at run time).
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libkda.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libkda.so")
    return path


def _compile(src: str, extra: list, build_dir: str = BUILD) -> str:
    obj = os.path.join(build_dir, os.path.basename(src) + ".o")
    cmd = [nvcc(), *ARCH, "-std=c++17", "-O3", "-lineinfo", "-Xcompiler", "-fPIC",
           "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC, *extra, "-c", src, "-o", obj]
    subprocess.run(cmd, check=True)
    return obj


# The phase-stamp variant: kernels record clock64 stamps per chunk of CTA 0 into the end of
# the workspace (KDA_PHASE_STAMPS); a separate library, never the one the package loads.
STAMPS_LIB = os.path.join(PKG, "libkda_stamps.so")


def build(force: bool = False, verbose_ptxas: bool = False, stamps: bool = False) -> str:
    """Build (if stale) and return the path of libkda.so (or of the stamps variant)."""
    lib = STAMPS_LIB if stamps else LIB
    bdir = BUILD + ("_stamps" if stamps else "")
    os.makedirs(bdir, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    deps = srcs + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h"))
    if not force and os.path.exists(lib):
        if os.path.getmtime(lib) >= max(os.path.getmtime(d) for d in deps):
            return lib
    extra = ["-Xptxas", "-v"] if verbose_ptxas else []
    if stamps:
        extra = extra + ["-DKDA_PHASE_STAMPS"]
    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        objs = list(ex.map(lambda s: _compile(s, extra, bdir), srcs))
    tmp = lib + f".tmp{os.getpid()}"
    subprocess.run([nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs], check=True)
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    import sys
    print(build(force=True, verbose_ptxas="-v" in sys.argv))
