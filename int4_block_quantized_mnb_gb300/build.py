"""Builds libmnb.so (the sm_103a kernels and their C ABI) in-tree with nvcc."""
from __future__ import annotations

import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
SOURCES = [os.path.join(PKG, "csrc", "mnb_gemv.cu"), os.path.join(PKG, "csrc", "mnb_cast.cu")]
INCLUDE = os.path.join(ROOT, "include")
LIBRARY = os.path.join(PKG, "libmnb.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-shared",
              "--expt-relaxed-constexpr"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libmnb.so")


def command(out: str = LIBRARY) -> list:
    return [nvcc(), *ARCH, *NVCC_FLAGS, "-I" + INCLUDE, "-o", out, *SOURCES]


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile libmnb.so unless it is newer than every source and the header."""
    deps = SOURCES + [os.path.join(INCLUDE, "mnb.h"), os.path.join(PKG, "csrc", "mnb_narrow.cuh")]
    if not force and os.path.exists(LIBRARY) and \
            all(os.path.getmtime(LIBRARY) >= os.path.getmtime(d) for d in deps):
        return LIBRARY
    tmp = LIBRARY + f".tmp{os.getpid()}"
    cmd = command(tmp)
    if verbose:
        print(" ".join(cmd))
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIBRARY)
    return LIBRARY


if __name__ == "__main__":
    print(build(force=True, verbose=True))
