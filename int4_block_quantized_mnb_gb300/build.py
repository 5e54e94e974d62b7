"""Builds libmnb.so (the sm_103a kernels and their C ABI) in-tree with nvcc."""
from __future__ import annotations

import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
SOURCES = [os.path.join(PKG, "csrc", "mnb_gemv.cu"), os.path.join(PKG, "csrc", "mnb_general.cu"),
           os.path.join(PKG, "csrc", "mnb_prefill.cu"), os.path.join(PKG, "csrc", "mnb_prefill_tc.cu"),
           os.path.join(PKG, "csrc", "mnb_cast.cu")]
INCLUDE = os.path.join(ROOT, "include")
LIBRARY = os.path.join(PKG, "libmnb.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr"]
OBJDIR = os.path.join(PKG, "_build")


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libmnb.so")


def compile_command(src: str, obj: str) -> list:
    csrc = os.path.join(PKG, "csrc")
    return [nvcc(), *ARCH, *NVCC_FLAGS, "-I" + INCLUDE, "-I" + csrc, "-c", "-o", obj, src]


def link_command(objs: list, out: str) -> list:
    return [nvcc(), *ARCH, "-shared", "-o", out, *objs]


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile libmnb.so unless it is newer than every source and header; the
    translation units compile in parallel, then link."""
    csrc = os.path.join(PKG, "csrc")
    deps = SOURCES + [os.path.join(INCLUDE, "mnb.h")] + \
        [os.path.join(csrc, f) for f in sorted(os.listdir(csrc)) if f.endswith(".cuh")]
    if not force and os.path.exists(LIBRARY) and \
            all(os.path.getmtime(LIBRARY) >= os.path.getmtime(d) for d in deps):
        return LIBRARY
    os.makedirs(OBJDIR, exist_ok=True)
    tag = f"{os.getpid()}"
    objs = [os.path.join(OBJDIR, os.path.basename(src) + f".{tag}.o") for src in SOURCES]
    procs = []
    for src, obj in zip(SOURCES, objs):
        cmd = compile_command(src, obj)
        if verbose:
            print(" ".join(cmd))
        procs.append((cmd, subprocess.Popen(cmd)))
    failed = [cmd for cmd, pr in procs if pr.wait() != 0]
    if failed:
        raise subprocess.CalledProcessError(1, failed[0])
    tmp = LIBRARY + f".tmp{tag}"
    cmd = link_command(objs, tmp)
    if verbose:
        print(" ".join(cmd))
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIBRARY)
    for obj in objs:
        os.remove(obj)
    return LIBRARY


if __name__ == "__main__":
    print(build(force=True, verbose=True))
