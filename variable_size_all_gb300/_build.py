"""Compile the CUDA library ``liba2av.so`` in-tree for sm_103a with nvcc."""
from __future__ import annotations

import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
SOURCES = [os.path.join(PKG, "csrc", "a2av.cu"), os.path.join(PKG, "csrc", "dispatch.cu")]
HEADERS = [os.path.join(PKG, "csrc", "a2av_device.cuh"), os.path.join(PKG, "csrc", "a2av_handle.h")]
INCLUDE = os.path.join(ROOT, "include")
LIBRARY = os.path.join(PKG, "liba2av.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the a2av library needs the CUDA toolkit to build")


def command(output: str = LIBRARY, extra=()) -> list:
    return [nvcc(), *ARCH, "-lineinfo", "-O3", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
            "-shared", "-I", INCLUDE, *extra, "-o", output, *SOURCES]


def stale(output: str = LIBRARY) -> bool:
    if not os.path.exists(output):
        return True
    deps = SOURCES + HEADERS + [os.path.join(INCLUDE, "a2av.h"), __file__]
    return os.path.getmtime(output) < max(os.path.getmtime(d) for d in deps)


def build(force: bool = False, verbose: bool = False, extra=()) -> str:
    """Build ``liba2av.so`` unless it is up to date; returns its path."""
    if force or stale():
        cmd = command(extra=extra)
        if verbose:
            print(" ".join(cmd))
        tmp = LIBRARY + ".tmp"
        subprocess.run(cmd[:-len(SOURCES) - 2] + ["-o", tmp, *SOURCES, "--threads", "0"],
                       check=True)
        os.replace(tmp, LIBRARY)
    return LIBRARY


if __name__ == "__main__":
    build(force=True, verbose=True, extra=["-Xptxas", "-v"])
