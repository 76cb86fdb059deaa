"""Build the CUDA library ``libfa_fwd.so`` in-tree with nvcc for sm_103a.

One translation unit, static CUDA runtime, no link-time dependency on the
driver library (the tensor-map encoder is looked up at run time).
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libfa_fwd.so")
MAIN = os.path.join(CSRC, "fa_fwd.cu")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found; the CUDA toolkit is required to build the library")


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*"))) + [os.path.join(INCLUDE, "fa.h")]


def build_cmd(extra: list[str] | None = None) -> list[str]:
    return [_nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
            "-cudart", "static", "-I", INCLUDE, "-I", CSRC, "-o", LIB, MAIN, *(extra or [])]


def needs_build() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(s) > t for s in sources())


def start_build(force: bool = False, extra: list[str] | None = None):
    """Start nvcc in the background; returns a Popen, or None when up to date."""
    if force or needs_build():
        return subprocess.Popen(build_cmd(extra))
    return None


def build(force: bool = False, extra: list[str] | None = None) -> str:
    proc = start_build(force, extra)
    if proc is not None and proc.wait() != 0:
        raise RuntimeError("nvcc failed building libfa_fwd.so")
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, extra=[a for a in sys.argv[1:] if a != "--force"]))
