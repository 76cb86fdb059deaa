"""Build the CUDA libraries in-tree with nvcc for sm_103a.

``libfa_fwd.so`` (release) and ``libfa_fwd_debug.so`` (the same sources with
``-DFA_DEBUG``: device-side bounds and schedule checks that record a violation
instead of making the access).  Each is four translation units (the C ABI and
helper kernels in ``fa_fwd.cu``, the attention kernel's instantiations per head
dimension in ``fa_attn_d32.cu`` / ``fa_attn_d64.cu`` / ``fa_attn_d128.cu``);
all eight objects are compiled in parallel, then each library is linked with
the static CUDA runtime.  There is no link-time dependency on the driver
library (the tensor-map encoder is looked up at run time).
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
LIB_DEBUG = os.path.join(PKG, "libfa_fwd_debug.so")
OBJ_DIR = os.path.join(PKG, "_build")
UNITS = ["fa_fwd.cu", "fa_attn_d32.cu", "fa_attn_d64.cu", "fa_attn_d128.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found; the CUDA toolkit is required to build the library")


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*"))) + [os.path.join(INCLUDE, "fa.h")]


def _obj(unit: str, debug: bool) -> str:
    return os.path.join(OBJ_DIR, ("debug_" if debug else "") + unit.replace(".cu", ".o"))


def compile_cmd(unit: str, debug: bool = False, extra: list[str] | None = None) -> list[str]:
    # Host symbols are hidden except the C ABI (FA_API in fa.h), so two builds of
    # the library (release and debug) can share a process without interposing
    # each other's template instantiations.
    return [_nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
            "-Xcompiler", "-fvisibility=hidden", "-I", INCLUDE,
            "-I", CSRC, *(["-DFA_DEBUG"] if debug else []), "-c", "-o", _obj(unit, debug),
            os.path.join(CSRC, unit), *(extra or [])]


def link_cmd(debug: bool = False) -> list[str]:
    return [_nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", LIB_DEBUG if debug else LIB,
            *(_obj(u, debug) for u in UNITS)]


def needs_build() -> bool:
    for lib in (LIB, LIB_DEBUG):
        if not os.path.exists(lib):
            return True
        t = os.path.getmtime(lib)
        if any(os.path.getmtime(s) > t for s in sources()):
            return True
    return False


def _compile_and_link(extra: list[str] | None = None) -> int:
    os.makedirs(OBJ_DIR, exist_ok=True)
    jobs = [(u, d) for d in (False, True) for u in UNITS]
    procs = [(u, d, subprocess.Popen(compile_cmd(u, d, extra))) for u, d in jobs]
    failed = [(u, d) for u, d, p in procs if p.wait() != 0]
    if failed:
        print(f"nvcc failed: {failed}", file=sys.stderr)
        return 1
    return subprocess.call(link_cmd(False)) or subprocess.call(link_cmd(True))


def start_build(force: bool = False, extra: list[str] | None = None):
    """Start the build in the background (a child process that compiles the
    units of both libraries in parallel and links them); returns its Popen, or
    None when up to date."""
    if force or needs_build():
        return subprocess.Popen([sys.executable, os.path.abspath(__file__), "--force", *(extra or [])])
    return None


def build(force: bool = False, extra: list[str] | None = None) -> str:
    proc = start_build(force, extra)
    if proc is not None and proc.wait() != 0:
        raise RuntimeError("nvcc failed building libfa_fwd.so")
    return LIB


if __name__ == "__main__":
    args = [a for a in sys.argv[1:] if a != "--force"]
    if "--force" in sys.argv or needs_build():
        sys.exit(_compile_and_link(args))
    print(LIB)
