"""Compile the CPU oracle (``fa_oracle.c``) into ``oracle/liboracle.so`` with gcc.

Test infrastructure: building the checker is not using it.  Plain ``-O2``
without fast-math or FMA contraction, so the fp64 arithmetic is the one the
source spells out.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "fa_oracle.c")
LIB = os.path.join(HERE, "liboracle.so")


def build_cmd() -> list[str]:
    cc = os.environ.get("CC", "gcc")
    return [cc, "-O2", "-fPIC", "-shared", "-pthread", "-ffp-contract=off", "-fno-fast-math",
            "-std=c11", "-Wall", "-Wextra", "-o", LIB, SRC, "-lm"]


def needs_build() -> bool:
    return not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC)


def build(force: bool = False) -> str:
    if force or needs_build():
        subprocess.run(build_cmd(), check=True)
    return LIB


def start_build(force: bool = False):
    """Start the compile in the background; returns a Popen or None if up to date."""
    if force or needs_build():
        return subprocess.Popen(build_cmd())
    return None


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
