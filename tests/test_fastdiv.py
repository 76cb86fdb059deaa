"""The kernels' division by launch-constant divisors (fa_fastdiv.h) agrees with
exact integer division: compiled with the host C++ compiler and run over small
divisors exhaustively and random 31-bit numerators and divisors."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "unet_fa_fwd_gb300", "csrc")


def test_fastdiv_matches_integer_division(tmp_path):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    exe = tmp_path / "fastdiv_check"
    subprocess.run([cxx, "-O2", "-std=c++17", "-I", CSRC, "-o", str(exe),
                    os.path.join(HERE, "fastdiv_check.cpp")], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stdout + out.stderr
    assert out.stdout.strip() == "ok"
