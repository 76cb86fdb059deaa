"""The window map of the attention kernel's window mode (multiply-shift division, fa_window_geom.h)
agrees with its division-by-division definition: compiled with the host C++
compiler and run over every row of a set of window geometries, packs and shifts."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "unet_fa_fwd_gb300", "csrc")


def test_window_index_map_matches_definition(tmp_path):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    exe = tmp_path / "window_index_check"
    subprocess.run([cxx, "-O2", "-std=c++17", "-I", CSRC, "-o", str(exe),
                    os.path.join(HERE, "window_index_check.cpp")], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stdout + out.stderr
    assert out.stdout.strip() == "ok"
