"""CPU replay of the GEMV weight-ring layout.

Builds tests/ring_layout_check.cpp against the kernels' own addressing
(transformer_layer_gb300/csrc/ring_layout.h) and runs it: every fragment load
reads the (row, byte) the MMA needs from where the swizzled TMA tensor copy
put it, and no 128-bit load has a shared-memory bank conflict.
"""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_ring_layout_replay(tmp_path):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    exe = str(tmp_path / "ring_layout_check")
    subprocess.run([cxx, "-std=c++17", "-O2", "-I", os.path.join(ROOT, "transformer_layer_gb300", "csrc"),
                    os.path.join(ROOT, "tests", "ring_layout_check.cpp"), "-o", exe], check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr
