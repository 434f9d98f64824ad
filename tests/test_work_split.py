"""CPU replay of the skinny-GEMM work split that the region kernels use.

Builds tests/work_split_check.cpp against the kernels' own split functions
(transformer_layer_gb300/csrc/work_split.h) with the host compiler and runs it:
every chunk processed once, streaming and epilogue warps agreeing on the
segments, split-K contributions matching each tile's arrival target.
"""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_work_split_replay(tmp_path):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    cuda_inc = "/usr/local/cuda/include"
    exe = str(tmp_path / "work_split_check")
    subprocess.run([cxx, "-std=c++17", "-O2", "-I", cuda_inc, "-I", os.path.join(ROOT, "include"), "-I",
                    os.path.join(ROOT, "transformer_layer_gb300", "csrc"),
                    os.path.join(ROOT, "tests", "work_split_check.cpp"), "-o", exe], check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr
