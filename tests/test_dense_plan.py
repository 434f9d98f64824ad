"""CPU replay of the tile GEMMs' work plan.

Builds tests/dense_plan_check.cpp against the planner the library uses
(transformer_layer_gb300/csrc/dense_plan.h) with the host compiler and sweeps
decode and prompt-chunk shapes (fp16, bf16, int8; 132-152 SMs): token tiles
covering the rows, ring stages within shared memory with one tile CTA per SM,
tensor-memory columns within 512, an even ring with two fp16 / bf16 MMA
issuers, and cluster K slices covering the K chunks exactly once.
"""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_dense_plan_invariants(tmp_path):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    exe = str(tmp_path / "dense_plan_check")
    subprocess.run([cxx, "-std=c++17", "-O2", "-I", "/usr/local/cuda/include", "-I", os.path.join(ROOT, "include"),
                    "-I", os.path.join(ROOT, "transformer_layer_gb300", "csrc"),
                    os.path.join(ROOT, "tests", "dense_plan_check.cpp"), "-o", exe], check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr
