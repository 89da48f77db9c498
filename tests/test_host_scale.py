"""Exponent rules of the bf16 path's power-of-two operand scaling, checked
exhaustively on the CPU.

tests/host_scale_check.cpp includes the library's csrc/fa_scale.cuh: for every
non-negative bf16 magnitude as a tensor's largest element it checks that the fp16
copy's exponent keeps that element finite in fp16 (and puts it in [2^14, 2^15) when
it rescales at all), and over a grid of largest |dO|, |V|, |delta| and head dims that
the dS exponent keeps the worst-case |dS| below 2^15.
"""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _cuda_include():
    for cand in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if cand and os.path.exists(os.path.join(cand, "include", "cuda.h")):
            return os.path.join(cand, "include")
    return None


def test_scale_exponent_rules(tmp_path):
    cxx, inc = shutil.which("g++"), _cuda_include()
    if cxx is None or inc is None:
        pytest.skip("needs g++ and the CUDA headers")
    exe = tmp_path / "host_scale_check"
    src = os.path.join(ROOT, "tests", "host_scale_check.cpp")
    r = subprocess.run([cxx, "-std=c++17", "-O2", "-I", inc, "-I", os.path.join(ROOT, "include"),
                        "-I", os.path.join(ROOT, "attention_fa_fwd_02_gb300", "csrc"), src,
                        "-o", str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-3000:]
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=600)
    assert out.returncode == 0 and out.stdout.startswith("ok"), out.stdout + out.stderr
