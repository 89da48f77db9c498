"""Host-side tiling arithmetic of the library, checked by brute force on the CPU.

tests/host_tiling_check.cpp includes the library's csrc/fa_common.cuh and compares
its tile-range functions, the interior-tile (no mask) test, the key-range count of
short query sequences and the dQ range-sum formula against exhaustive enumeration
of the visible (query, key) pairs on small shapes (causal / windowed / ragged).
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


def test_tiling_arithmetic_matches_brute_force(tmp_path):
    cxx, inc = shutil.which("g++"), _cuda_include()
    if cxx is None or inc is None:
        pytest.skip("needs g++ and the CUDA headers")
    exe = tmp_path / "host_tiling_check"
    src = os.path.join(ROOT, "tests", "host_tiling_check.cpp")
    r = subprocess.run([cxx, "-std=c++17", "-O2", "-I", inc, "-I", os.path.join(ROOT, "include"),
                        "-I", os.path.join(ROOT, "attention_fa_fwd_02_gb300", "csrc"), src,
                        "-o", str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-3000:]
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=600)
    assert out.returncode == 0 and out.stdout.startswith("ok"), out.stdout + out.stderr
