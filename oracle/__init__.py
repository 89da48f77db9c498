"""fp64 CPU oracle for exact attention (forward and backward).

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's
CPU-baseline leg may import this package; the product path (the CUDA library and
its Python binding) never does, and shares no code with it.

The arithmetic lives in ``attention_oracle.c`` (plain C, double precision, OpenMP
over rows). This module only compiles it with gcc and marshals numpy arrays
through ctypes. The definitions it follows are stated, with the passages of the
source pages they come from, in the header of ``attention_oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attention_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB) -> str:
    """Compile ``liboracle.so`` next to its source (gcc -O2 -fopenmp). ``src``/``out``
    let the tests compile a deliberately mutated copy elsewhere."""
    if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src):
        tmp = out + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c99", src, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, out)
    return out


class OracleLib:
    """ctypes view of one compiled copy of ``attention_oracle.c``."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        dp = ctypes.POINTER(ctypes.c_double)
        i = ctypes.c_int
        lib.oracle_attention_fwd.argtypes = [dp, dp, dp, dp, dp, i, i, i, i, i, i,
                                             ctypes.c_double, i, i]
        lib.oracle_attention_fwd.restype = i
        lib.oracle_attention_bwd.argtypes = [dp, dp, dp, dp, dp, dp, dp, i, i, i, i, i, i,
                                             ctypes.c_double, i, i]
        lib.oracle_attention_bwd.restype = i
        lib.oracle_num_threads.argtypes = []
        lib.oracle_num_threads.restype = i
        self.lib = lib

    def num_threads(self) -> int:
        return int(self.lib.oracle_num_threads())

    def attention_fwd(self, q, k, v, scale: float, causal: bool = False, window: int = 0):
        """Return (O [B,H,Sq,D], LSE [B,H,Sq]) in fp64."""
        q, k, v = _f64(q), _f64(k), _f64(v)
        B, H, HKV, Sq, Sk, D = _shape(q, k, v)
        o = np.empty((B, H, Sq, D), np.float64)
        lse = np.empty((B, H, Sq), np.float64)
        rc = self.lib.oracle_attention_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                           B, H, HKV, Sq, Sk, D, float(scale),
                                           int(bool(causal)), int(window))
        if rc != 0:
            raise ValueError(f"oracle_attention_fwd rejected the problem (rc={rc})")
        return o, lse

    def attention_bwd(self, q, k, v, do, scale: float, causal: bool = False, window: int = 0):
        """Return (dQ, dK, dV) in fp64 for the loss <dO, O>."""
        q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
        B, H, HKV, Sq, Sk, D = _shape(q, k, v)
        if do.shape != q.shape:
            raise ValueError("dO must have Q's shape")
        dq = np.empty_like(q)
        dk = np.empty_like(k)
        dv = np.empty_like(v)
        rc = self.lib.oracle_attention_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(do), _ptr(dq),
                                           _ptr(dk), _ptr(dv), B, H, HKV, Sq, Sk, D,
                                           float(scale), int(bool(causal)), int(window))
        if rc != 0:
            raise ValueError(f"oracle_attention_bwd rejected the problem (rc={rc})")
        return dq, dk, dv


def _load() -> OracleLib:
    global _lib
    with _lock:
        if _lib is None:
            _lib = OracleLib(build())
    return _lib


def _f64(x) -> np.ndarray:
    if hasattr(x, "detach"):  # torch tensor (any dtype, CPU) -> exact fp64 copy
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _shape(q, k, v):
    if q.ndim != 4 or k.ndim != 4 or v.ndim != 4:
        raise ValueError("oracle expects [B, heads, S, D] arrays")
    B, H, Sq, D = q.shape
    Bk, HKV, Sk, Dk = k.shape
    if (Bk, Dk) != (B, D) or v.shape != k.shape:
        raise ValueError(f"inconsistent shapes q{q.shape} k{k.shape} v{v.shape}")
    return B, H, HKV, Sq, Sk, D


def num_threads() -> int:
    """OpenMP threads the oracle uses (OMP_NUM_THREADS, else all host cores)."""
    return _load().num_threads()


def attention_fwd(q, k, v, scale: float, causal: bool = False, window: int = 0):
    """Return (O [B,H,Sq,D], LSE [B,H,Sq]) in fp64."""
    return _load().attention_fwd(q, k, v, scale, causal, window)


def attention_bwd(q, k, v, do, scale: float, causal: bool = False, window: int = 0):
    """Return (dQ, dK, dV) in fp64 for the loss <dO, O>."""
    return _load().attention_bwd(q, k, v, do, scale, causal, window)
