"""ctypes binding of libfa.so: same entry points as include/fa.h, argument
marshalling only. Every step of the attention computation runs in the library's
CUDA kernels; there is no Python or CPU fallback -- importing the binding fails
loudly when the library is missing.

The C calls take raw device pointers and a CUDA stream handle. The helpers
``forward`` / ``backward`` allocate outputs with torch (device memory and
streams are all torch is used for) and pass ``data_ptr()``s through.
"""
from __future__ import annotations

import ctypes
import math
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libfa.so")

FA_F32, FA_BF16 = 0, 1
FA_F32_MMA_F16X2, FA_F32_MMA_TF32X3 = 0, 1
F32_MMA = {"f16x2": FA_F32_MMA_F16X2, "tf32x3": FA_F32_MMA_TF32X3}
STATUS = {0: "FA_OK", 1: "FA_ERR_INVALID_ARG", 2: "FA_ERR_UNSUPPORTED", 3: "FA_ERR_ALIGNMENT",
          4: "FA_ERR_CUDA", 5: "FA_ERR_TIMEOUT", 6: "FA_ERR_SCRATCH_LIMIT", 7: "FA_ERR_LAYOUT"}
EXPORTS = ("fa_fwd", "fa_bwd", "fa_device_status", "fa_status_string", "fa_version",
           "fa_timing_enable", "fa_timing_read", "fa_fwd_noalloc", "fa_selftest_timeout",
           "fa_noalloc_scratch_bytes", "fa_bwd_dsmat")


class FAError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {STATUS.get(code, code)} ({status_string(code)})")


class fa_params(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("H", ctypes.c_int), ("HKV", ctypes.c_int),
                ("Sq", ctypes.c_int), ("Sk", ctypes.c_int), ("D", ctypes.c_int),
                ("scale", ctypes.c_float), ("causal", ctypes.c_int), ("window", ctypes.c_int),
                ("in_dtype", ctypes.c_int), ("out_dtype", ctypes.c_int), ("f32_mma", ctypes.c_int)]


class fa_kernel_time(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char_p), ("launches", ctypes.c_int), ("total_ms", ctypes.c_double)]


def _load(path: str = LIB_PATH) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise ImportError(f"libfa.so not built at {path}: run __graft_entry__.build() first "
                          "(the attention path has no fallback)")
    lib = ctypes.CDLL(path)
    vp, st = ctypes.c_void_p, ctypes.c_int
    P = ctypes.POINTER(fa_params)
    lib.fa_fwd.argtypes = [vp, vp, vp, vp, vp, P, vp]
    lib.fa_fwd.restype = st
    lib.fa_fwd_noalloc.argtypes = [vp, vp, vp, vp, vp, P, vp]
    lib.fa_fwd_noalloc.restype = st
    lib.fa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, P, vp]
    lib.fa_bwd.restype = st
    lib.fa_bwd_dsmat.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, P, vp]
    lib.fa_bwd_dsmat.restype = st
    lib.fa_device_status.argtypes = [vp]
    lib.fa_device_status.restype = st
    lib.fa_status_string.argtypes = [st]
    lib.fa_status_string.restype = ctypes.c_char_p
    lib.fa_version.argtypes = []
    lib.fa_version.restype = ctypes.c_char_p
    lib.fa_noalloc_scratch_bytes.argtypes = []
    lib.fa_noalloc_scratch_bytes.restype = ctypes.c_ulonglong
    lib.fa_selftest_timeout.argtypes = [ctypes.c_ulonglong, vp, vp]
    lib.fa_selftest_timeout.restype = st
    lib.fa_timing_enable.argtypes = [st]
    lib.fa_timing_enable.restype = st
    lib.fa_timing_read.argtypes = [ctypes.POINTER(fa_kernel_time), st]
    lib.fa_timing_read.restype = st
    return lib


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        _lib = _load()
    return _lib


def status_string(code: int) -> str:
    return lib().fa_status_string(int(code)).decode()


def version() -> str:
    return lib().fa_version().decode()


def noalloc_scratch_bytes() -> int:
    """Size of the static device scratch behind ``fa_fwd_noalloc``, as compiled into
    the loaded library (FA_NOALLOC_SCRATCH_BYTES)."""
    return int(lib().fa_noalloc_scratch_bytes())


# ------------------------------------------------------------ raw C entry points
def fa_fwd(Q: int, K: int, V: int, O: int, LSE: int, params: fa_params, stream: int) -> int:
    """Direct call of the C ``fa_fwd`` with integer device addresses; returns the status."""
    return lib().fa_fwd(Q, K, V, O, LSE, ctypes.byref(params), stream)


def fa_fwd_noalloc(Q: int, K: int, V: int, O: int, LSE: int, params: fa_params,
                   stream: int) -> int:
    """Direct call of the C ``fa_fwd_noalloc`` (same contract as ``fa_fwd``, but its
    scratch is the library's static device array, so it never allocates)."""
    return lib().fa_fwd_noalloc(Q, K, V, O, LSE, ctypes.byref(params), stream)


def fa_bwd(Q: int, K: int, V: int, O: int, dO: int, LSE: int, dQ: int, dK: int, dV: int,
           params: fa_params, stream: int) -> int:
    """Direct call of the C ``fa_bwd``; returns the status."""
    return lib().fa_bwd(Q, K, V, O, dO, LSE, dQ, dK, dV, ctypes.byref(params), stream)


def fa_bwd_dsmat(Q: int, K: int, V: int, O: int, dO: int, LSE: int, dQ: int, dK: int, dV: int,
                 params: fa_params, stream: int) -> int:
    """Direct call of the C ``fa_bwd_dsmat`` (the materialised-dS backward); returns the status."""
    return lib().fa_bwd_dsmat(Q, K, V, O, dO, LSE, dQ, dK, dV, ctypes.byref(params), stream)


def fa_device_status(stream: int) -> int:
    return lib().fa_device_status(stream)


def fa_selftest_timeout(limit_ns: int, roles_done: int, stream: int) -> int:
    """Enqueue the barrier-timeout self test (see include/fa.h)."""
    return lib().fa_selftest_timeout(int(limit_ns), roles_done, stream)


def fa_timing_enable(on: bool) -> int:
    return lib().fa_timing_enable(int(bool(on)))


def fa_timing_read() -> dict:
    """{kernel name: (launches, total_ms)} for the launches recorded since the last read."""
    buf = (fa_kernel_time * 64)()
    n = lib().fa_timing_read(buf, 64)
    if n < 0:
        raise FAError(4, "fa_timing_read")
    return {buf[i].name.decode(): (buf[i].launches, buf[i].total_ms) for i in range(min(n, 64))}


# ------------------------------------------------------------ torch helpers
def make_params(q, k, scale=None, causal=False, window=0, out_dtype=None,
                f32_mma="f16x2") -> fa_params:
    import torch
    B, H, Sq, D = q.shape
    HKV, Sk = k.shape[1], k.shape[2]
    in_dt = {torch.float32: FA_F32, torch.bfloat16: FA_BF16}.get(q.dtype)
    if in_dt is None:
        raise TypeError(f"unsupported input dtype {q.dtype}")
    out_dt = FA_F32 if out_dtype in (None, torch.float32) else FA_BF16
    if f32_mma not in F32_MMA:
        raise ValueError(f"f32_mma must be one of {sorted(F32_MMA)}")
    return fa_params(B, H, HKV, Sq, Sk, D, float(1.0 / math.sqrt(D) if scale is None else scale),
                     int(bool(causal)), int(window), in_dt, out_dt, F32_MMA[f32_mma])


def _check(t, name):
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor")


def _stream_handle(stream) -> int:
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return int(s.cuda_stream)


def forward(q, k, v, scale=None, causal=False, window=0, out_dtype=None, stream=None,
            f32_mma="f16x2"):
    """O, LSE = attention(q, k, v) on the GPU through ``fa_fwd``. ``f32_mma`` (fp32
    inputs): "f16x2" (two scaled fp16 terms per operand) or "tf32x3" (D <= 64)."""
    import torch
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check(t, n)
    p = make_params(q, k, scale, causal, window, out_dtype, f32_mma)
    o = torch.empty(q.shape, dtype=torch.float32 if p.out_dtype == FA_F32 else torch.bfloat16,
                    device=q.device)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device)
    rc = fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), p,
                _stream_handle(stream))
    if rc:
        raise FAError(rc, "fa_fwd")
    return o, lse


def backward(q, k, v, o, lse, do, scale=None, causal=False, window=0, out_dtype=None,
             stream=None, materialize_ds=False, f32_mma="f16x2"):
    """dQ, dK, dV through ``fa_bwd`` (o / lse as returned by ``forward``), or through
    ``fa_bwd_dsmat`` with ``materialize_ds``."""
    import torch
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o"), (lse, "lse"), (do, "do")):
        _check(t, n)
    p = make_params(q, k, scale, causal, window, out_dtype, f32_mma)
    odt = torch.float32 if p.out_dtype == FA_F32 else torch.bfloat16
    dq = torch.empty(q.shape, dtype=odt, device=q.device)
    dk = torch.empty(k.shape, dtype=odt, device=q.device)
    dv = torch.empty(v.shape, dtype=odt, device=q.device)
    entry = fa_bwd_dsmat if materialize_ds else fa_bwd
    rc = entry(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(),
               lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), p,
               _stream_handle(stream))
    if rc:
        raise FAError(rc, "fa_bwd_dsmat" if materialize_ds else "fa_bwd")
    return dq, dk, dv


def check_device_status(stream=None) -> None:
    """Synchronize and raise FAError if a kernel reported a barrier timeout."""
    rc = fa_device_status(_stream_handle(stream))
    if rc:
        raise FAError(rc, "fa_device_status")
