"""GPU parity of the 3xTF32 kernels (fa_params.f32_mma = FA_F32_MMA_TF32X3) against
the fp64 oracle.

fp32 inputs run by default as two scaled fp16 terms per operand; the other choice,
hi / lo tf32 splits on kind::tf32, serves head dims up to 64 and is held to the same
fp32 bounds (O <= 2e-3 and gradients <= 5e-3 of the oracle tensor's RMS, LSE <= 1e-3
absolute): every fp32 case of the forward / backward parity sets with D <= 64, and
the full fp32 workloads C1, C2, C5.
"""
import pytest
import torch

import oracle
from attention_fa_fwd_02_gb300.workloads import WORKLOADS, make_inputs
from _parity import TOL, lse_err, rms_err, to_np
from test_parity_fwd import SMALL

pytestmark = pytest.mark.gpu

CASES = [n for n, w in SMALL.items() if w.dtype == "f32" and w.D <= 64]


@pytest.fixture(scope="module")
def fa():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU parity tests need a CUDA device"
    from attention_fa_fwd_02_gb300 import fa as m
    return m


def _run(fa, w):
    q, k, v, do = make_inputs(w)
    dev = torch.device("cuda:0")
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    o, lse = fa.forward(qd, kd, vd, w.scale, w.causal, w.window, f32_mma="tf32x3")
    grads = fa.backward(qd, kd, vd, o, lse, dod, w.scale, w.causal, w.window, f32_mma="tf32x3")
    fa.check_device_status()
    return (q, k, v, do), (o, lse), grads


def _check(w, ins, fwd, grads, label):
    tol = TOL[w.dtype]
    ro, rl = oracle.attention_fwd(*ins[:3], w.scale, w.causal, w.window)
    ref = oracle.attention_bwd(*ins, w.scale, w.causal, w.window)
    errs = {"O": rms_err(to_np(fwd[0]), ro), "LSE": lse_err(to_np(fwd[1]), rl)}
    errs.update({n: rms_err(to_np(g), r) for n, g, r in zip(("dQ", "dK", "dV"), grads, ref)})
    lim = {"O": tol["O"], "LSE": tol["LSE"], "dQ": tol["grad"], "dK": tol["grad"], "dV": tol["grad"]}
    bad = {k: e for k, e in errs.items() if not e <= lim[k]}
    assert not bad, f"{label}: {errs}"


def test_cases_cover_the_fp32_parity_set():
    assert len(CASES) >= 10


@pytest.mark.parametrize("name", CASES)
def test_tf32x3_small(fa, name):
    w = SMALL[name]
    ins, fwd, grads = _run(fa, w)
    _check(w, ins, fwd, grads, name)


@pytest.mark.parametrize("cfg", ["c1", "c2", "c5"])
def test_tf32x3_full_config(fa, cfg):
    w = WORKLOADS[cfg]
    ins, fwd, grads = _run(fa, w)
    _check(w, ins, fwd, grads, cfg)


def test_tf32x3_rejects_head_dims_above_64(fa):
    q = torch.zeros(1, 1, 128, 80, device="cuda")
    with pytest.raises(fa.FAError):
        fa.forward(q, q, q, f32_mma="tf32x3")
