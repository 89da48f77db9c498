"""GPU parity of the backward pass (fa_bwd through the C ABI) against the fp64 oracle.

The GPU path takes O and LSE from its own forward pass, exactly as a caller
would; the oracle derives dQ / dK / dV from Q, K, V, dO alone through the softmax
Jacobian. Tolerances (max-abs error / RMS of the oracle tensor): 5e-3 for fp32
inputs (3xTF32 path), 2e-2 for bf16 inputs.
"""
import numpy as np
import pytest
import torch

import oracle
from attention_fa_fwd_02_gb300.workloads import WORKLOADS, make_inputs
from _parity import TOL, rms_err, to_np
from test_parity_fwd import SMALL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU parity tests need a CUDA device"
    from attention_fa_fwd_02_gb300 import fa as m
    return m


def _gpu_grads(fa, w, q, k, v, do, out_dtype=None):
    dev = torch.device("cuda:0")
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    o, lse = fa.forward(qd, kd, vd, w.scale, w.causal, w.window, out_dtype=out_dtype)
    dq, dk, dv = fa.backward(qd, kd, vd, o, lse, dod, w.scale, w.causal, w.window,
                             out_dtype=out_dtype)
    fa.check_device_status()
    return dq, dk, dv


def _check(w, got, ref, label):
    tol = TOL[w.dtype]["grad"]
    errs = {}
    for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
        errs[name] = rms_err(to_np(g), r)
    bad = {k: e for k, e in errs.items() if not e <= tol}
    assert not bad, f"{label}: {errs} (tol {tol})"
    return errs


# Rows that put almost all their weight on a few of many keys: 128 queries against
# 16384 keys with Q, K ~ N(0, 1.5^2), where max|dV| is ~80x RMS(dV). The fp16 operands
# of the accumulating products (P for dV += P^T dO, dS for dK += dS^T Q; relative
# rounding 2^-11, absolute 2^-25 below 2^-14) then put an error of about 2e-2 of the
# RMS on those few large entries by themselves: rounding exact P and dS to fp16 and
# nothing else gives dV 0.023, dK 0.017 in fp64. For these cases dK / dV get that
# rounding bound elementwise on top of the tolerance,
#   |g - r| <= 2^-11 sum_i max(|X_ij|, 2^-14) |Y_i| + tol RMS(r),
# X = P, Y = dO for dV and X = dS, Y = Q (times scale) for dK; dQ keeps the plain test.
FP16_OPERAND_BOUND = {"bf16-decode-sq128-sk16384"}


def _fp16_operand_bounds(w, q, k, v, do):
    """Elementwise fp16-operand rounding bounds for dK and dV (full attention only),
    from P and dS computed in fp64 from the inputs."""
    assert not w.causal and w.window == 0
    qn, kn, vn, don = (t.double().numpy() for t in (q, k, v, do))
    rep = w.H // w.HKV
    bk, bv = np.zeros_like(kn), np.zeros_like(vn)
    tiny = 2.0 ** -14
    for b in range(w.B):
        for h in range(w.H):
            g = h // rep
            s = w.scale * qn[b, h] @ kn[b, g].T
            p = np.exp(s - s.max(axis=1, keepdims=True))
            p /= p.sum(axis=1, keepdims=True)
            o = p @ vn[b, g]
            ds = p * (don[b, h] @ vn[b, g].T - (don[b, h] * o).sum(axis=1, keepdims=True))
            bv[b, g] += np.maximum(p, tiny).T @ np.abs(don[b, h])
            bk[b, g] += w.scale * (np.maximum(np.abs(ds), tiny).T @ np.abs(qn[b, h]))
    return 2.0 ** -11 * bk, 2.0 ** -11 * bv


@pytest.mark.parametrize("name", list(SMALL))
def test_backward_small(fa, name):
    w = SMALL[name]
    q, k, v, do = make_inputs(w)
    got = _gpu_grads(fa, w, q, k, v, do)
    ref = oracle.attention_bwd(q, k, v, do, w.scale, w.causal, w.window)
    if name not in FP16_OPERAND_BOUND:
        _check(w, got, ref, name)
        return
    tol = TOL[w.dtype]["grad"]
    assert rms_err(to_np(got[0]), ref[0]) <= tol, f"{name}: dQ"
    bk, bv = _fp16_operand_bounds(w, q, k, v, do)
    for n, g, r, bound in (("dK", got[1], ref[1], bk), ("dV", got[2], ref[2], bv)):
        excess = np.abs(to_np(g) - r) - bound
        assert excess.max() <= tol * np.sqrt(np.mean(r ** 2)), f"{name}: {n}"


@pytest.mark.parametrize("name", ["bf16-gqa-causal-ragged", "bf16-decode-gqa"])
def test_backward_deterministic(fa, name):
    # dK / dV are accumulated per key tile without atomics, dQ per query tile (or per
    # key range, the ranges then summed in order): bit-identical reruns.
    w = SMALL[name]
    q, k, v, do = make_inputs(w)
    a = _gpu_grads(fa, w, q, k, v, do)
    b = _gpu_grads(fa, w, q, k, v, do)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_backward_unseen_keys_get_zero_grad(fa):
    # causal with Sq < Sk: keys j >= Sq are visible to no query -> dK = dV = 0 there
    w = SMALL["bf16-causal-sq-lt-sk"]
    q, k, v, do = make_inputs(w)
    dq, dk, dv = _gpu_grads(fa, w, q, k, v, do)
    assert torch.all(dk[:, :, w.Sq:] == 0) and torch.all(dv[:, :, w.Sq:] == 0)


@pytest.mark.parametrize("name", ["bf16-gqa-causal-ragged", "bf16-decode-gqa"])
def test_backward_bf16_outputs(fa, name):
    # bf16 outputs: each gradient element is rounded on store (2^-9 relative, the
    # 2^-8 |r| term), and the forward's bf16-rounded O enters D_i = rowsum(dO * O),
    # which perturbs dS = P (dP - D) by up to 2^-9 sum_d |dO_id O_id| per row -- an
    # error of the same order as the fp16 dS rounding. The bound is therefore twice
    # the fp32-output tolerance: |g - r| <= 2^-8 |r| + 4e-2 * RMS(r). (The decode case
    # sums fp32 partial dQ over key ranges and rounds once.)
    w = SMALL[name]
    q, k, v, do = make_inputs(w)
    got = _gpu_grads(fa, w, q, k, v, do, out_dtype=torch.bfloat16)
    ref = oracle.attention_bwd(q, k, v, do, w.scale, w.causal, w.window)
    for g, r in zip(got, ref):
        assert g.dtype == torch.bfloat16
        excess = np.abs(to_np(g) - r) - 2.0 ** -8 * np.abs(r)
        assert excess.max() <= 4e-2 * np.sqrt(np.mean(r ** 2))


@pytest.mark.parametrize("cfg", ["c1", "c2", "c5"])
def test_backward_full_config_fp32(fa, cfg):
    w = WORKLOADS[cfg]
    q, k, v, do = make_inputs(w)
    got = _gpu_grads(fa, w, q, k, v, do)
    ref = oracle.attention_bwd(q, k, v, do, w.scale, w.causal, w.window)
    _check(w, got, ref, cfg)


@pytest.mark.parametrize("cfg,b,g", [("c3", 1, 5), ("c3", 0, 0), ("c4", 0, 3), ("c4", 0, 0)])
def test_backward_full_config_bf16_slice(fa, cfg, b, g):
    # Full-size launch; whole (batch, kv-group) slices are independent, so the
    # oracle checks one slice exactly (dK / dV of the group sum its query heads).
    w = WORKLOADS[cfg]
    q, k, v, do = make_inputs(w)
    dq, dk, dv = _gpu_grads(fa, w, q, k, v, do)
    rep = w.H // w.HKV
    hs = slice(g * rep, (g + 1) * rep)
    ref = oracle.attention_bwd(q[b:b + 1, hs], k[b:b + 1, g:g + 1], v[b:b + 1, g:g + 1],
                               do[b:b + 1, hs], w.scale, w.causal, w.window)
    _check(w, (dq[b:b + 1, hs], dk[b:b + 1, g:g + 1], dv[b:b + 1, g:g + 1]), ref,
           f"{cfg} b{b} g{g}")
    for t in (dq, dk, dv):
        assert torch.isfinite(t).all()
