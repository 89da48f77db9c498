"""GPU parity of the backward pass (fa_bwd through the C ABI) against the fp64 oracle.

The GPU path takes O and LSE from its own forward pass, exactly as a caller
would; the oracle derives dQ / dK / dV from Q, K, V, dO alone through the softmax
Jacobian. Tolerances (max-abs error / RMS of the oracle tensor): 5e-3 for fp32
inputs (either f32_mma), 2e-2 for bf16 inputs.
"""
import numpy as np
import pytest
import torch

import oracle
from attention_fa_fwd_02_gb300.workloads import WORKLOADS, make_inputs
from _parity import TOL, bf16_output_excess, delta_perturbation_bounds, rms_err, to_np
from test_parity_fwd import C2_D128, C3_D32, SMALL

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


@pytest.mark.parametrize("name", list(SMALL))
def test_backward_small(fa, name):
    w = SMALL[name]
    q, k, v, do = make_inputs(w)
    got = _gpu_grads(fa, w, q, k, v, do)
    ref = oracle.attention_bwd(q, k, v, do, w.scale, w.causal, w.window)
    _check(w, got, ref, name)


@pytest.mark.parametrize("name", ["bf16-gqa-causal-ragged", "bf16-decode-gqa", "bf16-decode-sq1",
                                  "f32-decode-sq2-gqa4-d80", "f32-decode",
                                  "bf16-short-keys-causal-window", "f32-short-keys-gqa-window"])
def test_backward_deterministic(fa, name):
    # dK / dV are accumulated per key tile without atomics, dQ per query tile (or per
    # key range, the ranges then summed in a fixed order): bit-identical reruns. (The
    # decode shapes' backward: every key's dK, dV formed by one lane pair, dQ summed
    # over the warps and the key ranges in fixed orders.)
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


@pytest.mark.parametrize("name", ["bf16-gqa-causal-ragged", "bf16-decode-gqa",
                                  "bf16-d32-causal-gqa-ragged", "bf16-decode-rows8-s20000",
                                  "bf16-short-keys"])
def test_backward_bf16_outputs(fa, name):
    # bf16 outputs: each gradient element is rounded on store (at most 2^-8 |r|), and
    # the backward forms Delta_i = rowsum(dO * O) from the bf16 O the forward stored,
    # which moves dQ and dK by at most the bounds delta_perturbation_bounds derives
    # (dV does not involve Delta). Beyond those two, the plain 2e-2 * RMS(r).
    w = SMALL[name]
    q, k, v, do = make_inputs(w)
    got = _gpu_grads(fa, w, q, k, v, do, out_dtype=torch.bfloat16)
    ref = oracle.attention_bwd(q, k, v, do, w.scale, w.causal, w.window)
    ro, rl = oracle.attention_fwd(q, k, v, w.scale, w.causal, w.window)
    bq, bk = delta_perturbation_bounds(q, k, do, ro, rl, w.scale, w.causal, w.window)
    for n, g, r, extra in (("dQ", got[0], ref[0], bq), ("dK", got[1], ref[1], bk),
                           ("dV", got[2], ref[2], 0.0)):
        assert g.dtype == torch.bfloat16
        ex = bf16_output_excess(to_np(g), r, extra)
        assert ex <= TOL["bf16"]["grad"], f"{name}: {n} excess {ex:.3e}"


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_backward_decode_16_byte_aligned_inputs(fa, dtype):
    # the C ABI promises 16-byte alignment only: Q, K, V and dO here start 16 bytes into
    # their allocations, so the decode backward reads K and V rows 16 bytes per load
    base = WORKLOADS["c3"] if dtype == "bf16" else WORKLOADS["c5"]
    w = base.with_(B=2, H=8, HKV=2, Sq=1, Sk=3001, D=128, scale=128 ** -0.5, causal=False,
                   window=0, seed=130)
    q, k, v, do = make_inputs(w)
    dev = torch.device("cuda:0")
    pad = 16 // q.element_size()

    def offset_copy(t):
        buf = torch.empty(t.numel() + pad, dtype=t.dtype, device=dev)
        view = buf[pad:].view(t.shape)
        view.copy_(t.to(dev))
        assert view.data_ptr() % 32 == 16 and view.is_contiguous()
        return view

    qd, kd, vd, dod = (offset_copy(t) for t in (q, k, v, do))
    o, lse = fa.forward(qd, kd, vd, w.scale, w.causal, w.window)
    got = fa.backward(qd, kd, vd, o, lse, dod, w.scale, w.causal, w.window)
    fa.check_device_status()
    ref = oracle.attention_bwd(q, k, v, do, w.scale, w.causal, w.window)
    _check(w, got, ref, f"decode-16B-aligned-{dtype}")


def test_backward_short_keys_tf32x3(fa):
    # fp32 through the 3xTF32 kernels with few key tiles: the dK / dV items split the
    # queries into ranges there too
    w = SMALL["f32-short-keys"]
    q, k, v, do = make_inputs(w)
    dev = torch.device("cuda:0")
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    o, lse = fa.forward(qd, kd, vd, w.scale, w.causal, w.window, f32_mma="tf32x3")
    got = fa.backward(qd, kd, vd, o, lse, dod, w.scale, w.causal, w.window, f32_mma="tf32x3")
    fa.check_device_status()
    ref = oracle.attention_bwd(q, k, v, do, w.scale, w.causal, w.window)
    _check(w, got, ref, "f32-short-keys-tf32x3")


@pytest.mark.parametrize("cfg", ["c1", "c2", "c5", "c2-d128"])
def test_backward_full_config_fp32(fa, cfg):
    w = C2_D128 if cfg == "c2-d128" else WORKLOADS[cfg]
    q, k, v, do = make_inputs(w)
    got = _gpu_grads(fa, w, q, k, v, do)
    ref = oracle.attention_bwd(q, k, v, do, w.scale, w.causal, w.window)
    _check(w, got, ref, cfg)


@pytest.mark.parametrize("cfg,b,g", [("c3", 1, 5), ("c3", 0, 0), ("c4", 0, 3), ("c4", 0, 0),
                                     ("c3-d32", 1, 2)])
def test_backward_full_config_bf16_slice(fa, cfg, b, g):
    # Full-size launch; whole (batch, kv-group) slices are independent, so the
    # oracle checks one slice exactly (dK / dV of the group sum its query heads).
    w = C3_D32 if cfg == "c3-d32" else WORKLOADS[cfg]
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
