"""GPU parity of the materialised-dS backward (fa_bwd_dsmat through the C ABI)
against the fp64 oracle.

fa_bwd_dsmat reaches the same gradients as fa_bwd by another route (the dK / dV
kernel also stores dS^T, and dQ is a GEMM over it; metal-flash-attention README,
backward pass), so it is held to the same bounds: 2e-2 of the oracle tensor's RMS for
bf16 inputs. O and LSE come from fa_fwd, as a caller would pass them.
"""
import pytest
import torch

import oracle
from attention_fa_fwd_02_gb300.workloads import WORKLOADS, make_inputs
from _parity import TOL, bf16_output_excess, delta_perturbation_bounds, rms_err, to_np
from test_parity_fwd import SMALL

pytestmark = pytest.mark.gpu

# causal / windowed / ragged / Sq != Sk / empty rows and tiles / head dims / GQA
# groups / short query sequences (two-term operands) / out-of-range magnitudes
CASES = ["bf16-gqa-causal-ragged", "bf16-gqa-window", "bf16-d64-causal", "bf16-noncausal-sq-ne-sk",
         "bf16-causal-sq-lt-sk", "bf16-empty-rows", "bf16-window1", "bf16-s1", "bf16-noncausal-window",
         "bf16-many-items-causal", "bf16-d96-causal-gqa", "bf16-d48-noncausal-sq-ne-sk",
         "bf16-d16-causal", "bf16-decode-gqa", "bf16-decode-causal-sq-lt-sk",
         "bf16-decode-window-empty-tail", "bf16-decode-sq128-sk16384",
         "bf16-decode-sq128-sk16384-std2", "bf16-gqa3-window-ragged", "bf16-decode-sq1",
         "bf16-mag-all", "bf16-mag-huge-dO-tiny-V"]


@pytest.fixture(scope="module")
def fa():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU parity tests need a CUDA device"
    from attention_fa_fwd_02_gb300 import fa as m
    return m


def _grads(fa, w, q, k, v, do):
    dev = torch.device("cuda:0")
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    o, lse = fa.forward(qd, kd, vd, w.scale, w.causal, w.window)
    g = fa.backward(qd, kd, vd, o, lse, dod, w.scale, w.causal, w.window, materialize_ds=True)
    fa.check_device_status()
    return g


def _check(w, got, ref, label):
    tol = TOL[w.dtype]["grad"]
    errs = {n: rms_err(to_np(g), r) for n, g, r in zip(("dQ", "dK", "dV"), got, ref)}
    bad = {k: e for k, e in errs.items() if not e <= tol}
    assert not bad, f"{label}: {errs} (tol {tol})"


@pytest.mark.parametrize("name", CASES)
def test_dsmat_backward_small(fa, name):
    w = SMALL[name]
    q, k, v, do = make_inputs(w)
    got = _grads(fa, w, q, k, v, do)
    ref = oracle.attention_bwd(q, k, v, do, w.scale, w.causal, w.window)
    _check(w, got, ref, name)


@pytest.mark.parametrize("cfg,b,g", [("c3", 1, 5), ("c4", 0, 3)])
def test_dsmat_backward_full_config_bf16_slice(fa, cfg, b, g):
    # full-size launch (a 2 GB dS buffer at C3); whole (batch, kv-group) slices checked
    w = WORKLOADS[cfg]
    q, k, v, do = make_inputs(w)
    dq, dk, dv = _grads(fa, w, q, k, v, do)
    rep = w.H // w.HKV
    hs = slice(g * rep, (g + 1) * rep)
    ref = oracle.attention_bwd(q[b:b + 1, hs], k[b:b + 1, g:g + 1], v[b:b + 1, g:g + 1],
                               do[b:b + 1, hs], w.scale, w.causal, w.window)
    _check(w, (dq[b:b + 1, hs], dk[b:b + 1, g:g + 1], dv[b:b + 1, g:g + 1]), ref, f"{cfg} b{b} g{g}")
    for t in (dq, dk, dv):
        assert torch.isfinite(t).all()


def test_dsmat_backward_deterministic(fa):
    w = SMALL["bf16-gqa-causal-ragged"]
    q, k, v, do = make_inputs(w)
    a = _grads(fa, w, q, k, v, do)
    b = _grads(fa, w, q, k, v, do)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_dsmat_backward_bf16_outputs(fa):
    # the bound of the bf16-output test of fa_bwd: per element u |r| (rounding on
    # store) plus the derived perturbation of dQ / dK by Delta from the bf16 O, then
    # 2e-2 * RMS(r)
    w = SMALL["bf16-gqa-causal-ragged"]
    q, k, v, do = make_inputs(w)
    dev = torch.device("cuda:0")
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    o, lse = fa.forward(qd, kd, vd, w.scale, w.causal, w.window, out_dtype=torch.bfloat16)
    got = fa.backward(qd, kd, vd, o, lse, dod, w.scale, w.causal, w.window,
                      out_dtype=torch.bfloat16, materialize_ds=True)
    fa.check_device_status()
    ref = oracle.attention_bwd(q, k, v, do, w.scale, w.causal, w.window)
    ro, rl = oracle.attention_fwd(q, k, v, w.scale, w.causal, w.window)
    bq, bk = delta_perturbation_bounds(q, k, do, ro, rl, w.scale, w.causal, w.window)
    for g, r, extra in zip(got, ref, (bq, bk, 0.0)):
        assert g.dtype == torch.bfloat16
        assert bf16_output_excess(to_np(g), r, extra) <= TOL["bf16"]["grad"]