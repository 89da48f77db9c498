"""Seeded shape fuzz: forward and backward of randomly drawn small problems, each
against the fp64 oracle at the stated tolerances (fp32 inputs: O 2e-3, LSE 1e-3,
gradients 5e-3; bf16 inputs: O 2e-2, LSE 1e-2, gradients 2e-2; max-abs error over
the oracle tensor's RMS, LSE absolute).

The fixed cases in test_parity_fwd.py pick each feature by hand; these draws (one
numpy Generator, seed 2024, so the list is the same on every run) combine them in
ways no fixed case names: batch 1-3, kv groups of 1-6 query heads, Sq and Sk drawn
independently from 1 to 700 (Sq above, equal to or below Sk, ragged tails, single
rows), every head dim that is a multiple of 16 up to 128, causal or not, windows
from 1 key to past the sequence, normal or uniform values with a wider Q / K spread
at times, a softmax scale off 1/sqrt(D), fp32 inputs through either tensor-core
form (the 3xTF32 one only where D <= 64), and for bf16 inputs at times bf16 outputs
(the bound of the fixed bf16-output tests: per element 2^-8 |ref| for the rounding
on store, plus for dQ and dK the derived effect of Delta formed from the stored bf16
O, then the plain bounds) or the materialised-dS backward (fa_bwd_dsmat).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from attention_fa_fwd_02_gb300.workloads import Workload, make_inputs
from _parity import TOL, bf16_output_excess, delta_perturbation_bounds, lse_err, rms_err, to_np


def _draw_cases(n=64, seed=2024):
    rng = np.random.default_rng(seed)
    cases = []
    for idx in range(n):
        dtype = "bf16" if rng.random() < 0.6 else "f32"
        D = int(rng.choice([16, 32, 48, 64, 80, 96, 112, 128]))
        HKV = int(rng.integers(1, 4))
        group = int(rng.integers(1, 7))
        B = int(rng.integers(1, 4))
        Sq = int(rng.choice([1, int(rng.integers(2, 130)), int(rng.integers(130, 701))],
                            p=[0.1, 0.3, 0.6]))
        Sk = int(rng.choice([1, int(rng.integers(2, 130)), int(rng.integers(130, 701))],
                            p=[0.1, 0.3, 0.6]))
        causal = bool(rng.random() < 0.5)
        window = 0 if rng.random() < 0.5 else int(rng.integers(1, max(Sq, Sk) + 50))
        dist = "normal" if rng.random() < 0.8 else "uniform"
        std_qk = float(rng.choice([1.0, 1.5]))
        scale = float(D ** -0.5 * rng.choice([0.5, 1.0, 1.0, 2.0]))
        mode = "f16x2"
        if dtype == "f32" and D <= 64 and rng.random() < 0.4:
            mode = "tf32x3"
        if dtype == "bf16":
            mode = str(rng.choice(["f32out", "f32out", "bf16out", "dsmat"]))
        w = Workload(f"fuzz{idx}", B, HKV * group, HKV, Sq, Sk, D, scale, causal, window, dtype,
                     dist, std_qk, 3000 + idx)
        cases.append((w, mode))
    return cases


CASES = _draw_cases()


def _draw_wide_cases(n=24, seed=2025):
    # longer sequences (more tiles, key ranges, several items per persistent CTA) and
    # per-tensor magnitudes far outside fp16's range (the operand copies' power-of-two
    # scaling), with sharper softmax rows (Q, K std up to 3)
    rng = np.random.default_rng(seed)
    cases = []
    for idx in range(n):
        dtype = "bf16" if rng.random() < 0.6 else "f32"
        D = int(rng.choice([32, 64, 96, 128]))
        HKV = int(rng.integers(1, 3))
        group = int(rng.integers(1, 5))
        Sq = int(rng.integers(1, 2501))
        Sk = int(rng.integers(1, 2501))
        causal = bool(rng.random() < 0.5)
        window = 0 if rng.random() < 0.5 else int(rng.integers(1, max(Sq, Sk) + 50))
        std_qk = float(rng.choice([1.0, 2.0, 3.0]))
        # Q and K by reciprocal powers of two (the scores, and so the softmax, unchanged:
        # scores of thousands would test fp32 itself), V and dO independently
        a_qk = int(rng.integers(-20, 21)) if rng.random() < 0.5 else 0
        mag = (2.0 ** a_qk, 2.0 ** -a_qk) + tuple(
            float(2.0 ** rng.integers(-24, 21)) if rng.random() < 0.5 else 1.0 for _ in range(2))
        mode = "f16x2"
        if dtype == "f32" and D <= 64 and rng.random() < 0.4:
            mode = "tf32x3"
        if dtype == "bf16":
            mode = str(rng.choice(["f32out", "f32out", "dsmat"]))
        w = Workload(f"wide{idx}", 1, HKV * group, HKV, Sq, Sk, D, D ** -0.5, causal, window,
                     dtype, "normal", std_qk, 4000 + idx, mag)
        cases.append((w, mode))
    return cases


WIDE = _draw_wide_cases()


def _label(case):
    w, mma = case
    mag = "" if w.mag == (1.0, 1.0, 1.0, 1.0) else "-mag" + "/".join(f"{m:.0e}" for m in w.mag)
    return (f"{w.name}-{w.dtype}-{mma}-B{w.B}H{w.H}/{w.HKV}"
            f"-Sq{w.Sq}-Sk{w.Sk}-D{w.D}{'-causal' if w.causal else ''}"
            f"{'-w' + str(w.window) if w.window else ''}{mag}")


@pytest.fixture(scope="module")
def fa():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU parity tests need a CUDA device"
    from attention_fa_fwd_02_gb300 import fa as m
    return m


def test_draws_cover_the_features():
    # the fixed seed's list must keep exercising what the docstring promises
    ws = [w for w, _ in CASES]
    assert {w.dtype for w in ws} == {"bf16", "f32"}
    assert {m for _, m in CASES} == {"f16x2", "tf32x3", "f32out", "bf16out", "dsmat"}
    assert any(w.causal for w in ws) and any(not w.causal for w in ws)
    assert any(w.window for w in ws) and any(not w.window for w in ws)
    assert any(w.Sq > w.Sk for w in ws) and any(w.Sq < w.Sk for w in ws)
    assert any(w.H > w.HKV for w in ws)
    assert len({w.D for w in ws}) >= 6
    assert any(w.D % 64 for w in ws)
    assert any(min(w.Sq, w.Sk) < 130 for w in ws)
    assert any(w.Sq % 128 and w.Sk % 128 for w in ws)
    wide = [w for w, _ in WIDE]
    assert any(max(w.Sq, w.Sk) > 2000 for w in wide)
    assert any(min(w.mag) < 2.0 ** -14 for w in wide) and any(max(w.mag) > 2.0 ** 15 for w in wide)
    assert {w.dtype for w in wide} == {"bf16", "f32"} and any(m == "dsmat" for _, m in WIDE)


@pytest.mark.gpu
@pytest.mark.parametrize("case", CASES + WIDE, ids=[_label(c) for c in CASES + WIDE])
def test_fuzz_forward_backward(fa, case):
    w, mode = case
    q, k, v, do = make_inputs(w)
    dev = torch.device("cuda:0")
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    f32_mma = mode if w.dtype == "f32" else "f16x2"
    out_dtype = torch.bfloat16 if mode == "bf16out" else None
    o, lse = fa.forward(qd, kd, vd, w.scale, w.causal, w.window, out_dtype=out_dtype,
                        f32_mma=f32_mma)
    dq, dk, dv = fa.backward(qd, kd, vd, o, lse, dod, w.scale, w.causal, w.window,
                             out_dtype=out_dtype, materialize_ds=mode == "dsmat",
                             f32_mma=f32_mma)
    fa.check_device_status()
    ro, rl = oracle.attention_fwd(q, k, v, w.scale, w.causal, w.window)
    rq, rk, rv = oracle.attention_bwd(q, k, v, do, w.scale, w.causal, w.window)
    if mode == "bf16out":
        # per element: bf16's rounding on store, plus (dQ, dK) the derived effect of
        # Delta formed from the stored bf16 O; beyond those the plain bounds
        bq, bk = delta_perturbation_bounds(q, k, do, ro, rl, w.scale, w.causal, w.window)
        errs = {}
        for name, g, r, extra in (("O", o, ro, 0.0), ("dQ", dq, rq, bq), ("dK", dk, rk, bk),
                                  ("dV", dv, rv, 0.0)):
            assert g.dtype == torch.bfloat16, name
            errs[name] = bf16_output_excess(to_np(g), r, extra)
        lim = {"O": TOL["bf16"]["O"], "dQ": TOL["bf16"]["grad"], "dK": TOL["bf16"]["grad"],
               "dV": TOL["bf16"]["grad"]}
        bad = {n: e for n, e in errs.items() if not e <= lim[n]}
        assert not bad, f"{_label(case)}: {errs}"
        assert lse_err(to_np(lse), rl) <= TOL["bf16"]["LSE"]
        return
    tol = TOL[w.dtype]
    errs = {"O": rms_err(to_np(o), ro), "LSE": lse_err(to_np(lse), rl)}
    for name, g, r in (("dQ", dq, rq), ("dK", dk, rk), ("dV", dv, rv)):
        errs[name] = rms_err(to_np(g), r)
    limit = {"O": tol["O"], "LSE": tol["LSE"], "dQ": tol["grad"], "dK": tol["grad"],
             "dV": tol["grad"]}
    bad = {n: e for n, e in errs.items() if not e <= limit[n]}
    assert not bad, f"{_label(case)}: {errs}"
    assert all(math.isfinite(e) for e in errs.values())
