"""GPU parity at the largest shapes the tests run: a million-token sequence under a
causal sliding window, a 131072-token sequence under full causality, and eighty
thousand heads.

The oracle cannot take these whole, so it checks sampled outputs exactly, each from a
small problem that holds everything that output depends on:
  * the causal and window masks depend on i - j only, so queries and keys sliced with
    the same offset keep exactly their visible pairs;
  * O_i, LSE_i and dQ_i depend on row i alone: q_i with its visible keys, i.e. the
    window slice, or keys [0, i] taken without a mask;
  * dK_j and dV_j depend on the queries that see key j, with their own visible keys:
    under a window w the queries [j, j + w) and the keys [j - w + 1, j + w); under full
    causality at the end of the sequence the last few queries, each a one-row problem
    over keys [0, i], whose backward contributions to key j add up to dK_j, dV_j.
Bounds as in the other parity tests (bf16 inputs: O 2e-2, LSE 1e-2, gradients 2e-2;
fp32 inputs: 2e-3, 1e-3, 5e-3), each error over the RMS of the sampled reference
values.
"""
import numpy as np
import pytest
import torch

import oracle
from attention_fa_fwd_02_gb300.workloads import WORKLOADS, make_inputs
from _parity import TOL, to_np

pytestmark = pytest.mark.gpu

C3 = WORKLOADS["c3"]
WINDOWED_1M = C3.with_(B=1, H=2, HKV=1, Sq=1 << 20, Sk=1 << 20, D=64, scale=0.125, window=512,
                       seed=111, name="window512-causal-gqa2-s1048576-d64-bf16")
CAUSAL_128K = C3.with_(B=1, H=1, HKV=1, Sq=1 << 17, Sk=1 << 17, seed=112,
                       name="causal-h1-s131072-d128-bf16")
MANY_HEADS = C3.with_(B=2, H=40000, HKV=10000, Sq=64, Sk=64, D=64, scale=0.125, seed=113,
                      name="causal-gqa-b2-h40000-hkv10000-s64-d64-bf16")


@pytest.fixture(scope="module")
def fa():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU parity tests need a CUDA device"
    from attention_fa_fwd_02_gb300 import fa as m
    return m


def _run(fa, w, q, k, v, do):
    dev = torch.device("cuda:0")
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    o, lse = fa.forward(qd, kd, vd, w.scale, w.causal, w.window)
    dq, dk, dv = fa.backward(qd, kd, vd, o, lse, dod, w.scale, w.causal, w.window)
    fa.check_device_status()
    del qd, kd, vd, dod
    out = [t.cpu() for t in (o, lse, dq, dk, dv)]
    del o, lse, dq, dk, dv
    torch.cuda.empty_cache()
    return out


def _err(got, ref):
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    assert np.all(np.isfinite(got))
    rms = np.sqrt(np.mean(ref ** 2))
    return float(np.abs(got - ref).max() / (rms if rms > 0 else 1.0))


def _check(errs, dtype="bf16"):
    tol = TOL[dtype]
    lim = {"O": tol["O"], "LSE": tol["LSE"], "dQ": tol["grad"], "dK": tol["grad"], "dV": tol["grad"]}
    bad = {n: e for n, e in errs.items() if not e <= lim[n]}
    assert not bad, errs


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_million_tokens_sliding_window(fa, dtype):
    w = WINDOWED_1M.with_(dtype=dtype)
    q, k, v, do = make_inputs(w)
    o, lse, dq, dk, dv = _run(fa, w, q, k, v, do)
    W, S = w.window, w.Sq
    got = {n: [] for n in ("O", "LSE", "dQ", "dK", "dV")}
    ref = {n: [] for n in got}
    # query rows: the first, tile edges, deep inside, the last
    for i in (0, 127, 128, 511, 512, 300000, 777777, S - 129, S - 1):
        lo = max(0, i - W + 1)
        qs, ks, vs, dos = q[:, :, lo:i + 1], k[:, :, lo:i + 1], v[:, :, lo:i + 1], do[:, :, lo:i + 1].clone()
        dos[:, :, :-1] = 0  # only row i's own gradient
        ro, rl = oracle.attention_fwd(qs, ks, vs, w.scale, True, W)
        rq, _, _ = oracle.attention_bwd(qs, ks, vs, dos, w.scale, True, W)
        got["O"].append(to_np(o[:, :, i])); ref["O"].append(ro[:, :, -1])
        got["LSE"].append(to_np(lse[:, :, i])); ref["LSE"].append(rl[:, :, -1])
        got["dQ"].append(to_np(dq[:, :, i])); ref["dQ"].append(rq[:, :, -1])
    # key rows: every query that sees key j, with all of its keys
    for j in (0, 1, 128, 4095, 555555, S - 512, S - 1):
        lo, hi = max(0, j - W + 1), min(S, j + W)
        qs, ks, vs, dos = q[:, :, lo:hi], k[:, :, lo:hi], v[:, :, lo:hi], do[:, :, lo:hi].clone()
        dos[:, :, :j - lo] = 0  # queries before j do not see it; their rows stay out
        _, rk, rv = oracle.attention_bwd(qs, ks, vs, dos, w.scale, True, W)
        got["dK"].append(to_np(dk[:, :, j])); ref["dK"].append(rk[:, :, j - lo])
        got["dV"].append(to_np(dv[:, :, j])); ref["dV"].append(rv[:, :, j - lo])
    errs = {n: _err(np.stack(got[n]), np.stack(ref[n])) for n in got if n != "LSE"}
    errs["LSE"] = float(np.abs(np.stack(got["LSE"]) - np.stack(ref["LSE"])).max())
    _check(errs, w.dtype)


def test_131072_tokens_full_causal(fa):
    w = CAUSAL_128K
    q, k, v, do = make_inputs(w)
    o, lse, dq, dk, dv = _run(fa, w, q, k, v, do)
    S, T = w.Sq, 16
    got = {n: [] for n in ("O", "LSE", "dQ", "dK", "dV")}
    ref = {n: [] for n in got}
    dk_last = np.zeros((1, 1, T, w.D))
    dv_last = np.zeros((1, 1, T, w.D))
    rows = sorted(set((0, 1, 127, 128, 65535, 100001)) | set(range(S - T, S)))
    for i in rows:
        # row i over its visible keys [0, i], no mask needed
        qs, ks, vs, dos = q[:, :, i:i + 1], k[:, :, :i + 1], v[:, :, :i + 1], do[:, :, i:i + 1]
        ro, rl = oracle.attention_fwd(qs, ks, vs, w.scale, False, 0)
        rq, rk, rv = oracle.attention_bwd(qs, ks, vs, dos, w.scale, False, 0)
        got["O"].append(to_np(o[:, :, i])); ref["O"].append(ro[:, :, 0])
        got["LSE"].append(to_np(lse[:, :, i])); ref["LSE"].append(rl[:, :, 0])
        got["dQ"].append(to_np(dq[:, :, i])); ref["dQ"].append(rq[:, :, 0])
        if i >= S - T:  # the only queries that see the last T keys
            dk_last[:, :, :i + 1 - (S - T)] += rk[:, :, S - T:i + 1]
            dv_last[:, :, :i + 1 - (S - T)] += rv[:, :, S - T:i + 1]
    got["dK"].append(to_np(dk[:, :, S - T:])); ref["dK"].append(dk_last)
    got["dV"].append(to_np(dv[:, :, S - T:])); ref["dV"].append(dv_last)
    errs = {n: _err(np.stack(got[n]), np.stack(ref[n])) for n in got if n != "LSE"}
    errs["LSE"] = float(np.abs(np.stack(got["LSE"]) - np.stack(ref["LSE"])).max())
    _check(errs)


def test_eighty_thousand_heads(fa):
    w = MANY_HEADS
    q, k, v, do = make_inputs(w)
    o, lse, dq, dk, dv = _run(fa, w, q, k, v, do)
    rep = w.H // w.HKV
    for b, g in ((0, 0), (1, 4321), (1, w.HKV - 1)):
        hs = slice(g * rep, (g + 1) * rep)
        args = (q[b:b + 1, hs], k[b:b + 1, g:g + 1], v[b:b + 1, g:g + 1])
        ro, rl = oracle.attention_fwd(*args, w.scale, w.causal, w.window)
        rq, rk, rv = oracle.attention_bwd(*args, do[b:b + 1, hs], w.scale, w.causal, w.window)
        errs = {"O": _err(to_np(o[b:b + 1, hs]), ro),
                "LSE": float(np.abs(to_np(lse[b:b + 1, hs]) - rl).max()),
                "dQ": _err(to_np(dq[b:b + 1, hs]), rq),
                "dK": _err(to_np(dk[b:b + 1, g:g + 1]), rk),
                "dV": _err(to_np(dv[b:b + 1, g:g + 1]), rv)}
        _check(errs)
