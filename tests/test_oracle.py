"""Pins for the fp64 oracle (CPU only).

The oracle is the yardstick for every GPU parity test, so it is checked here
against things other than itself: hand-derived examples, closed forms, special
cases that reduce to simpler results, invariants of softmax attention, an
independent library routine (torch fp64 + autograd) and central finite
differences. ``test_planted_mistakes_are_caught`` compiles mutated copies of the
oracle (a dropped term, an off-by-one mask, a wrong operand or head mapping) and
requires each to fail at least one pin.
"""
import json
import math
import os
import shutil

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_examples.json")
ORC = None


def _orc():
    global ORC
    if ORC is None:
        ORC = oracle._load()
    return ORC


def _rand(rng, *shape, std=1.0):
    return rng.standard_normal(shape) * std


def _problem(seed, B=1, H=4, HKV=2, Sq=12, Sk=12, D=8):
    rng = np.random.default_rng(seed)
    q = _rand(rng, B, H, Sq, D)
    k = _rand(rng, B, HKV, Sk, D)
    v = _rand(rng, B, HKV, Sk, D)
    do = _rand(rng, B, H, Sq, D)
    return q, k, v, do


def _visible(i, j, causal, window):
    if causal and j > i:
        return False
    if window > 0 and j < i - window + 1:
        return False
    return True


MODES = [(False, 0), (True, 0), (True, 3), (False, 4), (True, 1)]


# ----------------------------------------------------------------------------- pins
def pin_hand_examples(orc):
    env = {"ln2": math.log(2.0), "ln3": math.log(3.0), "inf": math.inf, "__builtins__": {}}
    ev = np.vectorize(lambda s: float(eval(s, env)))
    for ex in json.load(open(GOLDEN))["examples"]:
        scale = float(eval(ex["scale"], env))
        q, k, v, do = (np.array(ex[n], np.float64) for n in ("Q", "K", "V", "dO"))
        o, lse = orc.attention_fwd(q, k, v, scale, ex["causal"], ex["window"])
        dq, dk, dv = orc.attention_bwd(q, k, v, do, scale, ex["causal"], ex["window"])
        np.testing.assert_allclose(o, ev(np.array(ex["O"])), rtol=0, atol=1e-12, err_msg=ex["name"])
        want = ev(np.array(ex["LSE"]))
        assert np.array_equal(np.isneginf(lse), np.isneginf(want)), ex["name"]
        fin = np.isfinite(want)
        np.testing.assert_allclose(lse[fin], want[fin], rtol=0, atol=1e-12, err_msg=ex["name"])
        for got, key in ((dq, "dQ"), (dk, "dK"), (dv, "dV")):
            np.testing.assert_allclose(got, ev(np.array(ex[key])), rtol=0, atol=1e-12,
                                       err_msg=f"{ex['name']} {key}")


def pin_rows_sum_to_one(orc):
    # With V = identity (Sk == D), O_i is the probability row P_i itself.
    rng = np.random.default_rng(1)
    Sk = D = 8
    for causal, window in MODES:
        q = _rand(rng, 1, 2, 10, D)
        k = _rand(rng, 1, 2, Sk, D)
        v = np.broadcast_to(np.eye(Sk), (1, 2, Sk, D)).copy()
        o, lse = orc.attention_fwd(q, k, v, 0.7, causal, window)
        for h in range(2):
            for i in range(10):
                row = o[0, h, i]
                vis = [_visible(i, j, causal, window) for j in range(Sk)]
                if not any(vis):
                    assert np.all(row == 0) and np.isneginf(lse[0, h, i])
                    continue
                assert abs(row.sum() - 1.0) <= 1e-12
                assert np.all(row >= 0)
                assert all(row[j] == 0.0 for j in range(Sk) if not vis[j])


def pin_lse_independent(orc):
    # LSE recomputed in pure Python with exactly rounded sums (math.fsum).
    q, k, v, _ = _problem(2, B=1, H=2, HKV=1, Sq=9, Sk=11, D=5)
    for causal, window in MODES:
        _, lse = orc.attention_fwd(q, k, v, 0.4, causal, window)
        for h in range(2):
            for i in range(9):
                s = [0.4 * math.fsum(q[0, h, i, d] * k[0, 0, j, d] for d in range(5))
                     for j in range(11) if _visible(i, j, causal, window)]
                if not s:
                    assert np.isneginf(lse[0, h, i])
                    continue
                m = max(s)
                want = m + math.log(math.fsum(math.exp(x - m) for x in s))
                assert abs(lse[0, h, i] - want) <= 1e-12 * max(1.0, abs(want))


def pin_constant_v(orc):
    q, k, _, _ = _problem(3)
    v = np.full((1, 2, 12, 8), 2.5)
    for causal, window in MODES:
        o, lse = orc.attention_fwd(q, k, v, 0.35, causal, window)
        ok = np.isfinite(lse)
        assert np.abs(o[ok] - 2.5).max() <= 1e-12


def pin_causal_row0_and_window1(orc):
    q, k, v, do = _problem(4)
    scale = 0.3
    o, lse = orc.attention_fwd(q, k, v, scale, True, 0)
    dq, _, _ = orc.attention_bwd(q, k, v, do, scale, True, 0)
    kv = np.repeat(k, 2, axis=1)
    vv = np.repeat(v, 2, axis=1)
    np.testing.assert_allclose(o[:, :, 0], vv[:, :, 0], rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse[:, :, 0], scale * np.einsum("bhd,bhd->bh", q[:, :, 0], kv[:, :, 0]),
                               rtol=0, atol=1e-13)
    assert np.abs(dq[:, :, 0]).max() <= 1e-14
    # causal + window 1: each row sees only itself
    o, lse = orc.attention_fwd(q, k, v, scale, True, 1)
    dq, dk, dv = orc.attention_bwd(q, k, v, do, scale, True, 1)
    np.testing.assert_allclose(o, vv, rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse, scale * np.einsum("bhid,bhid->bhi", q, kv), rtol=0, atol=1e-13)
    assert np.abs(dq).max() <= 1e-14 and np.abs(dk).max() <= 1e-14
    np.testing.assert_allclose(dv, do.reshape(1, 2, 2, 12, 8).sum(2), rtol=0, atol=1e-13)


def pin_window_zero_is_full(orc):
    q, k, v, do = _problem(5)
    for causal in (False, True):
        a = orc.attention_fwd(q, k, v, 0.5, causal, 0)
        b = orc.attention_fwd(q, k, v, 0.5, causal, 12)
        c = orc.attention_fwd(q, k, v, 0.5, causal, 1000)
        for x, y, z in zip(a, b, c):
            assert np.array_equal(x, y) and np.array_equal(x, z)
        ga = orc.attention_bwd(q, k, v, do, 0.5, causal, 0)
        gb = orc.attention_bwd(q, k, v, do, 0.5, causal, 12)
        for x, y in zip(ga, gb):
            assert np.array_equal(x, y)


def pin_gqa_is_repeated_mha(orc):
    q, k, v, do = _problem(6, B=2, H=6, HKV=2, Sq=7, Sk=9, D=4)
    rep = 3
    for causal, window in MODES:
        o, lse = orc.attention_fwd(q, k, v, 0.6, causal, window)
        om, lm = orc.attention_fwd(q, np.repeat(k, rep, 1), np.repeat(v, rep, 1), 0.6, causal, window)
        np.testing.assert_allclose(o, om, rtol=0, atol=1e-13)
        assert np.array_equal(np.isneginf(lse), np.isneginf(lm))
        np.testing.assert_allclose(lse[np.isfinite(lse)], lm[np.isfinite(lm)], rtol=0, atol=1e-13)
        dq, dk, dv = orc.attention_bwd(q, k, v, do, 0.6, causal, window)
        dqm, dkm, dvm = orc.attention_bwd(q, np.repeat(k, rep, 1), np.repeat(v, rep, 1), do, 0.6,
                                          causal, window)
        np.testing.assert_allclose(dq, dqm, rtol=0, atol=1e-13)
        np.testing.assert_allclose(dk, dkm.reshape(2, 2, rep, 9, 4).sum(2), rtol=0, atol=1e-12)
        np.testing.assert_allclose(dv, dvm.reshape(2, 2, rep, 9, 4).sum(2), rtol=0, atol=1e-12)
    # HKV == H is plain multi-head attention
    q, k, v, do = _problem(7, H=3, HKV=3)
    o, _ = orc.attention_fwd(q, k, v, 0.6, True, 0)
    for h in range(3):
        oh, _ = orc.attention_fwd(q[:, h:h + 1], k[:, h:h + 1], v[:, h:h + 1], 0.6, True, 0)
        np.testing.assert_allclose(o[:, h:h + 1], oh, rtol=0, atol=0)


def pin_invariants(orc):
    q, k, v, do = _problem(8, B=1, H=4, HKV=2, Sq=13, Sk=10, D=6)
    for causal, window in MODES:
        o, lse = orc.attention_fwd(q, k, v, 0.45, causal, window)
        dq, dk, dv = orc.attention_bwd(q, k, v, do, 0.45, causal, window)
        nonempty = np.isfinite(lse)[..., None]
        # sum_j dV_j = sum over the group's non-empty query rows of dO_i
        want = (do * nonempty).reshape(1, 2, 2, 13, 6).sum(axis=(2, 3))
        np.testing.assert_allclose(dv.sum(2), want, rtol=0, atol=1e-12)
        # sum_j dK_j = 0 (each softmax row of dS sums to zero)
        assert np.abs(dk.sum(2)).max() <= 1e-12
        # a constant added to every key leaves O unchanged and shifts LSE by scale q.c
        c = np.linspace(-1.0, 1.0, 6)
        o2, lse2 = orc.attention_fwd(q, k + c, v, 0.45, causal, window)
        np.testing.assert_allclose(o2, o, rtol=0, atol=1e-12)
        fin = np.isfinite(lse)
        assert np.array_equal(fin, np.isfinite(lse2))
        np.testing.assert_allclose(lse2[fin] - lse[fin], (0.45 * q @ c)[fin], rtol=0, atol=1e-12)


def _torch_reference(q, k, v, do, scale, causal, window):
    """Naive torch fp64 attention with an explicit boolean mask, gradients by autograd."""
    q, k, v, do = (torch.tensor(x, dtype=torch.float64) for x in (q, k, v, do))
    rep = q.shape[1] // k.shape[1]
    q.requires_grad_(True); k.requires_grad_(True); v.requires_grad_(True)
    kk, vv = k.repeat_interleave(rep, 1), v.repeat_interleave(rep, 1)
    Sq, Sk = q.shape[2], k.shape[2]
    mask = torch.tensor([[_visible(i, j, causal, window) for j in range(Sk)] for i in range(Sq)])
    s = scale * q @ kk.transpose(-1, -2)
    s = s.masked_fill(~mask, -math.inf)
    lse = torch.logsumexp(s, -1)
    p = torch.softmax(s, -1).nan_to_num(0.0)
    o = p @ vv
    (o * do).sum().backward()
    sdpa = torch.nn.functional.scaled_dot_product_attention(
        q.detach(), kk.detach(), vv.detach(), attn_mask=mask, scale=scale)
    return o.detach(), lse.detach(), q.grad, k.grad, v.grad, sdpa, mask


def pin_library_crosscheck(orc):
    for seed, (causal, window) in enumerate(MODES):
        q, k, v, do = _problem(20 + seed, B=2, H=4, HKV=2, Sq=11, Sk=14, D=8)
        o, lse = orc.attention_fwd(q, k, v, 0.33, causal, window)
        dq, dk, dv = orc.attention_bwd(q, k, v, do, 0.33, causal, window)
        to, tl, tdq, tdk, tdv, sdpa, mask = _torch_reference(q, k, v, do, 0.33, causal, window)
        rows = mask.any(-1).numpy()
        np.testing.assert_allclose(o, to.numpy(), rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(o[:, :, rows], sdpa.numpy()[:, :, rows], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(lse[:, :, rows], tl.numpy()[:, :, rows], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(dq, tdq.numpy(), rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(dk, tdk.numpy(), rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(dv, tdv.numpy(), rtol=1e-11, atol=1e-12)


def pin_finite_differences(orc):
    h = 1e-6
    for seed, (causal, window) in enumerate(MODES[:4]):
        q, k, v, do = _problem(40 + seed, B=1, H=4, HKV=2, Sq=6, Sk=7, D=3)
        scale = 0.55

        def loss(q_, k_, v_):
            o, _ = orc.attention_fwd(q_, k_, v_, scale, causal, window)
            return float((o * do).sum())

        grads = orc.attention_bwd(q, k, v, do, scale, causal, window)
        for which, g in enumerate(grads):
            base = [q, k, v]
            fd = np.zeros_like(g)
            it = np.nditer(g, flags=["multi_index"])
            for _ in it:
                idx = it.multi_index
                plus = [x.copy() for x in base]
                minus = [x.copy() for x in base]
                plus[which][idx] += h
                minus[which][idx] -= h
                fd[idx] = (loss(*plus) - loss(*minus)) / (2 * h)
            err = np.abs(fd - g).max() / max(np.abs(g).max(), 1e-30)
            assert err <= 1e-7, (causal, window, which, err)


def pin_empty_rows(orc):
    # Sq > Sk with causal + window: rows i >= Sk + window - 1 see no key.
    q, k, v, do = _problem(9, B=1, H=2, HKV=1, Sq=12, Sk=6, D=4)
    o, lse = orc.attention_fwd(q, k, v, 0.5, True, 3)
    dq, dk, dv = orc.attention_bwd(q, k, v, do, 0.5, True, 3)
    assert np.all(o[:, :, 8:] == 0) and np.all(np.isneginf(lse[:, :, 8:]))
    assert np.all(np.isfinite(lse[:, :, :8]))
    assert np.all(dq[:, :, 8:] == 0)
    # empty rows contribute nothing to dK/dV
    _, dk2, dv2 = orc.attention_bwd(q[:, :, :8], k, v, do[:, :, :8], 0.5, True, 3)
    np.testing.assert_allclose(dk, dk2, rtol=0, atol=1e-14)
    np.testing.assert_allclose(dv, dv2, rtol=0, atol=1e-14)


def pin_magnitude_homogeneity(orc):
    # O is linear in V and LSE does not depend on it; the gradients are linear in dO;
    # dQ and dK are linear in V while dV does not depend on it. With powers of two every
    # product and sum scales exactly, so the results must match bit for bit, at the
    # magnitudes the GPU parity cases use (V of 1e5, dO of 1e-7 and 1e4, V of 1e-6).
    for causal, window in MODES[:3]:
        q, k, v, do = _problem(61, B=1, H=4, HKV=2, Sq=10, Sk=9, D=4)
        o, lse = orc.attention_fwd(q, k, v, 0.6, causal, window)
        g = orc.attention_bwd(q, k, v, do, 0.6, causal, window)
        for c in (2.0 ** 17, 2.0 ** -23, 2.0 ** 13, 2.0 ** -20):
            o2, lse2 = orc.attention_fwd(q, k, v * c, 0.6, causal, window)
            assert np.array_equal(o2, o * c) and np.array_equal(lse2, lse)
            gd = orc.attention_bwd(q, k, v, do * c, 0.6, causal, window)
            for x, y in zip(gd, g):
                assert np.array_equal(x, y * c)
            gv = orc.attention_bwd(q, k, v * c, do, 0.6, causal, window)
            assert np.array_equal(gv[0], g[0] * c) and np.array_equal(gv[1], g[1] * c)
            assert np.array_equal(gv[2], g[2])
        # scores of 2^-40: the softmax is uniform over each row's visible keys to ~1e-12
        c = 2.0 ** -20
        o3, lse3 = orc.attention_fwd(q * c, k * c, v, 0.6, causal, window)
        for i in range(q.shape[2]):
            vis = [j for j in range(k.shape[2]) if _visible(i, j, causal, window)]
            for h in range(4):
                np.testing.assert_allclose(o3[0, h, i], v[0, h // 2, vis].mean(axis=0),
                                           rtol=0, atol=1e-10)
                assert abs(lse3[0, h, i] - math.log(len(vis))) < 1e-10


PINS = [pin_hand_examples, pin_rows_sum_to_one, pin_lse_independent, pin_constant_v,
        pin_causal_row0_and_window1, pin_window_zero_is_full, pin_gqa_is_repeated_mha,
        pin_invariants, pin_library_crosscheck, pin_finite_differences, pin_empty_rows,
        pin_magnitude_homogeneity]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_oracle_pin(pin):
    pin(_orc())


def test_oracle_rejects_bad_shapes():
    q, k, v, do = _problem(10, H=3, HKV=2)
    with pytest.raises(ValueError):
        _orc().attention_fwd(q, k, v, 0.5, True, 0)
    with pytest.raises(ValueError):
        _orc().attention_bwd(q, k, v, do, 0.5, True, 0)


def test_oracle_deterministic_across_thread_counts(tmp_path):
    # each output element comes from one OpenMP iteration in a fixed order
    import subprocess, sys
    code = ("import numpy as np, oracle;"
            "r=np.random.default_rng(3);q=r.standard_normal((1,4,40,8));k=r.standard_normal((1,2,40,8));"
            "v=r.standard_normal((1,2,40,8));d=r.standard_normal((1,4,40,8));"
            "o,l=oracle.attention_fwd(q,k,v,.4,True,9);g=oracle.attention_bwd(q,k,v,d,.4,True,9);"
            "np.save(%r,np.concatenate([o.ravel(),l.ravel()]+[x.ravel() for x in g]))")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    outs = []
    for n in (1, 3):
        f = str(tmp_path / f"t{n}.npy")
        env = dict(os.environ, OMP_NUM_THREADS=str(n), PYTHONPATH=root)
        subprocess.run([sys.executable, "-c", code % f], check=True, env=env, cwd=root)
        outs.append(np.load(f))
    assert np.array_equal(outs[0], outs[1])


# Plausible mistakes, each planted in a copy of the oracle source; every one must
# be caught by at least one pin.
MUTATIONS = [
    ("causal off by one", "if (s->causal && j > i) return 0;", "if (s->causal && j >= i) return 0;"),
    ("window off by one", "j < i - (long)s->window + 1", "j < i - (long)s->window"),
    ("lse drops the max", "return m + log(sum);", "return log(sum);"),
    ("scale dropped in S", "p[j] = s->scale * dot(", "p[j] = dot("),
    ("wrong gqa head map", "h = bh % H, b = bh / H, g = h / rep;\n      const double* qi",
     "h = bh % H, b = bh / H, g = h % HKV;\n      const double* qi"),
    ("dropped r_i term", "ri += p[j] * dp[j];", "ri += 0.0 * dp[j];"),
    ("dK uses K not Q", "dkj[d] += ds * qi[d];", "dkj[d] += ds * kj[d];"),
    ("dV uses P.V", "dvj[d] += pij * doi[d];", "dvj[d] += pij * vj[d];"),
    ("dQ scale dropped", "for (int d = 0; d < D; ++d) dqi[d] *= scale;", ""),
    ("sign of dS flipped", "const double ds = p[j] * (dp[j] - ri);", "const double ds = p[j] * (ri - dp[j]);"),
    ("O not normalised", "for (long j = 0; j < Sk; ++j) p[j] /= sum;", ""),
    ("dK over one head only", "for (int t = 0; t < rep; ++t) {", "for (int t = 0; t < 1; ++t) {"),
]


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistakes_are_caught(tmp_path, name, old, new):
    src = open(oracle._SRC).read()
    assert src.count(old) == 1, f"mutation anchor not unique: {name}"
    mutant = tmp_path / "mutant.c"
    mutant.write_text(src.replace(old, new))
    lib = oracle.OracleLib(oracle.build(force=True, src=str(mutant), out=str(tmp_path / "mut.so")))
    caught = []
    for pin in PINS:
        try:
            pin(lib)
        except (AssertionError, ValueError, FloatingPointError):
            caught.append(pin.__name__)
    assert caught, f"no pin caught the planted mistake: {name}"
