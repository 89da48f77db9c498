"""GPU parity of the forward pass (fa_fwd through the C ABI) against the fp64 oracle.

Tolerances (from the problem statement): fp32 inputs (either f32_mma) O <= 2e-3
max-abs / RMS, LSE <= 1e-3 absolute; bf16 inputs O <= 2e-2, LSE <= 1e-2. The
oracle runs on the same (bf16-rounded) inputs.
"""
import numpy as np
import pytest
import torch

import oracle
from attention_fa_fwd_02_gb300.workloads import WORKLOADS, make_inputs
from _parity import TOL, lse_err, rms_err, to_np

pytestmark = pytest.mark.gpu

C1, C2, C3, C4, C5 = (WORKLOADS[k] for k in ("c1", "c2", "c3", "c4", "c5"))

SMALL = {
    "bf16-gqa-causal-ragged": C3.with_(B=1, H=4, HKV=2, Sq=600, Sk=600, seed=11),
    "bf16-gqa-window": C4.with_(B=1, H=4, HKV=1, Sq=1000, Sk=1000, window=300, seed=12),
    "bf16-d64-causal": C3.with_(B=2, H=2, HKV=2, Sq=333, Sk=333, D=64, scale=1 / 8, seed=13),
    "bf16-noncausal-sq-ne-sk": C3.with_(B=1, H=2, HKV=1, Sq=257, Sk=390, causal=False, seed=14),
    "bf16-causal-sq-lt-sk": C3.with_(B=1, H=2, HKV=2, Sq=200, Sk=500, seed=15),
    "bf16-empty-rows": C3.with_(B=1, H=2, HKV=1, Sq=500, Sk=200, window=64, seed=16),
    "bf16-window1": C3.with_(B=1, H=2, HKV=2, Sq=260, Sk=260, window=1, seed=21),
    "bf16-s1": C3.with_(B=1, H=1, HKV=1, Sq=1, Sk=1, seed=17),
    "bf16-noncausal-window": C3.with_(B=1, H=2, HKV=2, Sq=384, Sk=384, causal=False,
                                      window=200, seed=22),
    "f32-c1": C1,
    "f32-causal-ragged": C2.with_(B=1, H=2, HKV=2, Sq=300, Sk=300, seed=18),
    "f32-noncausal": C5.with_(Sq=700, Sk=700, seed=19),
    "f32-gqa-window": C2.with_(B=1, H=4, HKV=2, Sq=450, Sk=450, window=100, seed=20),
    "f32-empty-rows": C2.with_(B=1, H=2, HKV=2, Sq=400, Sk=150, window=40, seed=23),
    # more work items than SMs: every persistent CTA runs several items, of mixed
    # lengths, some with one key tile and some with none
    "bf16-many-items-causal": C3.with_(B=1, H=96, HKV=24, Sq=700, Sk=700, seed=24),
    "bf16-many-items-empty": C3.with_(B=1, H=160, HKV=40, Sq=800, Sk=200, window=64, seed=25),
    "f32-many-items-causal": C2.with_(B=1, H=64, HKV=16, Sq=500, Sk=500, seed=26),
    "f32-many-items-empty": C2.with_(B=1, H=64, HKV=16, Sq=600, Sk=150, window=40, seed=27),
    # head dims below the kernels' 64 / 128 (the missing columns read as zeros)
    "bf16-d96-causal-gqa": C3.with_(B=1, H=4, HKV=2, Sq=333, Sk=333, D=96, scale=96 ** -0.5, seed=41),
    "bf16-d80-window": C4.with_(B=1, H=2, HKV=1, Sq=400, Sk=400, D=80, window=100, scale=80 ** -0.5,
                                seed=42),
    "bf16-d48-noncausal-sq-ne-sk": C3.with_(B=1, H=2, HKV=2, Sq=200, Sk=300, D=48, causal=False,
                                            scale=48 ** -0.5, seed=43),
    "bf16-d32-empty-rows": C3.with_(B=1, H=2, HKV=1, Sq=500, Sk=200, D=32, window=64,
                                    scale=32 ** -0.5, seed=44),
    "bf16-d16-causal": C3.with_(B=2, H=2, HKV=1, Sq=150, Sk=150, D=16, scale=0.25, seed=45),
    "f32-d48-window": C2.with_(B=1, H=2, HKV=1, Sq=260, Sk=260, D=48, window=60, scale=48 ** -0.5,
                               seed=46),
    "f32-d32-causal": C2.with_(B=1, H=2, HKV=2, Sq=200, Sk=200, D=32, scale=32 ** -0.5, seed=47),
    "f32-d16-noncausal": C5.with_(Sq=190, Sk=250, D=16, scale=0.25, seed=48),
    # short query sequences against long key sequences: fewer work items than SMs, so
    # each item's keys are split into ranges whose partial results are combined
    "bf16-decode-gqa": C3.with_(B=2, H=8, HKV=2, Sq=64, Sk=3000, causal=False, seed=51),
    "bf16-decode-causal-sq-lt-sk": C3.with_(B=1, H=4, HKV=2, Sq=130, Sk=2000, seed=52),
    "bf16-decode-d96": C3.with_(B=1, H=4, HKV=1, Sq=32, Sk=4000, D=96, causal=False,
                                scale=96 ** -0.5, seed=53),
    "f32-decode": C5.with_(Sq=100, Sk=4000, seed=54),
    # fp32 at D <= 64 with few items and long keys: two query tiles per item (two row
    # tiles of one head; two heads of one kv head), keys split into ranges
    "f32-two-tile-causal-ragged": C2.with_(B=1, H=2, HKV=1, Sq=700, Sk=2100, seed=91),
    "f32-two-tile-head-pairs-window": C2.with_(B=1, H=4, HKV=2, Sq=300, Sk=2500, window=700,
                                               causal=False, seed=92),
    # window ending before the keys do, with the dQ keys split into ranges: tile 10
    # sees only the last range, tile 11 no key at all (its dQ rows must come out 0)
    "bf16-decode-window-empty-tail": C4.with_(B=1, H=4, HKV=1, Sq=1500, Sk=1200, window=100,
                                              seed=55),
    # the decode-shaped measurement line's launch: 128 queries against 16384 keys, where
    # a few keys take almost all of a row's weight (max|dV| ~ 80 RMS(dV)); and a second
    # seed with Q, K ~ N(0, 2^2), more peaked still
    "bf16-decode-sq128-sk16384": C4.with_(Sq=128, causal=False, window=0, seed=56),
    "bf16-decode-sq128-sk16384-std2": C4.with_(Sq=128, causal=False, window=0, seed=57,
                                               std_qk=2.0),
    # forward items pair two query heads of a kv head when the group size is even
    # (three pairs per kv head here), else two row tiles of one head (group of 3)
    "bf16-gqa6-causal-ragged": C3.with_(B=1, H=12, HKV=2, Sq=300, Sk=300, seed=57),
    "bf16-gqa3-window-ragged": C4.with_(B=1, H=6, HKV=2, Sq=420, Sk=420, window=150, seed=58),
    "bf16-decode-gqa6": C3.with_(B=1, H=6, HKV=1, Sq=90, Sk=2600, causal=False, seed=59),
    "bf16-decode-gqa3": C3.with_(B=1, H=3, HKV=1, Sq=90, Sk=2600, causal=False, seed=60),
    # a single query row: many key ranges; causal (top-left) sees key 0 only, so every
    # range but the first is empty
    "bf16-decode-sq1": C3.with_(B=1, H=8, HKV=2, Sq=1, Sk=5000, causal=False, seed=61),
    "bf16-decode-sq1-causal": C3.with_(B=1, H=8, HKV=2, Sq=1, Sk=5000, seed=62),
    # at most 8 query rows per kv head (grouped heads x Sq) take the CUDA-core decode
    # kernel: 8 rows over 20000 keys; fp32 with Dv = 80 in the kernel built for 128
    # (8 rows), D = 32 causal (3 rows, key 0 only), a window narrower than Sq (8 rows)
    "bf16-decode-rows8-s20000": C3.with_(B=1, H=8, HKV=1, Sq=1, Sk=20000, causal=False,
                                         seed=63),
    "f32-decode-sq2-gqa4-d80": C5.with_(B=2, H=8, HKV=2, Sq=2, Sk=2500, D=80, scale=80 ** -0.5,
                                        seed=64),
    "f32-decode-sq1-d32-causal": C5.with_(H=3, Sq=1, Sk=777, D=32, scale=32 ** -0.5,
                                          causal=True, seed=65),
    "f32-decode-sq8-window3": C5.with_(Sq=8, Sk=3000, window=3, seed=66),
    # short key sequences: fewer (kv head, key tile) dK / dV items than SMs, so the bf16
    # backward splits the queries into ranges (partial dK, dV summed afterwards)
    "bf16-short-keys": C3.with_(B=1, H=4, HKV=1, Sq=3000, Sk=200, causal=False, seed=67),
    "bf16-short-keys-causal-window": C4.with_(B=1, H=4, HKV=2, Sq=2500, Sk=300, window=700,
                                              seed=68),
    "bf16-short-keys-d64-gqa": C3.with_(B=2, H=6, HKV=3, Sq=2048, Sk=64, D=64, scale=0.125,
                                        seed=69),
    # (fp32: the one-CTA-per-item dK / dV kernel splits below half the SMs)
    "f32-short-keys": C5.with_(Sq=3000, Sk=200, seed=70),
    "f32-short-keys-gqa-window": C2.with_(B=1, H=4, HKV=2, Sq=2000, Sk=256, window=500, seed=75),
    "f32-short-keys-d128": C5.with_(Sq=1500, Sk=130, D=128, scale=128 ** -0.5, seed=76),
    # bf16 inputs far outside fp16's range (largest finite 65504, normal from 2^-14):
    # the fp16 operand copies must be scaled by powers of two (gradients dO of 1e-7,
    # V of 1e5, Q and K of 2^-20, dO of 1e4 and V of 1e-6; alone and together)
    "bf16-mag-tiny-dO": C3.with_(B=1, H=4, HKV=2, Sq=300, Sk=300, seed=71, mag=(1, 1, 1, 1e-7)),
    "bf16-mag-huge-V": C3.with_(B=1, H=4, HKV=2, Sq=300, Sk=300, seed=72, mag=(1, 1, 1e5, 1)),
    "bf16-mag-tiny-QK": C3.with_(B=1, H=4, HKV=2, Sq=300, Sk=300, seed=73,
                                 mag=(2.0 ** -20, 2.0 ** -20, 1, 1)),
    "bf16-mag-all": C4.with_(B=1, H=4, HKV=1, Sq=700, Sk=700, window=200, seed=74,
                             mag=(2.0 ** -20, 2.0 ** -20, 1e5, 1e-7)),
    "bf16-mag-huge-dO-tiny-V": C3.with_(B=1, H=2, HKV=1, Sq=400, Sk=500, causal=False, seed=75,
                                        mag=(1, 1, 1e-6, 1e4)),
    "bf16-mag-decode": C3.with_(B=1, H=8, HKV=2, Sq=64, Sk=3000, causal=False, seed=76,
                                mag=(1, 1, 3e4, 1e-6)),
    # bf16 at D <= 32 runs in kernels built for D = 32 (64-byte rows and swizzle)
    "bf16-d32-causal-gqa-ragged": C3.with_(B=1, H=4, HKV=2, Sq=333, Sk=333, D=32,
                                           scale=32 ** -0.5, seed=91),
    "bf16-d32-window-sq-ne-sk": C4.with_(B=1, H=4, HKV=1, Sq=500, Sk=700, D=32, window=150,
                                         scale=32 ** -0.5, seed=92),
    "bf16-d32-decode": C4.with_(H=8, HKV=2, Sq=100, Sk=5000, D=32, causal=False, window=0,
                                scale=32 ** -0.5, seed=93),
    "bf16-d16-gqa3-noncausal": C3.with_(B=1, H=6, HKV=2, Sq=260, Sk=300, D=16, causal=False,
                                        scale=0.25, seed=94),
    # fp32 inputs at head dims above 64: two scaled fp16 terms per operand (3xTF32 tiles
    # would not fit shared memory there); D = 80 / 96 run in the D = 128 kernels
    "f32-d128-causal-ragged": C2.with_(B=1, H=2, HKV=2, Sq=300, Sk=300, D=128,
                                       scale=128 ** -0.5, seed=81),
    "f32-d128-gqa-window": C2.with_(B=1, H=4, HKV=2, Sq=450, Sk=450, D=128, window=100,
                                    scale=128 ** -0.5, seed=82),
    "f32-d96-noncausal-sq-ne-sk": C5.with_(Sq=257, Sk=390, D=96, scale=96 ** -0.5, seed=83),
    "f32-d80-empty-rows": C2.with_(B=1, H=2, HKV=1, Sq=400, Sk=150, D=80, window=40,
                                   scale=80 ** -0.5, seed=84),
    "f32-d128-decode": C5.with_(Sq=100, Sk=3000, D=128, scale=128 ** -0.5, seed=85),
    "f32-d128-many-items": C2.with_(B=1, H=64, HKV=16, Sq=300, Sk=300, D=128, scale=128 ** -0.5,
                                    seed=86),
    "f32-d128-mag": C2.with_(B=1, H=2, HKV=1, Sq=260, Sk=330, D=128, scale=128 ** -0.5, seed=87,
                             mag=(2.0 ** -20, 3.0, 1e5, 1e-7)),
}

# fp32 inputs at D = 128 at the multi-head causal workload's full size (B4 H8 S1024)
C2_D128 = C2.with_(D=128, scale=128 ** -0.5, name="causal-mha-b4-h8-s1024-d128-f32")
# bf16 at D = 32 at the GQA causal workload's full size (B2 H32/8 S4096)
C3_D32 = C3.with_(D=32, scale=32 ** -0.5, name="causal-gqa-b2-h32-hkv8-s4096-d32-bf16")


@pytest.fixture(scope="module")
def fa():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU parity tests need a CUDA device"
    from attention_fa_fwd_02_gb300 import fa as m
    return m


def _run(fa, w, q, k, v, out_dtype=None):
    dev = torch.device("cuda:0")
    qd, kd, vd = (t.to(dev) for t in (q, k, v))
    o, lse = fa.forward(qd, kd, vd, w.scale, w.causal, w.window, out_dtype=out_dtype)
    fa.check_device_status()
    return o, lse


def _check(w, o, lse, ro, rl, label):
    tol = TOL[w.dtype]
    eo = rms_err(to_np(o), ro)
    el = lse_err(to_np(lse), rl)
    assert eo <= tol["O"], f"{label}: O err {eo:.3e} > {tol['O']}"
    assert el <= tol["LSE"], f"{label}: LSE err {el:.3e} > {tol['LSE']}"
    return eo, el


@pytest.mark.parametrize("name", list(SMALL))
def test_forward_small(fa, name):
    w = SMALL[name]
    q, k, v, _ = make_inputs(w)
    o, lse = _run(fa, w, q, k, v)
    ro, rl = oracle.attention_fwd(q, k, v, w.scale, w.causal, w.window)
    _check(w, o, lse, ro, rl, name)


@pytest.mark.parametrize("name", ["bf16-gqa-causal-ragged", "bf16-decode-gqa",
                                  "bf16-decode-sq128-sk16384"])
def test_forward_deterministic(fa, name):
    # the decode cases split the keys into ranges (6 and 19) combined in range order
    w = SMALL[name]
    q, k, v, _ = make_inputs(w)
    o1, l1 = _run(fa, w, q, k, v)
    o2, l2 = _run(fa, w, q, k, v)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("name", ["bf16-gqa-causal-ragged", "bf16-decode-gqa",
                                  "bf16-d32-causal-gqa-ragged"])
def test_forward_bf16_output(fa, name):
    # bf16 outputs: rounding O to bf16 moves each element by at most half an ulp,
    # 2^-8 |O| (round to nearest, 8 significant bits). Allow that per element on top
    # of the fp32-output tolerance: |o - ref| <= 2^-8 |ref| + 2e-2 * RMS(ref). (The
    # decode case combines fp32 partial outputs of 6 key ranges and rounds once.)
    w = SMALL[name]
    q, k, v, _ = make_inputs(w)
    o, lse = _run(fa, w, q, k, v, out_dtype=torch.bfloat16)
    assert o.dtype == torch.bfloat16
    ro, rl = oracle.attention_fwd(q, k, v, w.scale, w.causal, w.window)
    got = to_np(o)
    excess = np.abs(got - ro) - 2.0 ** -8 * np.abs(ro)
    assert excess.max() <= 2e-2 * np.sqrt(np.mean(ro ** 2))
    assert lse_err(to_np(lse), rl) <= 1e-2


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("D", [64, 128])
def test_forward_decode_16_byte_aligned_inputs(fa, dtype, D):
    # the C ABI promises 16-byte alignment only: Q, K and V here start 16 bytes into
    # their allocations (torch's are 256-byte aligned), so the decode kernel's K rows
    # must be read 16 bytes per load instead of 32
    base = C3 if dtype == "bf16" else C5
    w = base.with_(B=2, H=8, HKV=2, Sq=1, Sk=3001, D=D, scale=D ** -0.5, causal=False,
                   window=700, seed=120 + D)
    q, k, v, _ = make_inputs(w)
    dev = torch.device("cuda:0")
    pad = 16 // q.element_size()

    def offset_copy(t):
        buf = torch.empty(t.numel() + pad, dtype=t.dtype, device=dev)
        view = buf[pad:].view(t.shape)
        view.copy_(t.to(dev))
        assert view.data_ptr() % 32 == 16 and view.is_contiguous()
        return view

    o, lse = fa.forward(offset_copy(q), offset_copy(k), offset_copy(v), w.scale, w.causal,
                        w.window)
    fa.check_device_status()
    ro, rl = oracle.attention_fwd(q, k, v, w.scale, w.causal, w.window)
    _check(w, o, lse, ro, rl, f"decode-16B-aligned-{dtype}-d{D}")


def test_forward_zero_keys(fa):
    w = C3.with_(B=1, H=2, HKV=1, Sq=130, Sk=0, seed=5)
    q = torch.randn(1, 2, 130, 128).to(torch.bfloat16).cuda()
    k = torch.empty(1, 1, 0, 128, dtype=torch.bfloat16, device="cuda")
    o, lse = fa.forward(q, k, k, w.scale, True, 0)
    fa.check_device_status()
    assert torch.all(o == 0) and torch.all(torch.isneginf(lse))


@pytest.mark.parametrize("cfg", ["c1", "c2", "c5", "c2-d128"])
def test_forward_full_config_fp32(fa, cfg):
    w = C2_D128 if cfg == "c2-d128" else WORKLOADS[cfg]
    q, k, v, _ = make_inputs(w)
    o, lse = _run(fa, w, q, k, v)
    ro, rl = oracle.attention_fwd(q, k, v, w.scale, w.causal, w.window)
    _check(w, o, lse, ro, rl, cfg)


@pytest.mark.parametrize("cfg,b,g", [("c3", 1, 5), ("c3", 0, 0), ("c4", 0, 3), ("c4", 0, 0),
                                     ("c3-d32", 1, 2)])
def test_forward_full_config_bf16_slice(fa, cfg, b, g):
    # Full-size launch (the benchmark's configuration); the oracle checks whole
    # (batch, kv-group) slices, which are independent of the rest.
    w = C3_D32 if cfg == "c3-d32" else WORKLOADS[cfg]
    q, k, v, _ = make_inputs(w)
    o, lse = _run(fa, w, q, k, v)
    rep = w.H // w.HKV
    hs = slice(g * rep, (g + 1) * rep)
    qs, ks, vs = q[b:b + 1, hs], k[b:b + 1, g:g + 1], v[b:b + 1, g:g + 1]
    ro, rl = oracle.attention_fwd(qs, ks, vs, w.scale, w.causal, w.window)
    _check(w, o[b:b + 1, hs], lse[b:b + 1, hs], ro, rl, f"{cfg} b{b} g{g}")
    # every other row must at least be finite and every LSE finite (no empty rows here)
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()
