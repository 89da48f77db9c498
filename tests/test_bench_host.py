"""Host-side logic of bench.py: the metric's FLOP accounting, the workload variants
its options select, and the DRAM-traffic lookup that feeds the roofline line."""
import itertools
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from attention_fa_fwd_02_gb300.workloads import WORKLOADS, visible_pairs  # noqa: E402


def _brute_visible(w):
    n = 0
    for i in range(w.Sq):
        for j in range(w.Sk):
            if w.causal and j > i:
                continue
            if w.window > 0 and j < i - w.window + 1:
                continue
            n += 1
    return n


@pytest.mark.parametrize("sq,sk,causal,window", list(itertools.product(
    [1, 7, 64, 130], [1, 9, 64, 200], [False, True], [0, 1, 5, 100])))
def test_visible_pairs_match_enumeration(sq, sk, causal, window):
    w = WORKLOADS["c3"].with_(Sq=sq, Sk=sk, causal=causal, window=window)
    assert visible_pairs(w) == _brute_visible(w)


def test_visible_fractions_and_flops_of_the_five_workloads():
    # closed forms: causal S x S has S (S + 1) / 2 visible pairs; a causal window w
    # adds w (w + 1) / 2 for the first w rows and w for each later row; non-causal S^2.
    def causal(s):
        return s * (s + 1) // 2

    def windowed(s, w):
        return w * (w + 1) // 2 + (s - w) * w
    expect = {"c1": causal(128), "c2": causal(1024), "c3": causal(4096),
              "c4": windowed(16384, 4096), "c5": 16384 * 16384}
    # the fractions and forward GFLOP the problem statement's table gives
    table = {"c1": (0.503906, 0.00211), "c2": (0.500488, 4.299), "c3": (0.500122, 274.95),
             "c4": (0.218758, 481.05), "c5": (1.0, 68.72)}
    for name, w in WORKLOADS.items():
        fwd, bwd, vis = bench.flops_for(w)
        assert vis == expect[name]
        frac, gflop = table[name]
        assert vis / (w.Sq * w.Sk) == pytest.approx(frac, abs=1e-6)
        assert fwd / 1e9 == pytest.approx(gflop, rel=3e-3)
        assert bwd == pytest.approx(2.5 * fwd)


class _Args:
    def __init__(self, workload="c3", head_dim=None, sq=None, non_causal=False, sk=None):
        self.workload, self.head_dim, self.sq, self.non_causal = workload, head_dim, sq, non_causal
        self.sk = sk


def test_workload_options():
    assert bench.workload_of(_Args()) == WORKLOADS["c3"]
    w = bench.workload_of(_Args(head_dim=64))
    assert (w.D, w.scale) == (64, 64 ** -0.5) and w.Sq == WORKLOADS["c3"].Sq
    w = bench.workload_of(_Args(workload="c4", sq=128, non_causal=True))
    assert (w.Sq, w.Sk, w.causal, w.window) == (128, 16384, False, 0)
    assert "sq128" in w.name and "noncausal" in w.name
    w = bench.workload_of(_Args(workload="c4", sk=256))
    assert (w.Sq, w.Sk) == (16384, 256) and "sk256" in w.name


def test_traffic_is_reported_only_for_the_sources_it_was_measured_on(monkeypatch):
    # a committed ncu figure is used only while the kernel's sources hash to the value
    # recorded with it (after a kernel change the roofline line reports null)
    entries = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))
    assert {e["kernel"] for e in entries} >= {"fa_fwd_kernel", "fa_bwd_dkdv_kernel",
                                              "fa_bwd_dq_kernel", "bwd_prepass"}
    recorded = {e["kernel"]: e for e in entries if e["workload"] == "c3"}
    monkeypatch.setattr(bench, "source_sha", lambda k: recorded[k]["source_sha"])
    for k, e in recorded.items():
        assert bench.committed_traffic(k, "c3") == e["bytes_per_launch"]
    assert bench.committed_traffic("fa_bwd_dkdv_kernel", "c4") is None
    monkeypatch.setattr(bench, "source_sha", lambda k: "0" * 16)
    assert bench.committed_traffic("fa_bwd_dkdv_kernel", "c3") is None


def test_source_hash_covers_the_kernel_sources():
    for k in ("fa_fwd_kernel", "fa_bwd_dkdv_kernel", "fa_bwd_dq_kernel", "bwd_prepass"):
        h = bench.source_sha(k)
        assert len(h) == 16 and int(h, 16) >= 0
    assert bench.source_sha("fa_fwd_kernel") != bench.source_sha("fa_bwd_dkdv_kernel")


def test_step_hbm_bytes_counts_each_tensor_once():
    from attention_fa_fwd_02_gb300.workloads import WORKLOADS
    w = WORKLOADS["c1"]  # fp32 B1 H1 S128 D64: every tensor 128 x 64 x 4 bytes, LSE 512
    t = 128 * 64 * 4
    # fwd: Q, K, V in, O out, LSE out; bwd: Q, K, V, O, dO in, LSE in, dQ, dK, dV out
    assert bench.step_hbm_bytes(w, 4) == (4 * t + 512) + (8 * t + 512)
    c3 = WORKLOADS["c3"]  # bf16 inputs, fp32 or bf16 outputs
    nq, nk, rows = 2 * 32 * 4096 * 128, 2 * 8 * 4096 * 128, 2 * 32 * 4096
    f32 = bench.step_hbm_bytes(c3, 4)
    assert f32 == 2 * (nq + 2 * nk) + 4 * nq + 4 * rows + 2 * (2 * nq + 2 * nk) + 4 * nq + 4 * rows \
        + 4 * (nq + 2 * nk)
    assert bench.step_hbm_bytes(c3, 2) == f32 - 2 * (2 * nq + nq + 2 * nk)


def test_decode_kernels_take_the_hbm_roofline_of_their_pass():
    # the decode shapes' kernels each do a whole pass in one launch: forward = Q, K, V in,
    # O, LSE out; backward = Q, K, V, O, dO, LSE in, dQ, dK, dV out
    from attention_fa_fwd_02_gb300.workloads import WORKLOADS
    w = WORKLOADS["c4"].with_(Sq=1, causal=False, window=0)  # bf16 B1 H16/HKV4 Sk 16384 D128
    nq, nk, rows = 16 * 128, 4 * 16384 * 128, 16
    fwd, bwd = bench.pass_hbm_bytes(w, 4)
    assert fwd == 2 * (nq + 2 * nk) + 4 * nq + 4 * rows
    assert bwd == 2 * (2 * nq + 2 * nk) + 4 * nq + 4 * rows + 4 * (nq + 2 * nk)
    assert fwd + bwd == bench.step_hbm_bytes(w, 4)
    assert set(bench.HBM_PASS_KERNELS) == {"fa_decode_kernel", "fa_decode_bwd_kernel"}
    peaks = {"bf16_tflops": 1965.9, "bf16_tflops_sustained": 1727.6, "hbm_gbs": 6795.1}
    r = bench.hbm_roofline("fa_decode_kernel", fwd, 0.02, peaks, "measured", None)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] == 6795.1
    assert abs(r["achieved"] - fwd / 20e-6 / 1e9) < 0.01
    assert abs(r["frac"] - r["achieved"] / 6795.1) < 1e-4


def test_roofline_denominator_is_the_burst_peak():
    # the kernels are timed for well under a second at full clocks: the burst cuBLAS
    # figure is their denominator, the power-capped sustained one is reported beside it
    peaks = {"bf16_tflops": 1965.9, "bf16_tflops_sustained": 1727.6, "hbm_gbs": 6795.1}
    assert bench.tensor_peaks(peaks, "bf16") == (1965.9, 1727.6)
    # fp32 inputs: two fp16 terms run at the kind::f16 rate, 3xTF32 at the tf32 rate
    assert bench.tensor_peaks(peaks, "f32") == (1965.9, 1727.6)
    assert bench.tensor_peaks(peaks, "f32", "tf32x3") == (1965.9 / 2, 1727.6 / 2)
