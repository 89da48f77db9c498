#!/usr/bin/env python3
"""Benchmark of the attention hot path (fa_fwd + fa_bwd through the C ABI).

One step = one forward pass (fa_fwd) and one backward pass (fa_bwd) over one
batch of synthetic inputs of the workload (default: causal GQA attention, bf16
inputs, B=2 H=32 HKV=8 S=4096 D=128). Counted FLOPs follow the metric: forward
4*B*H*vis*D, backward 2.5x that, with vis the number of visible (query, key)
pairs per head. ``value`` is whole-job TFLOP/s with inputs resident in HBM;
``e2e`` is the same metric with host->device copies of Q/K/V/dO and
device->host copies of O/LSE/dQ/dK/dV inside the timed region.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload c3]
  python bench.py --impl reference ...   # the fp64 CPU oracle on the host cores

Under torchrun (N > 1) every rank runs its own independent problem (weak
scaling; no collective on the data path) and rank 0 prints the JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attention fwd/bwd TFLOP/s (H32/HKV8 S4096 D128 bf16 causal); % tensor peak"
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}
# Algorithmic FLOPs per visible (query, key) pair per query head, per kernel:
# forward 2 GEMMs (QK^T, PV); dK/dV kernel 4 (S^T, dP^T, dV, dK); dQ kernel 3 (S, dP, dQ).
# The materialised-dS backward's dQ GEMM: 1 (dS K).
KERNEL_FLOPS_PER_PAIR_PER_D = {"fa_fwd_kernel": 4, "fa_bwd_dkdv_kernel": 8, "fa_bwd_dq_kernel": 6,
                               "dq_from_ds_kernel": 2, "fa_decode_kernel": 4,
                               "fa_decode_bwd_kernel": 10}
# Source files whose change invalidates a committed DRAM-traffic figure.
_COMMON_SOURCES = ["ptx.cuh", "fa_common.cuh", "fa_epilogue.cuh", "fa_prepass.cuh"]
# head dim of each named workload (traffic figures in profiles/ are for these)
# fa_fwd's launches besides its kernel (operand conversion and scaling, the key-range combine)
FWD_AUX_KERNELS = ("cvt_bf16_to_f16(V)", "fwd_scales", "amax(Q,K,V)", "x16_split(Q,K,V)",
                   "split_tf32(Q,K,V)", "combine_splits")
WORKLOADS_D = {"c1": 64, "c2": 64, "c3": 128, "c4": 128, "c5": 64}
KERNEL_SOURCES = {"fa_fwd_kernel": ["fa_fwd.cu"] + _COMMON_SOURCES,
                  "fa_bwd_dkdv_kernel": ["fa_bwd.cu"] + _COMMON_SOURCES,
                  "fa_bwd_dq_kernel": ["fa_bwd.cu"] + _COMMON_SOURCES,
                  "bwd_prepass": ["fa_bwd.cu"] + _COMMON_SOURCES}


def _env_int(name, default):
    try:
        return int(os.environ.get(name, default))
    except ValueError:
        return default


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS if k in d}, "measured"
    except (OSError, ValueError, KeyError):
        return dict(FALLBACK_PEAKS), "fallback"


def tensor_peaks(peaks, dtype, f32_mma="f16x2"):
    """(burst, sustained) dense tensor peak in TFLOP/s of the tensor-core kind the path
    runs on: the measured bf16 figures for kind::f16 (bf16 inputs, and fp32 inputs as
    two fp16 terms), half of them for the tf32 products of the 3xTF32 path (the nominal
    tf32 / bf16 rate ratio). The burst figure is the roofline denominator for kernels of
    well under a second timed at full clocks; the sustained one (a seconds-long loop
    under the power cap) is reported beside it."""
    div = 2.0 if (dtype == "f32" and f32_mma == "tf32x3") else 1.0
    return peaks["bf16_tflops"] / div, peaks["bf16_tflops_sustained"] / div


def source_sha(kernel_base):
    h = hashlib.sha256()
    for f in KERNEL_SOURCES.get(kernel_base, []):
        with open(os.path.join(ROOT, "attention_fa_fwd_02_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def committed_traffic(kernel_base, workload):
    """DRAM bytes per launch from a committed ncu summary, if it matches the current source."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            entries = json.load(f)
    except (OSError, ValueError):
        return None
    for e in entries:
        if e.get("kernel") == kernel_base and e.get("workload") == workload:
            if e.get("source_sha") == source_sha(kernel_base):
                return e.get("bytes_per_launch")
    return None


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 25 ms while running."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self):
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "25", "-f", self.path], stdout=subprocess.DEVNULL,
                stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


def flops_for(w):
    from attention_fa_fwd_02_gb300.workloads import visible_pairs
    vis = visible_pairs(w)
    fwd = 4.0 * w.B * w.H * vis * w.D
    return fwd, 2.5 * fwd, vis


def pass_hbm_bytes(w, out_bytes):
    """Algorithmic HBM bytes of the forward and of the backward pass: every tensor a
    pass takes in read once, every tensor it hands out written once. Forward: Q, K, V
    in; O, LSE out. Backward: Q, K, V, O, dO, LSE in; dQ, dK, dV out. (in_bytes /
    out_bytes: element sizes of the inputs and of O, dQ, dK, dV; LSE is fp32.)"""
    in_bytes = 2 if w.dtype == "bf16" else 4
    nq = w.B * w.H * w.Sq * w.D
    nk = w.B * w.HKV * w.Sk * w.D
    rows = w.B * w.H * w.Sq
    fwd = in_bytes * (nq + 2 * nk) + out_bytes * nq + 4 * rows
    bwd = in_bytes * (2 * nq + 2 * nk) + out_bytes * nq + 4 * rows + out_bytes * (nq + 2 * nk)
    return fwd, bwd


def step_hbm_bytes(w, out_bytes):
    """Algorithmic HBM bytes of one fwd + bwd step (both passes of pass_hbm_bytes)."""
    return sum(pass_hbm_bytes(w, out_bytes))


# Kernels that do a whole pass in one launch and are bound by HBM (the decode shapes'
# CUDA-core kernels): their roofline is the pass's algorithmic bytes over the launch's
# time, against the copy bandwidth. Value: the pass (0 forward, 1 backward).
HBM_PASS_KERNELS = {"fa_decode_kernel": 0, "fa_decode_bwd_kernel": 1}


def hbm_roofline(kernel, nbytes, ms_per_launch, peaks, peak_src, traffic):
    """The roofline entry of an HBM-bound kernel: nbytes algorithmic bytes per launch over
    its average launch time, against the measured copy bandwidth."""
    gbs = nbytes / (ms_per_launch * 1e-3) / 1e9
    return {"bound": "hbm", "kernel": kernel, "achieved": round(gbs, 2), "peak": peaks["hbm_gbs"],
            "unit": "GB/s", "frac": round(gbs / peaks["hbm_gbs"], 4), "traffic": traffic,
            "bytes_per_launch": nbytes,
            "peak_source": ("measured HBM copy (MEASURED_PEAKS.json)" if peak_src == "measured"
                            else "fallback 6.8 TB/s copy")}


_INPUT_CACHE = {}


def oracle_sample(w, n_groups, batch=0):
    """Time the oracle (fwd + bwd) on the first n_groups kv groups of one batch element."""
    import oracle
    from attention_fa_fwd_02_gb300.workloads import make_inputs
    if w not in _INPUT_CACHE:
        _INPUT_CACHE.clear()
        _INPUT_CACHE[w] = make_inputs(w)
    q, k, v, do = _INPUT_CACHE[w]
    rep = w.H // w.HKV
    hs = slice(0, n_groups * rep)
    qs, ks, vs, dos = (q[batch:batch + 1, hs], k[batch:batch + 1, :n_groups],
                       v[batch:batch + 1, :n_groups], do[batch:batch + 1, hs])
    t0 = time.perf_counter()
    oracle.attention_fwd(qs, ks, vs, w.scale, w.causal, w.window)
    oracle.attention_bwd(qs, ks, vs, dos, w.scale, w.causal, w.window)
    dt = time.perf_counter() - t0
    fwd, bwd, _ = flops_for(w.with_(B=1, H=n_groups * rep, HKV=n_groups))
    return (fwd + bwd) / dt / 1e12, dt, oracle.num_threads(), n_groups * rep


def config_of(w, out_dtype="f32", extra=None, bwd="recompute", f32_mma="f16x2"):
    c = {"workload": w.name, "B": w.B, "H": w.H, "HKV": w.HKV, "Sq": w.Sq, "Sk": w.Sk, "D": w.D,
         "causal": bool(w.causal), "window": w.window, "scale": w.scale, "in_dtype": w.dtype,
         "out_dtype": out_dtype, "backward": bwd,
         "l2": "256 MiB memset between timed steps; inputs also exceed L2"}
    if w.dtype == "f32":
        c["f32_mma"] = f32_mma
    if extra:
        c.update(extra)
    return c


def workload_of(args):
    """The named workload, with another head dim (scale 1/sqrt(D)) if --head-dim is given."""
    from attention_fa_fwd_02_gb300.workloads import WORKLOADS
    w = WORKLOADS[args.workload]
    if args.head_dim and args.head_dim != w.D:
        w = w.with_(D=args.head_dim, scale=args.head_dim ** -0.5,
                    name=w.name.replace(f"-d{w.D}-", f"-d{args.head_dim}-"))
    if args.sq and args.sq != w.Sq:  # short query sequence against the same keys
        w = w.with_(Sq=args.sq, name=f"{w.name}-sq{args.sq}")
    if args.sk and args.sk != w.Sk:  # short key sequence for the same queries
        w = w.with_(Sk=args.sk, name=f"{w.name}-sk{args.sk}")
    if args.non_causal and w.causal:
        w = w.with_(causal=False, window=0, name=f"{w.name}-noncausal")
    return w


# ------------------------------------------------------------------ reference arm
def run_reference(args, rank, world):
    if rank != 0:
        return 0
    w = workload_of(args)
    # each step: one whole (batch, kv-group) slice of the workload through the oracle
    for _ in range(args.warmup):
        oracle_sample(w, 1)
    vals, times = [], []
    cores = 1
    for _ in range(args.steps):
        v, dt, cores, heads = oracle_sample(w, 1)
        vals.append(v)
        times.append(dt)
    value = statistics.mean(vals)
    ms = statistics.mean(times) * 1e3
    sample = (f"one (batch, kv-group) slice per step: {w.H // w.HKV} query heads of "
              f"{w.B * w.H}, full sequence, fwd+bwd in fp64")
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config_of(w, args.out_dtype, bwd=args.bwd, f32_mma=args.f32_mma),
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": cores,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ ranks
# Under torchrun every rank runs an independent problem of the same shape (the
# path partitions by batch / kv group with no exchange), so the only cross-rank
# operations are a barrier around the timed region and a max-reduce of the time.
def rank_workload(w, rank):
    """The workload a rank runs: same shape, its own seed."""
    return w.with_(seed=w.seed + 7919 * rank)


def max_over_ranks(value, dist, device=None):
    """Max of a per-rank float over the process group (identity without one)."""
    if dist is None:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(flops_per_rank, world, ms_max):
    """Aggregate throughput: every rank's work over the slowest rank's time."""
    return world * flops_per_rank / (ms_max * 1e-3) / 1e12


# ------------------------------------------------------------------ our arm
def run_ours(args, rank, world, local_rank):
    import torch
    import __graft_entry__
    __graft_entry__.build_library()
    from attention_fa_fwd_02_gb300 import fa
    from attention_fa_fwd_02_gb300.workloads import make_inputs

    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    w = workload_of(args)
    wr = rank_workload(w, rank)
    q, k, v, do = make_inputs(wr)
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    odt = torch.bfloat16 if args.out_dtype == "bf16" else torch.float32
    p = fa.make_params(qd, kd, w.scale, w.causal, w.window, out_dtype=odt, f32_mma=args.f32_mma)
    o = torch.empty(q.shape, dtype=odt, device=dev)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
    dq = torch.empty(q.shape, dtype=odt, device=dev)
    dk = torch.empty(k.shape, dtype=odt, device=dev)
    dv = torch.empty(v.shape, dtype=odt, device=dev)
    stream = torch.cuda.current_stream()
    sh = int(stream.cuda_stream)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    # the backward entry point: fa_bwd, or the materialised-dS variant
    bwd_entry = fa.fa_bwd_dsmat if args.bwd == "dsmat" else fa.fa_bwd

    def step():
        rc = fa.fa_fwd(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(), lse.data_ptr(), p, sh)
        if rc:
            raise fa.FAError(rc, "fa_fwd")
        rc = bwd_entry(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(), dod.data_ptr(),
                       lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), p, sh)
        if rc:
            raise fa.FAError(rc, "fa_bwd")

    def barrier():
        if dist is not None:
            dist.barrier()

    for _ in range(args.warmup):
        flush.zero_()
        step()
    fa.check_device_status()

    # ---- device-resident timed region
    sampler = ClockSampler() if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    barrier()
    torch.cuda.synchronize()
    for s, e in ev:
        flush.zero_()
        s.record(stream)
        step()
        e.record(stream)
    torch.cuda.synchronize()
    barrier()
    clocks = sampler.stop() if sampler else None
    fa.check_device_status()
    ms = statistics.mean(s.elapsed_time(e) for s, e in ev)
    ms_max = max_over_ranks(ms, dist, dev)

    # ---- per-kernel times: the same steps again with a CUDA event pair around every
    # library kernel, on the stream it runs on. These events also order the dQ kernel
    # after dK / dV (without them it starts on the SMs dK / dV's last wave leaves idle),
    # so the step time above comes from the pass without them.
    barrier()
    torch.cuda.synchronize()
    fa.fa_timing_enable(True)
    for _ in range(args.steps):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    kernels = fa.fa_timing_read()
    fa.fa_timing_enable(False)
    fa.check_device_status()

    # ---- end to end through host buffers (pinned), copies inside the timed region.
    # Every step copies its inputs in from pinned host memory and all its results
    # (O, LSE, dQ, dK, dV) out, the way a caller streaming many problems would: two
    # sets of device buffers, inputs in on one copy stream, results out on another,
    # the library on the compute stream, events ordering each set's reuse -- so one
    # step's transfers overlap its neighbours' compute.
    hq, hk, hv, hdo = (t.pin_memory() for t in (q, k, v, do))
    n_sets = 2
    dsets = [dict(q=qd, k=kd, v=vd, do=dod, o=o, lse=lse, dq=dq, dk=dk, dv=dv)]
    dsets += [{n: torch.empty_like(t) for n, t in dsets[0].items()} for _ in range(n_sets - 1)]
    hsets = [{n: torch.empty(dsets[0][n].shape, dtype=dsets[0][n].dtype, pin_memory=True)
              for n in ("o", "lse", "dq", "dk", "dv")} for _ in range(n_sets)]
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hdo))
    d2h = sum(t.numel() * t.element_size() for t in hsets[0].values())
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    done_cmp, done_out = [None] * n_sets, [None] * n_sets

    def fwd_call(b):
        rc = fa.fa_fwd(b["q"].data_ptr(), b["k"].data_ptr(), b["v"].data_ptr(), b["o"].data_ptr(),
                       b["lse"].data_ptr(), p, sh)
        if rc:
            raise fa.FAError(rc, "fa_fwd")
        ev_fwd = torch.cuda.Event()
        ev_fwd.record(stream)
        return ev_fwd

    def e2e_step(i):
        j = i % n_sets
        b, hb = dsets[j], hsets[j]
        if done_cmp[j] is not None:  # the inputs of set j were last read by that compute
            s_in.wait_event(done_cmp[j])
        with torch.cuda.stream(s_in):
            for n, src in (("q", hq), ("k", hk), ("v", hv)):
                b[n].copy_(src, non_blocking=True)
            ev_qkv = torch.cuda.Event()
            ev_qkv.record(s_in)
            b["do"].copy_(hdo, non_blocking=True)
            ev_do = torch.cuda.Event()
            ev_do.record(s_in)
        stream.wait_event(ev_qkv)
        if done_out[j] is not None:  # the outputs of set j were last read by those copies
            stream.wait_event(done_out[j])
        ev_fwd = fwd_call(b)
        stream.wait_event(ev_do)
        rc = bwd_entry(b["q"].data_ptr(), b["k"].data_ptr(), b["v"].data_ptr(), b["o"].data_ptr(),
                       b["do"].data_ptr(), b["lse"].data_ptr(), b["dq"].data_ptr(),
                       b["dk"].data_ptr(), b["dv"].data_ptr(), p, sh)
        if rc:
            raise fa.FAError(rc, "fa_bwd")
        ev_bwd = torch.cuda.Event()
        ev_bwd.record(stream)
        done_cmp[j] = ev_bwd
        s_out.wait_event(ev_fwd)
        with torch.cuda.stream(s_out):
            hb["o"].copy_(b["o"], non_blocking=True)
            hb["lse"].copy_(b["lse"], non_blocking=True)
        s_out.wait_event(ev_bwd)
        with torch.cuda.stream(s_out):
            for n in ("dq", "dk", "dv"):
                hb[n].copy_(b[n], non_blocking=True)
            ev_out = torch.cuda.Event()
            ev_out.record(s_out)
        done_out[j] = ev_out
        return ev_out

    for i in range(max(n_sets, args.warmup // 2)):
        e2e_step(i)
    torch.cuda.synchronize()
    done_cmp, done_out = [None] * n_sets, [None] * n_sets
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    t_start.record(stream)
    s_in.wait_event(t_start)
    s_out.wait_event(t_start)
    last = None
    for i in range(args.steps):
        last = e2e_step(i)
    stream.wait_event(last)
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier()
    fa.check_device_status()
    ms_e2e = max_over_ranks(t_start.elapsed_time(t_end) / args.steps, dist, dev)

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return 0

    fwd_fl, bwd_fl, vis = flops_for(w)
    value = whole_job_tflops(fwd_fl + bwd_fl, world, ms_max)
    peaks, peak_src = load_peaks()
    peak, peak_sus = tensor_peaks(peaks, w.dtype, args.f32_mma)
    per_kernel = {}
    fwd_ms = 0.0
    launches = 0
    for name, (n, tot) in kernels.items():
        launches += n
        base = name.split("<")[0]
        entry = {"launches": n, "ms_per_launch": tot / n}
        if base in KERNEL_FLOPS_PER_PAIR_PER_D:
            fl = KERNEL_FLOPS_PER_PAIR_PER_D[base] * w.B * w.H * vis * w.D
            entry["tflops"] = fl / (tot / n * 1e-3) / 1e12
        per_kernel[name] = entry
        if base.startswith("fa_fwd") or base == "fa_decode_kernel" or name in FWD_AUX_KERNELS:
            fwd_ms += tot / n
    dom = max((k_ for k_ in per_kernel if "tflops" in per_kernel[k_]),
              key=lambda k_: per_kernel[k_]["launches"] * per_kernel[k_]["ms_per_launch"])
    dom_base = dom.split("<")[0]
    achieved = per_kernel[dom]["tflops"]
    traffic = (committed_traffic(dom_base, args.workload)
               if w.D == WORKLOADS_D[args.workload] and args.out_dtype == "f32" and not args.sq
               and not args.sk
               and not args.non_causal and args.f32_mma == "f16x2" and args.bwd == "recompute"
               else None)
    cpu = None
    if not args.no_cpu_baseline:
        # every kv group of batch element 0: ~10 s of oracle work on the 16 host cores at C3
        groups = w.HKV
        cv, cdt, cores, heads = oracle_sample(w, groups)
        cpu = {"value": round(cv, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
               "sample": (f"batch 0, kv groups 0..{groups - 1} ({heads} of {w.B * w.H} query "
                          f"heads, full sequence), fwd+bwd in fp64, {cdt:.1f} s")}
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_max, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
        "data": "synthetic", "config": config_of(w, args.out_dtype, bwd=args.bwd, f32_mma=args.f32_mma),
        "fwd_tflops": round(fwd_fl / (fwd_ms * 1e-3) / 1e12, 3) if fwd_ms else None,
        # the backward's share of the step: step time minus the forward kernels' time
        # (its dK / dV and dQ kernels overlap inside the step)
        "bwd_tflops": (round(bwd_fl / ((ms - fwd_ms) * 1e-3) / 1e12, 3)
                       if world == 1 and ms > fwd_ms else None),
        "pct_tensor_peak": round(100 * value / world / peak, 2),
        "roofline": {"bound": "tensor", "kernel": dom, "achieved": round(achieved, 2),
                     "peak": peak, "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                     "traffic": traffic,
                     "peak_source": (f"{peak_src} bf16 burst (MEASURED_PEAKS.json)"
                                     if peak_src == "measured" else "fallback 1.9 PFLOP/s burst")
                     + ("" if w.dtype == "bf16" else
                        " x 1/2, the nominal tf32 / bf16 rate ratio; 3 products per GEMM"
                        if args.f32_mma == "tf32x3" else " (kind::f16); 3 products per GEMM"),
                     "peak_sustained": peak_sus, "frac_sustained": round(achieved / peak_sus, 4)}
        if dom_base not in HBM_PASS_KERNELS else
        hbm_roofline(dom, pass_hbm_bytes(w, 2 if args.out_dtype == "bf16" else 4)[HBM_PASS_KERNELS[dom_base]],
                     per_kernel[dom]["ms_per_launch"], peaks, peak_src, traffic),
        "kernels": {k_: {kk: (round(vv, 4) if isinstance(vv, float) else vv)
                         for kk, vv in e.items()} for k_, e in per_kernel.items()},
        "e2e": {"value": round(whole_job_tflops(fwd_fl + bwd_fl, world, ms_e2e), 3),
                "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": launches,
        "clocks": clocks,
        "cpu_baseline": cpu,
    }
    # the step's algorithmic HBM traffic over its time: what a latency-bound case (small
    # shapes) reaches against the copy bandwidth
    hbm_b = step_hbm_bytes(w, 2 if args.out_dtype == "bf16" else 4)
    gbs = hbm_b * world / (ms_max * 1e-3) / 1e9
    line["hbm"] = {"bytes_per_step": hbm_b, "achieved": round(gbs, 2), "peak": peaks["hbm_gbs"],
                   "unit": "GB/s", "frac": round(gbs / world / peaks["hbm_gbs"], 4)}
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="c3", choices=["c1", "c2", "c3", "c4", "c5"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sq", type=int, default=None,
                    help="query rows per head (measurement lines, e.g. decode-shaped)")
    ap.add_argument("--sk", type=int, default=None,
                    help="key rows per kv head (measurement lines, e.g. short key sequences)")
    ap.add_argument("--non-causal", action="store_true",
                    help="full attention over the keys (measurement lines)")
    ap.add_argument("--out-dtype", choices=["f32", "bf16"], default="f32",
                    help="dtype of O, dQ, dK, dV (measurement lines; the headline is f32)")
    ap.add_argument("--bwd", choices=["recompute", "dsmat"], default="recompute",
                    help="backward route: fa_bwd (recomputes S and dP for dQ) or fa_bwd_dsmat "
                         "(materialised dS; measurement lines)")
    ap.add_argument("--f32-mma", choices=["f16x2", "tf32x3"], default="f16x2",
                    help="fp32 workloads: tensor-core terms (two scaled fp16 terms per operand, "
                         "or 3xTF32 for head dims up to 64)")
    ap.add_argument("--head-dim", type=int, default=None,
                    help="run the workload with another head dim (measurement lines; the "
                         "headline is the workload's own)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    rank = _env_int("RANK", 0)
    world = _env_int("WORLD_SIZE", 1)
    local_rank = _env_int("LOCAL_RANK", 0)
    if args.impl == "reference":
        return run_reference(args, rank, world)
    return run_ours(args, rank, world, local_rank)


if __name__ == "__main__":
    sys.exit(main())
