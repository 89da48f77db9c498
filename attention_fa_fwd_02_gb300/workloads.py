"""Seeded synthetic workloads for the attention path.

This module holds only shapes, dtypes, value distributions and seeds -- none of
the attention arithmetic. It is the one module that both the fp64 oracle's tests
and the CUDA path's tests/benchmark draw inputs from, so the two sides see
bit-identical tensors.

The five workloads mirror the problem statements the source pages work with:
causal single- and multi-head fp32 attention (rustytorch
"flash_attention_forward.metal"; forge "flash_attention.metal", head_dim 64),
grouped-query attention with a sliding window (forge FlashParams: H, HKV,
window; boostr "flash.wgsl" FlashParams: num_kv_heads, window_size), and a long
non-causal single head. The pages use no public dataset; all values are drawn
from the stated distributions.

Draw order is fixed: Q, K, V, dO from one CPU ``torch.Generator`` seeded with
``seed``, in fp32, each multiplied by its ``mag`` factor (1 unless stated), then
cast (round-to-nearest-even) to the workload dtype.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    HKV: int
    Sq: int
    Sk: int
    D: int
    scale: float
    causal: bool
    window: int            # 0 = full attention; else keys j >= i - window + 1 (self included)
    dtype: str             # "f32" or "bf16": dtype of Q, K, V, dO
    dist: str              # "normal" or "uniform"
    std_qk: float = 1.0    # std of Q and K for "normal"
    seed: int = 0
    # multipliers of the Q, K, V, dO draws (applied in fp32 before the cast): inputs of
    # very large or very small magnitude, as gradients dO often are
    mag: tuple = (1.0, 1.0, 1.0, 1.0)

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.float32 if self.dtype == "f32" else torch.bfloat16


WORKLOADS = {
    "c1": Workload("causal-mha-b1-h1-s128-d64-f32", 1, 1, 1, 128, 128, 64, 1 / 8, True, 0,
                   "f32", "normal", 1.0, 1001),
    "c2": Workload("causal-mha-b4-h8-s1024-d64-f32", 4, 8, 8, 1024, 1024, 64, 1 / math.sqrt(64),
                   True, 0, "f32", "normal", 1.0, 1002),
    "c3": Workload("causal-gqa-b2-h32-hkv8-s4096-d128-bf16", 2, 32, 8, 4096, 4096, 128,
                   1 / math.sqrt(128), True, 0, "bf16", "normal", 1.0, 1003),
    "c4": Workload("window4096-causal-gqa-b1-h16-hkv4-s16384-d128-bf16", 1, 16, 4, 16384, 16384,
                   128, 1 / math.sqrt(128), True, 4096, "bf16", "normal", 1.5, 1004),
    "c5": Workload("noncausal-mha-b1-h1-s16384-d64-f32", 1, 1, 1, 16384, 16384, 64,
                   1 / math.sqrt(64), False, 0, "f32", "uniform", 1.0, 1005),
}


def make_inputs(w: Workload):
    """Return CPU tensors (q, k, v, do) in the workload dtype, contiguous [B, heads, S, D]."""
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed)
    shapes = [(w.B, w.H, w.Sq, w.D), (w.B, w.HKV, w.Sk, w.D), (w.B, w.HKV, w.Sk, w.D),
              (w.B, w.H, w.Sq, w.D)]
    out = []
    for idx, shp in enumerate(shapes):
        if w.dist == "normal":
            t = torch.randn(shp, generator=g, dtype=torch.float32)
            if idx < 2 and w.std_qk != 1.0:
                t = t * w.std_qk
        elif w.dist == "uniform":
            t = torch.rand(shp, generator=g, dtype=torch.float32) * 2.0 - 1.0
        else:
            raise ValueError(f"unknown distribution {w.dist}")
        if w.mag[idx] != 1.0:
            t = t * w.mag[idx]
        out.append(t.to(w.torch_dtype).contiguous())
    return tuple(out)


def visible_pairs(w: Workload) -> int:
    """Count of (i, j) pairs that a query row may attend to, per head (the mask rule
    restated from the pages' problem statement; used only for FLOP accounting)."""
    total = 0
    for i in range(w.Sq):
        hi = min(i, w.Sk - 1) if w.causal else w.Sk - 1
        lo = max(0, i - w.window + 1) if w.window > 0 else 0
        if hi >= lo:
            total += hi - lo + 1
    return total
