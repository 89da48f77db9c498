"""fa_fwd and fa_bwd inside a CUDA graph.

A caller that runs the same attention shapes over and over captures the calls once
and replays the graph. The library's stream-ordered scratch (pool allocations) and
the kernels' programmatic dependent launches (the dQ kernel after dK/dV; the fp32
path's chains; the key- and query-range sums) must both survive capture; every replay must recompute all outputs (they are overwritten with NaN
before each replay) and match eager calls bit for bit -- the kernels are
deterministic (dK/dV without atomics; the dQ items each computed by one CTA).
"""
import pytest
import torch

from attention_fa_fwd_02_gb300.workloads import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu

CASES = {
    "bf16-causal-gqa": WORKLOADS["c3"].with_(B=1, H=8, HKV=2, Sq=700, Sk=700, seed=31),
    "bf16-window": WORKLOADS["c4"].with_(B=1, H=4, HKV=1, Sq=900, Sk=900, window=200, seed=33),
    "f32-causal": WORKLOADS["c2"].with_(B=1, H=4, HKV=2, Sq=300, Sk=300, seed=32),
    # short queries: forward and dQ split the keys into ranges (scratch for the partial
    # results allocated and freed inside the graph)
    "bf16-decode": WORKLOADS["c3"].with_(B=1, H=4, HKV=2, Sq=100, Sk=2500, causal=False, seed=34),
    # fp32 through the 3xTF32 kernels, and at D = 128 with keys split into ranges (the
    # fp32 kernels run as chains of programmatic dependent launches)
    "f32-tf32x3": WORKLOADS["c2"].with_(B=1, H=4, HKV=2, Sq=300, Sk=300, seed=35),
    "f32-d128-decode": WORKLOADS["c5"].with_(Sq=100, Sk=3000, D=128, scale=128 ** -0.5, seed=36),
    # decode shapes (at most 8 query rows per kv head): the CUDA-core kernels, their
    # key-range partials and the fixed-order merges launched as programmatic dependents
    "bf16-decode-sq1": WORKLOADS["c3"].with_(B=1, H=8, HKV=2, Sq=1, Sk=5000, causal=False,
                                             seed=37),
    "f32-decode-sq2": WORKLOADS["c5"].with_(Sq=2, Sk=3000, seed=38),
    # short key sequences: the dK / dV items split the queries into ranges, summed after dQ
    "bf16-short-keys": WORKLOADS["c3"].with_(B=1, H=4, HKV=1, Sq=3000, Sk=200, causal=False,
                                             seed=39),
}
MMA = {"f32-tf32x3": "tf32x3"}


@pytest.fixture(scope="module")
def fa():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from attention_fa_fwd_02_gb300 import fa as m
    return m


@pytest.mark.parametrize("name", list(CASES))
def test_graph_replay_matches_eager(fa, name):
    w = CASES[name]
    mma = MMA.get(name, "f16x2")
    q, k, v, do = (t.cuda() for t in make_inputs(w))
    o, lse = fa.forward(q, k, v, w.scale, w.causal, w.window, f32_mma=mma)
    dq, dk, dv = fa.backward(q, k, v, o, lse, do, w.scale, w.causal, w.window, f32_mma=mma)
    torch.cuda.synchronize()
    fa.check_device_status()

    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(graph, stream=side):
        go, glse = fa.forward(q, k, v, w.scale, w.causal, w.window, f32_mma=mma)
        gdq, gdk, gdv = fa.backward(q, k, v, go, glse, do, w.scale, w.causal, w.window, f32_mma=mma)
    torch.cuda.synchronize()
    for _ in range(3):
        for t in (go, glse, gdq, gdk, gdv):
            t.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        fa.check_device_status()
        for got, ref, n in ((go, o, "O"), (glse, lse, "LSE"), (gdq, dq, "dQ"), (gdk, dk, "dK"),
                            (gdv, dv, "dV")):
            assert torch.equal(got, ref), f"{name}: graph replay {n} differs from the eager call"
