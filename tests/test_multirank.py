"""The multi-rank (torchrun) path of bench.py on CPU with the gloo backend.

The attention path shards by independent problems, so N ranks run N replicas:
each rank draws its own problem, a barrier brackets the timed region, and the
reported value is every rank's work over the slowest rank's time. These tests
run those host-side pieces in a world of two gloo processes.
"""
import os
import socket
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        from attention_fa_fwd_02_gb300.workloads import WORKLOADS, make_inputs
        w = bench.rank_workload(WORKLOADS["c1"], rank)
        q, k, v, do = make_inputs(w)
        digest = float(q.double().sum() + 3 * k.double().sum() + 5 * v.double().sum())
        dist.barrier()
        t_rank = 10.0 + 7.5 * rank             # a per-rank step time in ms
        t_max = bench.max_over_ranks(t_rank, dist)
        fl = 4.0 * 1e9
        out[rank] = (digest, t_max, bench.whole_job_tflops(fl, world, t_max), w.seed)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_replicas_and_max_reduce():
    world = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, port, out), nprocs=world, join=True,
                       start_method="spawn")
    (d0, t0, v0, s0), (d1, t1, v1, s1) = out[0], out[1]
    assert s0 != s1 and d0 != d1                  # independent problems per rank
    assert t0 == t1 == 17.5                       # both ranks see the slowest time
    assert v0 == v1 == pytest.approx(2 * 4.0e9 / 17.5e-3 / 1e12)


def test_single_rank_helpers_without_process_group():
    sys.path.insert(0, ROOT)
    import bench
    from attention_fa_fwd_02_gb300.workloads import WORKLOADS
    assert bench.max_over_ranks(3.25, None) == 3.25
    assert bench.rank_workload(WORKLOADS["c3"], 0) == WORKLOADS["c3"]
    assert bench.whole_job_tflops(1e12, 1, 1000.0) == pytest.approx(1.0)
