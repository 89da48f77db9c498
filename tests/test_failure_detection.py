"""Failure detection on the GPU without faulting it.

Every barrier wait in the library's kernels is bounded. fa_selftest_timeout
launches a kernel with the attention kernels' control skeleton in which a copy
is never issued, so its waits run out: the test checks that the expiry is
reported as FA_ERR_TIMEOUT, that all three waiting roles left, that reading the
status clears it, and that the same context still computes a correct forward
pass afterwards. No trap, fault or hang is involved.
"""
import pytest
import torch

import oracle
from attention_fa_fwd_02_gb300.workloads import WORKLOADS, make_inputs
from _parity import TOL, lse_err, rms_err, to_np

pytestmark = pytest.mark.gpu

FA_ERR_TIMEOUT = 5


@pytest.fixture(scope="module")
def fa():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "this test needs a CUDA device"
    from attention_fa_fwd_02_gb300 import fa as m
    return m


def test_barrier_timeout_is_reported_and_context_survives(fa):
    stream = int(torch.cuda.current_stream().cuda_stream)
    assert fa.fa_device_status(stream) == 0
    roles = torch.zeros(4, dtype=torch.int32, device="cuda")
    assert fa.fa_selftest_timeout(50_000_000, roles.data_ptr(), stream) == 0  # 50 ms limit
    assert fa.fa_device_status(stream) == FA_ERR_TIMEOUT
    assert int(roles[0].item()) == 3
    assert fa.fa_device_status(stream) == 0  # reading clears the word

    w = WORKLOADS["c3"].with_(B=1, H=2, HKV=1, Sq=256, Sk=256, seed=41)
    q, k, v, _ = make_inputs(w)
    o, lse = fa.forward(q.cuda(), k.cuda(), v.cuda(), w.scale, w.causal, w.window)
    fa.check_device_status()
    ro, rl = oracle.attention_fwd(q, k, v, w.scale, w.causal, w.window)
    assert rms_err(to_np(o), ro) <= TOL["bf16"]["O"]
    assert lse_err(to_np(lse), rl) <= TOL["bf16"]["LSE"]
