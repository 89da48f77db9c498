"""GPU test of fa_fwd_noalloc, the forward pass for callers that cannot allocate.

Some callers of this library may not allocate device memory at call time: an
inference runtime that reserves its whole footprint at start-up and must not
grow afterwards, a host application whose own allocator owns the device, or code
running where a cudaMalloc is forbidden or could block. fa_fwd serves them badly
because it takes scratch from a pool it grows on demand; fa_fwd_noalloc instead
keeps its scratch in a fixed array compiled into libfa.so.

This file checks, through the C ABI, that two calls in a row of fa_fwd_noalloc
(on different inputs, so the second call cannot reuse what the first left in the
shared array) give O and LSE within the parity tolerances of the fp64 oracle and
of fa_fwd, for both input precisions, and that a problem too large for the array
is refused with FA_ERR_SCRATCH_LIMIT. It is named to run after every other test
file and also passes when run on its own in a fresh process.
"""
import pytest
import torch

import oracle
from attention_fa_fwd_02_gb300.workloads import WORKLOADS, make_inputs
from _parity import TOL, lse_err, rms_err, to_np

pytestmark = pytest.mark.gpu

FA_ERR_SCRATCH_LIMIT = 6


@pytest.fixture(scope="module")
def fa():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "this test needs a CUDA device"
    from attention_fa_fwd_02_gb300 import fa as m
    return m


def _call(fa, entry, w, tensors, f32_mma="f16x2"):
    qd, kd, vd = tensors
    p = fa.make_params(qd, kd, w.scale, w.causal, w.window, f32_mma=f32_mma)
    o = torch.empty(qd.shape, dtype=torch.float32, device=qd.device)
    lse = torch.empty(qd.shape[:3], dtype=torch.float32, device=qd.device)
    rc = entry(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(), lse.data_ptr(), p,
               int(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, fa.status_string(rc)
    return o, lse


PAIRS = {
    "bf16": (WORKLOADS["c3"].with_(B=1, H=8, HKV=2, Sq=1000, Sk=1000, seed=31),
             WORKLOADS["c4"].with_(B=1, H=4, HKV=4, Sq=700, Sk=900, window=256, causal=False,
                                   seed=32)),
    "f32": (WORKLOADS["c2"].with_(B=1, H=2, HKV=2, Sq=500, Sk=500, seed=33),
            WORKLOADS["c5"].with_(Sq=300, Sk=450, seed=34)),
    # the same pair through the 3xTF32 kernels (fa_params.f32_mma)
    "f32-tf32x3": (WORKLOADS["c2"].with_(B=1, H=2, HKV=2, Sq=500, Sk=500, seed=33),
                   WORKLOADS["c5"].with_(Sq=300, Sk=450, seed=34)),
    # fp32 at D = 128 (two scaled fp16 terms per operand)
    "f32-d128": (WORKLOADS["c2"].with_(B=1, H=2, HKV=1, Sq=400, Sk=400, D=128, scale=128 ** -0.5,
                                       seed=35),
                 WORKLOADS["c5"].with_(Sq=200, Sk=350, D=96, scale=96 ** -0.5, seed=36)),
}


@pytest.mark.parametrize("kind", list(PAIRS))
def test_noalloc_matches_oracle_and_fa_fwd_on_two_calls_in_a_row(fa, kind):
    ws = PAIRS[kind]
    mode = "tf32x3" if kind.endswith("tf32x3") else "f16x2"
    cpu = [make_inputs(w)[:3] for w in ws]
    ins = [tuple(t.cuda() for t in c) for c in cpu]
    # two no-allocation calls back to back, the second on different data
    got = [_call(fa, fa.fa_fwd_noalloc, w, t, mode) for w, t in zip(ws, ins)]
    fa.check_device_status()
    ref = [_call(fa, fa.fa_fwd, w, t, mode) for w, t in zip(ws, ins)]
    fa.check_device_status()
    for w, c, (o, lse), (ro, rl) in zip(ws, cpu, got, ref):
        tol = TOL[w.dtype]
        # against the fp64 oracle on the same inputs ...
        xo, xl = oracle.attention_fwd(*c, w.scale, w.causal, w.window)
        assert rms_err(to_np(o), xo) <= tol["O"], w.name
        assert lse_err(to_np(lse), xl) <= tol["LSE"], w.name
        # ... and against the allocating entry point
        assert rms_err(to_np(o), to_np(ro)) <= tol["O"]
        assert lse_err(to_np(lse), to_np(rl)) <= tol["LSE"]


def test_noalloc_refuses_problems_larger_than_its_scratch(fa):
    # bf16 inputs on the tensor-core path need B*HKV*Sk*D*2 bytes of scratch: Sk = 2^17
    # + 1 keys at D = 128 is just over the 32 MiB array. (9 query rows: above the decode
    # shapes, whose kernel needs only its small partial results.) The tensors are real,
    # so even a wrong answer here would stay inside allocated memory.
    sk = (fa.noalloc_scratch_bytes() // (128 * 2)) + 1
    q = torch.zeros(1, 1, 9, 128, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(1, 1, sk, 128, dtype=torch.bfloat16, device="cuda")
    p = fa.make_params(q, k, 0.1, False, 0)
    o = torch.empty(1, 1, 9, 128, dtype=torch.float32, device="cuda")
    lse = torch.empty(1, 1, 9, dtype=torch.float32, device="cuda")
    rc = fa.fa_fwd_noalloc(q.data_ptr(), k.data_ptr(), k.data_ptr(), o.data_ptr(), lse.data_ptr(),
                           p, int(torch.cuda.current_stream().cuda_stream))
    assert rc == FA_ERR_SCRATCH_LIMIT
    assert "static scratch" in fa.status_string(rc)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_noalloc_decode_shapes_match_fa_fwd_bit_for_bit(fa, dtype):
    # decode shapes (at most 8 query rows per kv head) run fa_fwd's decode kernel, with
    # its key-range partial results in the array: the same outputs, bit for bit, and
    # within the parity bounds of the oracle
    base = WORKLOADS["c3"] if dtype == "bf16" else WORKLOADS["c5"]
    w = base.with_(B=2, H=8, HKV=2, Sq=2, Sk=7000, causal=False, window=0, seed=37)
    c = make_inputs(w)[:3]
    t = tuple(x.cuda() for x in c)
    got = _call(fa, fa.fa_fwd_noalloc, w, t)
    ref = _call(fa, fa.fa_fwd, w, t)
    fa.check_device_status()
    assert torch.equal(got[0], ref[0]) and torch.equal(got[1], ref[1])
    xo, xl = oracle.attention_fwd(*c, w.scale, w.causal, w.window)
    assert rms_err(to_np(got[0]), xo) <= TOL[w.dtype]["O"]
    assert lse_err(to_np(got[1]), xl) <= TOL[w.dtype]["LSE"]
