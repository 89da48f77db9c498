"""A CPU model of the fp32 dQ kernel's synchronisation protocol.

fa_bwd_dq_kernel (fa_bwd.cu, 3xTF32 inputs) walks the 32-key chunks of one query
tile. Q and dO (hi / lo) stay resident; each chunk's K, V and K^T copies (hi / lo)
share one full barrier of a two-stage ring. The score issuer runs S = Q K^T and
dP = dO V^T into one of three TMEM slots, refilled once the accumulation of the
chunk three back completed; the softmax turns the slot into dS; the accumulate
issuer runs dQ += dS K (reading K^T) and releases the stage and the slot.

The accumulate issuer waits only for the softmax's dS: the chunk's K^T is ordered
by the stage's full barrier, which the score issuer observed before the S and dP
MMAs whose completion the softmax waited for. This test replays the roles under
random interleavings (copies land in any order, the tensor pipe runs in issue order)
and checks every read of the stage and the TMEM slots. Planted faults must be caught.
"""
import random

import pytest

from test_fwd_sync_model import MBarrier, ProtocolError

NST, NSL = 2, 3


def run_protocol(nc, seed, release_after_acc=True, wait_accdone=True, commit_before_mma=False):
    rnd = random.Random(seed)
    mb = {}

    def M(name):
        if name not in mb:
            mb[name] = MBarrier(name)
        return mb[name]

    stage = [None] * NST      # chunk whose K, V, K^T the stage holds
    pending = set()           # chunks whose stage an MMA still has to read
    slot = [None] * NSL       # ("SP", c) -> ("DS", c) -> ("DONE", c)
    acc = {"n": 0}
    copies, pipe = [], []

    def commit(bar):
        pipe.append(bar.arrive)

    def tma():
        for c in range(nc):
            st = c % NST
            yield (lambda st=st, c=c: M(("empty", st)).passed(((c // NST) & 1) ^ 1))
            bar = M(("full", st))
            bar.arrive_expect_tx(1)
            pending.add(c)

            def land(st=st, c=c, bar=bar):
                old = stage[st]
                if old is not None and old in pending:
                    raise ProtocolError(f"chunk {c} landed on chunk {old} still read by an MMA")
                stage[st] = c
                bar.complete_tx(1)
            copies.append(land)

    def score_issuer():
        for c in range(nc):
            st, bb = c % NST, c % NSL
            yield (lambda st=st, c=c: M(("full", st)).passed((c // NST) & 1))
            if c >= NSL and wait_accdone:
                yield (lambda bb=bb, c=c: M(("accdone", bb)).passed(((c // NSL) - 1) & 1))

            def mma(st=st, bb=bb, c=c):
                if stage[st] != c:
                    raise ProtocolError(f"S / dP of chunk {c} read the stage of chunk {stage[st]}")
                if slot[bb] is not None and slot[bb] != ("DONE", c - NSL):
                    raise ProtocolError(f"TMEM slot {bb} refilled while holding {slot[bb]}")
                slot[bb] = ("SP", c)
            pipe.append(mma)
            commit(M(("sp", bb)))
            if not release_after_acc:  # planted: stage released after the score MMAs
                commit(M(("empty", st)))

    def acc_issuer():
        for c in range(nc):
            pb, pst = c % NSL, c % NST
            yield (lambda pb=pb, c=c: M(("ds", pb)).passed((c // NSL) & 1))

            def mma(pb=pb, pst=pst, c=c):
                if slot[pb] != ("DS", c) or stage[pst] != c:
                    raise ProtocolError(f"dQ += dS K of chunk {c} read {slot[pb]}, stage {stage[pst]}")
                if acc["n"] != c:
                    raise ProtocolError(f"chunk {c} accumulated after {acc['n']} chunks")
                acc["n"] += 1
                slot[pb] = ("DONE", c)
                pending.discard(c)
            if commit_before_mma and release_after_acc:  # planted: released before it ran
                commit(M(("empty", pst)))
            pipe.append(mma)
            if release_after_acc and not commit_before_mma:
                commit(M(("empty", pst)))
            commit(M(("accdone", pb)))
        commit(M("done"))

    def softmax():
        for c in range(nc):
            bb = c % NSL
            yield (lambda bb=bb, c=c: M(("sp", bb)).passed((c // NSL) & 1))
            if slot[bb] != ("SP", c):
                raise ProtocolError(f"softmax of chunk {c} read {slot[bb]}")
            yield None
            slot[bb] = ("DS", c)
            M(("ds", bb)).arrive()
        yield (lambda: M("done").passed(0))
        if acc["n"] != nc:
            raise ProtocolError("epilogue before every chunk was accumulated")

    roles = {"tma": tma(), "score": score_issuer(), "acc": acc_issuer(), "softmax": softmax()}
    waiting = {r: None for r in roles}
    done = set()
    for _ in range(1_000_000):
        runnable = [r for r in roles if r not in done and (waiting[r] is None or waiting[r]())]
        choices = len(runnable) + (1 if copies else 0) + (1 if pipe else 0)
        if choices == 0:
            if len(done) == len(roles):
                return
            raise ProtocolError(f"deadlock: {sorted(set(roles) - done)} wait forever")
        k = rnd.randrange(choices)
        if k < len(runnable):
            r = runnable[k]
            try:
                waiting[r] = next(roles[r])
            except StopIteration:
                done.add(r)
                waiting[r] = None
        elif copies and k == len(runnable):
            copies.pop(rnd.randrange(len(copies)))()
        else:
            pipe.pop(0)()
    raise ProtocolError("no progress")


def test_protocol_holds_under_random_interleavings():
    rnd = random.Random(20261207)
    for _ in range(2000):
        run_protocol(rnd.randint(1, 12), seed=rnd.randrange(10 ** 9))


def _caught(trials, **fault):
    rnd = random.Random(23)
    for _ in range(trials):
        try:
            run_protocol(rnd.randint(3, 12), seed=rnd.randrange(10 ** 9), **fault)
        except ProtocolError:
            return True
    return False


def test_planted_fault_stage_released_after_the_score_mmas_is_caught():
    # K^T of the chunk is still to be read by dQ += dS K
    assert _caught(3000, release_after_acc=False)


def test_planted_fault_stage_released_before_the_accumulation_ran_is_caught():
    assert _caught(3000, commit_before_mma=True)


def test_tmem_slot_wait_is_implied_by_the_stage_ring():
    # The copy of chunk c lands only after dQ += dS K of chunk c - 2 freed its stage
    # (two stages, three TMEM slots), and the score issuer waits for that copy, so
    # chunk c - 3 was accumulated before its slot is refilled: the accdone wait never
    # blocks (the kernel keeps it, as it would matter with a deeper stage ring).
    rnd = random.Random(29)
    for _ in range(2000):
        run_protocol(rnd.randint(1, 12), seed=rnd.randrange(10 ** 9), wait_accdone=False)
