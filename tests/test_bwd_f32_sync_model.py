"""A CPU model of the fp32 dK/dV kernel's synchronisation protocol.

fa_bwd_dkdv_kernel (fa_bwd.cu, 3xTF32 inputs) walks the query chunks of one key
tile. Each shared-memory stage of chunk operands has two halves with their own
full / empty mbarriers:

  * the score half (Q, dO chunks), read by the S^T and dP^T MMAs and released by
    the score issuer's commit after them, so the next chunk's copy can land while
    this chunk's softmax and accumulating MMAs run;
  * the accumulate half (Q^T, dO^T chunks and the lse2 / delta vectors), read by the
    softmax (the vectors) and by the dV / dK MMAs, released by the accumulate
    issuer's commit after them.

Two TMEM slots hold S^T / dP^T of alternate chunks: the softmax turns a slot into P^T
/ dS^T and the accumulating MMAs consume it; the score issuer refills a slot only
after the accumulation of the chunk two back. This test replays the roles in the
kernel's order under random interleavings -- copies land in any order, the tensor
pipe runs MMAs and commits in issue order -- and checks that every MMA and the
softmax read the chunk they were meant to, that no copy lands on a half that an MMA
or the softmax still has to read, and that a TMEM slot is refilled only after it was
consumed. Two planted faults must be caught.
"""
import random

import pytest

from test_fwd_sync_model import MBarrier, ProtocolError


def run_protocol(nc, NST, seed, score_release_after_mma=True, acc_half_released_by_acc=True):
    """Play one CTA's chunks; raises ProtocolError on any violation."""
    rnd = random.Random(seed)
    mb = {}

    def M(name):
        if name not in mb:
            mb[name] = MBarrier(name)
        return mb[name]

    smem_s = [None] * NST  # ("S", c): score half holding chunk c
    smem_a = [None] * NST  # ("A", c): accumulate half holding chunk c
    pending_s = set()      # chunks whose score half an MMA still has to read
    pending_a = set()      # chunks whose accumulate half the softmax or an MMA still reads
    tmem = [None, None]    # slot contents: ("SP", c) -> ("DS", c) -> ("DONE", c)
    acc = {"n": 0}         # chunks accumulated into dV / dK, in order
    copies, pipe = [], []

    def commit(bar):
        pipe.append(bar.arrive)

    def load(half, c):
        st = c % NST
        bar = M((half + "full", st))
        bar.arrive_expect_tx(1)

        def land():
            if half == "s":
                old = smem_s[st]
                if old is not None and old[1] in pending_s:
                    raise ProtocolError(f"score half of chunk {old[1]} overwritten before its MMAs")
                smem_s[st] = ("S", c)
                pending_s.add(c)
            else:
                old = smem_a[st]
                if old is not None and old[1] in pending_a:
                    raise ProtocolError(f"accumulate half of chunk {old[1]} overwritten while read")
                smem_a[st] = ("A", c)
                pending_a.add(c)
            bar.complete_tx(1)
        copies.append(land)

    def tma():
        for c in range(nc):
            st = c % NST
            yield (lambda st=st, c=c: M(("sempty", st)).passed(((c // NST) & 1) ^ 1))
            load("s", c)
            yield (lambda st=st, c=c: M(("aempty", st)).passed(((c // NST) & 1) ^ 1))
            load("a", c)

    def score_issuer():
        for c in range(nc):
            st, bb = c % NST, c & 1
            yield (lambda st=st, c=c: M(("sfull", st)).passed((c // NST) & 1))
            if c >= 2:
                yield (lambda bb=bb, c=c: M(("accdone", bb)).passed(((c - 2) >> 1) & 1))

            def mma(st=st, bb=bb, c=c):
                if smem_s[st] != ("S", c):
                    raise ProtocolError(f"S^T / dP^T of chunk {c} read {smem_s[st]}")
                if tmem[bb] is not None and tmem[bb] != ("DONE", c - 2):
                    raise ProtocolError(f"TMEM slot {bb} refilled while holding {tmem[bb]}")
                tmem[bb] = ("SP", c)
                pending_s.discard(c)
            if score_release_after_mma:
                pipe.append(mma)
                commit(M(("sp", bb)))
                commit(M(("sempty", st)))
                if not acc_half_released_by_acc:
                    commit(M(("aempty", st)))
            else:  # planted: the score half released before its MMAs ran
                commit(M(("sempty", st)))
                pipe.append(mma)
                commit(M(("sp", bb)))

    def acc_issuer():
        for c in range(nc):
            pb, pst = c & 1, c % NST
            yield (lambda pb=pb, c=c: M(("ds", pb)).passed((c >> 1) & 1))
            yield (lambda pst=pst, c=c: M(("afull", pst)).passed((c // NST) & 1))

            def mma(pb=pb, pst=pst, c=c):
                if tmem[pb] != ("DS", c):
                    raise ProtocolError(f"dV / dK of chunk {c} read TMEM {tmem[pb]}")
                if smem_a[pst] != ("A", c):
                    raise ProtocolError(f"dV / dK of chunk {c} read {smem_a[pst]}")
                if acc["n"] != c:
                    raise ProtocolError(f"chunk {c} accumulated after {acc['n']} chunks")
                acc["n"] += 1
                tmem[pb] = ("DONE", c)
                pending_a.discard(c)
            pipe.append(mma)
            if acc_half_released_by_acc:
                commit(M(("aempty", pst)))
            commit(M(("accdone", pb)))
        commit(M("done"))

    def softmax():
        for c in range(nc):
            bb, st = c & 1, c % NST
            yield (lambda bb=bb, st=st, c=c: M(("sp", bb)).passed((c >> 1) & 1)
                   and M(("afull", st)).passed((c // NST) & 1))
            if tmem[bb] != ("SP", c) or smem_a[st] != ("A", c):
                raise ProtocolError(f"softmax of chunk {c} read {tmem[bb]}, {smem_a[st]}")
            yield None  # exponentials (reads lse2)
            yield None  # dS = P (dP - delta) (reads delta)
            if smem_a[st] != ("A", c):
                raise ProtocolError(f"lse2 / delta of chunk {c} overwritten while read")
            tmem[bb] = ("DS", c)
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


@pytest.mark.parametrize("NST", [1, 2])
def test_protocol_holds_under_random_interleavings(NST):
    # NST = 1 is the kernel's configuration (fp32, D = 64); 2 checks the ring logic
    rnd = random.Random(20261204 + NST)
    for _ in range(1500):
        run_protocol(rnd.randint(1, 9), NST, seed=rnd.randrange(10 ** 9))


def _caught(trials, **fault):
    rnd = random.Random(11)
    for _ in range(trials):
        try:
            run_protocol(rnd.randint(2, 9), 1, seed=rnd.randrange(10 ** 9), **fault)
        except ProtocolError:
            return True
    return False


def test_planted_fault_score_half_released_before_its_mmas_is_caught():
    assert _caught(3000, score_release_after_mma=False)


def test_planted_fault_accumulate_half_released_with_the_score_half_is_caught():
    # releasing lse2 / delta and Q^T / dO^T after the score MMAs, as for the score half
    assert _caught(3000, acc_half_released_by_acc=False)
