"""A CPU model of the bf16 dK/dV kernel's synchronisation protocol.

fa_bwd_dkdv16_kernel (fa_bwd.cu) walks the 128-query chunks of one key tile:

  * the TMA producer keeps K, V resident and streams Q and dO chunks through two-slot
    rings; a Q slot is free once S^T = K Q^T and dK += dS^T Q of its chunk have read
    it (two commits), a dO slot once dP^T = V dO^T and dV += P^T dO have (two commits);
  * the S issuer runs S^T(c) into the S^T slot once the softmax loaded S^T(c - 1);
  * the B issuer runs dP^T(c) into the dP^T slot, then, once the softmax wrote
    dS^T(c) over the first half of that slot, dK += dS^T Q; dP^T(c + 1) follows dK(c)
    from the same thread, so the tensor pipe reads dS^T(c) before overwriting it;
  * the dV issuer runs dV += P^T(c) dO once the softmax wrote P^T(c) into the shared
    P^T tile, which the softmax refills only after that MMA completed (dv_done);
  * the softmax warps wait for S^T(c), chunk c's vectors (with Q_c) and dO_c, load S^T
    (freeing the slot), exponentiate, write P^T, wait for dP^T, write dS^T. The dO_c
    wait is what orders the dV MMA after the dO copy (P^T would otherwise be written
    as soon as S^T, i.e. Q_c, is in); dropping it is one of the planted faults.

The variant with two-term P and dS (SPLIT, chosen for short query sequences): the
softmax writes P^T = P_hi + P_lo into the S^T slot it has just read, instead of the
shared P^T tile, and dV += P^T dO reads it from there (two MMAs); dS^T_lo goes into the
half of the dP^T slot that dS^T_hi leaves free, and dK takes two MMAs. The S^T slot is
then freed by the dV MMAs' commit, not by the softmax's load; keeping the early
release is a planted fault.

This test replays the roles in the kernel's order under random interleavings (copies
land in any order, the tensor pipe runs in issue order) and checks every read of Q,
dO, the TMEM slots and the P^T tile, and the accumulation order of dV and dK. Planted
faults must be caught.
"""
import random

import pytest

from test_fwd_sync_model import MBarrier, ProtocolError

NS = 2  # Q / dO ring depth at D = 128


def run_protocol(nc, seed, q_release_count=2, wait_dv_done=True, wait_sfree=True,
                 softmax_waits_do=True, split=False, split_softmax_frees_s=False):
    """Play the chunks of one key tile; raises ProtocolError on a violation."""
    rnd = random.Random(seed)
    mb = {}

    def M(name, count=1):
        if name not in mb:
            mb[name] = MBarrier(name, count)
        return mb[name]

    for s in range(NS):
        M(("qempty", s), q_release_count)
        M(("doempty", s), 2)
    smem_q, smem_do = [None] * NS, [None] * NS
    reads = {"Q": {}, "dO": {}}  # chunk -> MMAs still to read that slot
    pt = {"tile": None, "read": True}  # P^T smem tile: chunk and whether dV read it
    tmem = {"S": None, "dP": None}
    acc = {"dV": 0, "dK": 0}
    copies, pipe = [], []

    def commit(bar):
        pipe.append(bar.arrive)

    def load(kind, c):
        st = c % NS
        bar = M((kind + "full", st))
        buf = smem_q if kind == "q" else smem_do
        name = "Q" if kind == "q" else "dO"
        bar.arrive_expect_tx(1)
        reads[name][c] = 2  # the two MMAs that read this chunk's tile

        def land():
            old = buf[st]
            if old is not None and reads[name].get(old[1], 0) > 0:
                raise ProtocolError(f"{name} chunk {c} landed on chunk {old[1]} still read by an MMA")
            buf[st] = (name, c)
            bar.complete_tx(1)
        copies.append(land)

    def read(name, buf, c):
        st = c % NS
        if buf[st] != (name, c):
            raise ProtocolError(f"an MMA of chunk {c} read {buf[st]}")
        reads[name][c] -= 1

    def tma():
        for c in range(nc):
            st = c % NS
            yield (lambda st=st, c=c: M(("doempty", st)).passed(((c // NS) & 1) ^ 1))
            load("do", c)
            yield (lambda st=st, c=c: M(("qempty", st)).passed(((c // NS) & 1) ^ 1))
            load("q", c)

    def s_issuer():
        for c in range(nc):
            st = c % NS
            yield (lambda st=st, c=c: M(("qfull", st)).passed((c // NS) & 1))
            if c > 0 and wait_sfree:
                yield (lambda c=c: M("sfree").passed((c - 1) & 1))

            def mma(c=c):
                read("Q", smem_q, c)
                if tmem["S"] is not None and not tmem["S"][2]:
                    raise ProtocolError(f"S^T({c}) overwrote {tmem['S'][0]}({tmem['S'][1]}) before "
                                        "it was read")
                tmem["S"] = ("S", c, False)
            pipe.append(mma)
            commit(M("s"))
            commit(M(("qempty", st)))

    def dv_issuer():
        for c in range(nc):
            st = c % NS
            yield (lambda c=c: M("p").passed(c & 1))

            def mma(c=c):
                if split:
                    if tmem["S"] != ("P", c, False):
                        raise ProtocolError(f"dV({c}) read {tmem['S']} from the S^T slot")
                    tmem["S"] = ("P", c, True)
                elif pt["tile"] != c:
                    raise ProtocolError(f"dV({c}) read the P^T tile of chunk {pt['tile']}")
                read("dO", smem_do, c)
                if acc["dV"] != c:
                    raise ProtocolError(f"dV accumulated chunk {c} after {acc['dV']} chunks")
                acc["dV"] += 1
                pt["read"] = True
            pipe.append(mma)  # (split: the P_hi and P_lo MMAs, one after the other)
            commit(M(("doempty", st)))
            if split:
                commit(M("sfree"))  # P^T(c) has left the S^T slot: S^T(c + 1) may go in
            else:
                commit(M("dvdone"))
        commit(M("done", 2))

    def b_issuer():
        for c in range(nc):
            st = c % NS
            yield (lambda st=st, c=c: M(("dofull", st)).passed((c // NS) & 1))

            def dp(c=c):
                read("dO", smem_do, c)
                if tmem["dP"] is not None and tmem["dP"][0] != "USED":
                    raise ProtocolError(f"dP^T({c}) overwrote {tmem['dP']}")
                tmem["dP"] = ("dP", c)
            pipe.append(dp)
            commit(M("dp"))
            commit(M(("doempty", st)))
            yield (lambda c=c: M("ds").passed(c & 1))

            def dk(c=c):
                if tmem["dP"] != ("dS", c):
                    raise ProtocolError(f"dK({c}) read {tmem['dP']}")
                read("Q", smem_q, c)
                if acc["dK"] != c:
                    raise ProtocolError(f"dK accumulated chunk {c} after {acc['dK']} chunks")
                acc["dK"] += 1
                tmem["dP"] = ("USED", c)
            pipe.append(dk)
            commit(M(("qempty", st)))
        commit(M("done", 2))

    def softmax():
        for c in range(nc):
            st = c % NS
            yield (lambda st=st, c=c: M("s").passed(c & 1) and M(("qfull", st)).passed((c // NS) & 1)
                   and (not softmax_waits_do or M(("dofull", st)).passed((c // NS) & 1)))
            if tmem["S"] != ("S", c, False):
                raise ProtocolError(f"softmax read S^T {tmem['S']}, wanted chunk {c}")
            tmem["S"] = ("S", c, True)
            if not split or split_softmax_frees_s:
                M("sfree").arrive()
            yield None  # exponentials (lse2 of the chunk from the ring's vector slot)
            if split:
                # P^T hi / lo over the S^T columns this thread has just read
                if tmem["S"] != ("S", c, True):
                    raise ProtocolError(f"P^T({c}) written over {tmem['S']}")
                tmem["S"] = ("P", c, False)
            else:
                if c > 0 and wait_dv_done:
                    yield (lambda c=c: M("dvdone").passed((c - 1) & 1))
                if not pt["read"]:
                    raise ProtocolError(f"P^T({c}) written over P^T({pt['tile']}) before dV read it")
                pt["tile"], pt["read"] = c, False
            M("p").arrive()
            yield (lambda c=c: M("dp").passed(c & 1))
            if tmem["dP"] != ("dP", c):
                raise ProtocolError(f"softmax read dP^T {tmem['dP']}, wanted chunk {c}")
            yield None
            tmem["dP"] = ("dS", c)
            M("ds").arrive()
        yield (lambda: M("done", 2).passed(0))
        if acc["dV"] != nc or acc["dK"] != nc:
            raise ProtocolError("epilogue before every chunk was accumulated")

    roles = {"tma": tma(), "S": s_issuer(), "dV": dv_issuer(), "B": b_issuer(), "softmax": softmax()}
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
    rnd = random.Random(20261206)
    for _ in range(2000):
        run_protocol(rnd.randint(1, 10), seed=rnd.randrange(10 ** 9))


def test_split_protocol_holds_under_random_interleavings():
    rnd = random.Random(20261207)
    for _ in range(2000):
        run_protocol(rnd.randint(1, 10), seed=rnd.randrange(10 ** 9), split=True)


def test_planted_fault_split_st_slot_freed_by_the_softmax_is_caught():
    # with P^T in the S^T slot, the softmax's early release lets S^T(c + 1) overwrite
    # P^T(c) before dV has read it
    assert _caught(3000, split=True, split_softmax_frees_s=True)


def test_planted_fault_split_without_the_sfree_wait_is_caught():
    assert _caught(3000, split=True, wait_sfree=False)


def _caught(trials, **fault):
    rnd = random.Random(19)
    for _ in range(trials):
        try:
            run_protocol(rnd.randint(2, 10), seed=rnd.randrange(10 ** 9), **fault)
        except ProtocolError:
            return True
    return False


def test_planted_fault_q_slot_freed_by_one_reader_is_caught():
    # a Q slot released after S^T alone (dK of the chunk still has to read it)
    assert _caught(3000, q_release_count=1)


def test_planted_fault_pt_refilled_before_dv_read_it_is_caught():
    assert _caught(3000, wait_dv_done=False)


def test_planted_fault_st_slot_refilled_before_the_softmax_read_it_is_caught():
    assert _caught(3000, wait_sfree=False)


def test_planted_fault_dv_not_ordered_after_the_do_copy_is_caught():
    assert _caught(3000, softmax_waits_do=False)


# ---------------------------------------------------------------- persistent CTAs
# The persistent form of the kernel: one CTA walks several work items (key tiles),
# each with its own number of query chunks (0 for a key tile no query sees). The
# Q / dO rings and the per-chunk hand-offs count chunks across items (g); per item
# with chunks (j):
#   * K / V are loaded into the one resident buffer once the previous item's last
#     S^T and dP^T MMAs have read it (kv_free: a commit from the S and the B issuer
#     after their item's last score MMA);
#   * the first dV and dK MMAs of an item (accumulate = false) overwrite the
#     accumulators: they run only once the softmax has written that item's first P^T
#     / dS^T, which it does only after its epilogue of the previous item has read both
#     accumulators out of TMEM -- so no barrier of its own is needed (the model can add
#     one, acc_free, and shows that dropping it is never caught);
#   * the epilogue waits for every MMA of the item (done: the dV issuer's and the B
#     issuer's commit) and stages the stores in the P^T tile, which the softmax
#     refills only after the epilogue.
# An item without chunks writes zeros and touches none of these barriers.

def run_protocol_persistent(ncs, seed, split=False, wait_kv_free=True, wait_acc_free=False,
                            kv_free_count=2, epilogue_waits_done=True):
    rnd = random.Random(seed)
    mb = {}

    def M(name, count=1):
        if name not in mb:
            mb[name] = MBarrier(name, count)
        return mb[name]

    for s in range(NS):
        M(("qempty", s), 2)
        M(("doempty", s), 2)
    M("kvfree", kv_free_count)
    M("done", 2)
    smem_q, smem_do = [None] * NS, [None] * NS
    reads = {"Q": {}, "dO": {}}
    kv = {"item": None, "pending": 0}  # resident K / V: item, score MMAs still to read it
    pt = {"tile": None, "read": True, "staging": False}
    tmem = {"S": None, "dP": None}
    acc = {"item": None, "dV": 0, "dK": 0, "read": True}
    copies, pipe = [], []
    items = [(k, n) for k, n in enumerate(ncs)]
    with_chunks = [(k, n) for k, n in items if n > 0]
    # global chunk index of each (item, chunk)
    gidx, g = {}, 0
    for k, n in items:
        for c in range(n):
            gidx[(k, c)] = g
            g += 1

    def commit(bar):
        pipe.append(bar.arrive)

    def load(kind, gg, item):
        st = gg % NS
        bar = M((kind + "full", st))
        buf = smem_q if kind == "q" else smem_do
        name = "Q" if kind == "q" else "dO"
        bar.arrive_expect_tx(1)
        reads[name][gg] = 2

        def land():
            old = buf[st]
            if old is not None and reads[name].get(old[1], 0) > 0:
                raise ProtocolError(f"{name} chunk {gg} landed on chunk {old[1]} still read by an MMA")
            buf[st] = (name, gg)
            bar.complete_tx(1)
        copies.append(land)

    def read(name, buf, gg):
        st = gg % NS
        if buf[st] != (name, gg):
            raise ProtocolError(f"an MMA of chunk {gg} read {buf[st]}")
        reads[name][gg] -= 1

    def tma():
        for j, (k, n) in enumerate(with_chunks):
            if j > 0 and wait_kv_free:
                yield (lambda j=j: M("kvfree", kv_free_count).passed((j - 1) & 1))
            M("kv").arrive_expect_tx(1)

            def land_kv(k=k):
                if kv["pending"] > 0:
                    raise ProtocolError(f"K / V of item {k} landed on item {kv['item']} still read")
                kv["item"], kv["pending"] = k, 2 * ncs[k]
                M("kv").complete_tx(1)
            copies.append(land_kv)
            for c in range(n):
                gg = gidx[(k, c)]
                st = gg % NS
                yield (lambda st=st, gg=gg: M(("doempty", st)).passed(((gg // NS) & 1) ^ 1))
                load("do", gg, k)
                yield (lambda st=st, gg=gg: M(("qempty", st)).passed(((gg // NS) & 1) ^ 1))
                load("q", gg, k)

    def kv_read(k):
        if kv["item"] != k:
            raise ProtocolError(f"a score MMA of item {k} read K / V of item {kv['item']}")
        kv["pending"] -= 1

    def s_issuer():
        for j, (k, n) in enumerate(with_chunks):
            yield (lambda j=j: M("kv").passed(j & 1))
            for c in range(n):
                gg = gidx[(k, c)]
                st = gg % NS
                yield (lambda st=st, gg=gg: M(("qfull", st)).passed((gg // NS) & 1))
                if gg > 0:
                    yield (lambda gg=gg: M("sfree").passed((gg - 1) & 1))

                def mma(gg=gg, k=k):
                    kv_read(k)
                    read("Q", smem_q, gg)
                    if tmem["S"] is not None and not tmem["S"][2]:
                        raise ProtocolError(f"S^T({gg}) overwrote {tmem['S'][0]}({tmem['S'][1]})")
                    tmem["S"] = ("S", gg, False)
                pipe.append(mma)
                commit(M("s"))
                commit(M(("qempty", st)))
            commit(M("kvfree", kv_free_count))

    def acc_mma(kind, k, c):
        if c == 0:
            if not acc["read"] and acc["item"] != k:
                raise ProtocolError(f"the first {kind} MMA of item {k} overwrote the accumulators "
                                    f"of item {acc['item']} before the epilogue read them")
            if acc["item"] != k:
                acc["item"], acc["dV"], acc["dK"], acc["read"] = k, 0, 0, False
        if acc["item"] != k:
            raise ProtocolError(f"{kind} of item {k} accumulated into item {acc['item']}")
        if acc[kind] != c:
            raise ProtocolError(f"{kind} accumulated chunk {c} of item {k} after {acc[kind]}")
        acc[kind] += 1

    def dv_issuer():
        for j, (k, n) in enumerate(with_chunks):
            for c in range(n):
                gg = gidx[(k, c)]
                st = gg % NS
                yield (lambda gg=gg: M("p").passed(gg & 1))
                if c == 0 and j > 0 and wait_acc_free:
                    yield (lambda j=j: M("accfree").passed((j - 1) & 1))

                def mma(gg=gg, k=k, c=c):
                    if split:
                        if tmem["S"] != ("P", gg, False):
                            raise ProtocolError(f"dV({gg}) read {tmem['S']} from the S^T slot")
                        tmem["S"] = ("P", gg, True)
                    else:
                        if pt["tile"] != gg or pt["staging"]:
                            raise ProtocolError(f"dV({gg}) read the P^T tile holding {pt}")
                        pt["read"] = True
                    read("dO", smem_do, gg)
                    acc_mma("dV", k, c)
                pipe.append(mma)
                commit(M(("doempty", st)))
                commit(M("sfree") if split else M("dvdone"))
            commit(M("done", 2))

    def b_issuer():
        for j, (k, n) in enumerate(with_chunks):
            yield (lambda j=j: M("kv").passed(j & 1))
            for c in range(n):
                gg = gidx[(k, c)]
                st = gg % NS
                yield (lambda st=st, gg=gg: M(("dofull", st)).passed((gg // NS) & 1))

                def dp(gg=gg, k=k):
                    kv_read(k)
                    read("dO", smem_do, gg)
                    if tmem["dP"] is not None and tmem["dP"][0] != "USED":
                        raise ProtocolError(f"dP^T({gg}) overwrote {tmem['dP']}")
                    tmem["dP"] = ("dP", gg)
                pipe.append(dp)
                commit(M("dp"))
                commit(M(("doempty", st)))
                if c == n - 1:
                    commit(M("kvfree", kv_free_count))
                yield (lambda gg=gg: M("ds").passed(gg & 1))
                if c == 0 and j > 0 and wait_acc_free:
                    yield (lambda j=j: M("accfree").passed((j - 1) & 1))

                def dk(gg=gg, k=k, c=c):
                    if tmem["dP"] != ("dS", gg):
                        raise ProtocolError(f"dK({gg}) read {tmem['dP']}")
                    read("Q", smem_q, gg)
                    acc_mma("dK", k, c)
                    tmem["dP"] = ("USED", gg)
                pipe.append(dk)
                commit(M(("qempty", st)))
            commit(M("done", 2))

    def softmax():
        j = 0
        for k, n in items:
            for c in range(n):
                gg = gidx[(k, c)]
                st = gg % NS
                yield (lambda st=st, gg=gg: M("s").passed(gg & 1) and M(("qfull", st)).passed((gg // NS) & 1)
                       and M(("dofull", st)).passed((gg // NS) & 1))
                if tmem["S"] != ("S", gg, False):
                    raise ProtocolError(f"softmax read S^T {tmem['S']}, wanted chunk {gg}")
                tmem["S"] = ("S", gg, True)
                if not split:
                    M("sfree").arrive()
                yield None
                if split:
                    tmem["S"] = ("P", gg, False)
                else:
                    if gg > 0:
                        yield (lambda gg=gg: M("dvdone").passed((gg - 1) & 1))
                    if not pt["read"]:
                        raise ProtocolError(f"P^T({gg}) written over P^T({pt['tile']}) before dV read it")
                    if pt["staging"]:
                        raise ProtocolError(f"P^T({gg}) written over the epilogue's staging")
                    pt["tile"], pt["read"] = gg, False
                M("p").arrive()
                yield (lambda gg=gg: M("dp").passed(gg & 1))
                if tmem["dP"] != ("dP", gg):
                    raise ProtocolError(f"softmax read dP^T {tmem['dP']}, wanted chunk {gg}")
                yield None
                tmem["dP"] = ("dS", gg)
                M("ds").arrive()
            if n == 0:
                continue  # zeros straight to the outputs
            if epilogue_waits_done:
                yield (lambda j=j: M("done", 2).passed(j & 1))
            if acc["item"] != k or acc["dV"] != n or acc["dK"] != n:
                raise ProtocolError(f"epilogue of item {k} read accumulators {acc}")
            acc["read"] = True
            # stage the stores in the P^T tile: no dV MMA may still read it
            if not split and not pt["read"]:
                raise ProtocolError(f"epilogue of item {k} staged over P^T({pt['tile']}) before dV read it")
            pt["staging"] = True
            M("accfree").arrive()  # (after the TMEM loads)
            yield None  # TMA stores read the staging area
            pt["staging"] = False
            j += 1

    roles = {"tma": tma(), "S": s_issuer(), "dV": dv_issuer(), "B": b_issuer(), "softmax": softmax()}
    waiting = {r: None for r in roles}
    done = set()
    for _ in range(2_000_000):
        runnable = [r for r in roles if r not in done and (waiting[r] is None or waiting[r]())]
        choices = len(runnable) + (1 if copies else 0) + (1 if pipe else 0)
        if choices == 0:
            if len(done) == len(roles):
                return
            raise ProtocolError(f"deadlock: {sorted(set(roles) - done)} wait forever")
        kk = rnd.randrange(choices)
        if kk < len(runnable):
            r = runnable[kk]
            try:
                waiting[r] = next(roles[r])
            except StopIteration:
                done.add(r)
                waiting[r] = None
        elif copies and kk == len(runnable):
            copies.pop(rnd.randrange(len(copies)))()
        else:
            pipe.pop(0)()
    raise ProtocolError("no progress")


def _items(rnd):
    return [rnd.choice([0, 1, 2, 3, 5, 8]) for _ in range(rnd.randint(1, 5))]


@pytest.mark.parametrize("split", [False, True])
def test_persistent_protocol_holds_under_random_interleavings(split):
    rnd = random.Random(20261208 + split)
    for _ in range(1500):
        run_protocol_persistent(_items(rnd), seed=rnd.randrange(10 ** 9), split=split)


def _caught_persistent(trials, **fault):
    rnd = random.Random(23)
    for _ in range(trials):
        ncs = [rnd.randint(1, 6) for _ in range(rnd.randint(2, 5))]
        try:
            run_protocol_persistent(ncs, seed=rnd.randrange(10 ** 9), **fault)
        except ProtocolError:
            return True
    return False


def test_planted_fault_kv_reloaded_before_the_last_score_mma_is_caught():
    assert _caught_persistent(3000, wait_kv_free=False)


def test_planted_fault_kv_free_from_one_issuer_only_is_caught():
    assert _caught_persistent(3000, kv_free_count=1)


def test_accumulator_reuse_is_ordered_by_the_softmax_alone():
    # with or without an acc_free barrier no first dV / dK MMA of an item reaches the
    # accumulators before the previous item's epilogue has read them (the kernel has none)
    assert not _caught_persistent(3000, wait_acc_free=False)
    assert not _caught_persistent(1000, wait_acc_free=True)


def test_planted_fault_epilogue_before_the_last_mma_is_caught():
    assert _caught_persistent(3000, epilogue_waits_done=False)
