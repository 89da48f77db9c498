"""A CPU model of the persistent bf16 dQ kernel's synchronisation protocol.

fa_bwd_dq16_kernel (fa_bwd.cu) runs one CTA per SM over work items (a query tile,
possibly one key range of it) fetched at run time. Its roles:

  * the TMA producer publishes each item into a four-entry shared ring (read by the
    S issuer, the dP issuer, the accumulate issuer and the softmax warps), then
    loads the item's Q and dO tiles -- each once the previous item's last S (dP) MMA
    on that buffer has completed (q_rel / do_rel) -- and its K / V chunks into a
    three- / two-stage ring; the first V chunk of an item also waits until the
    previous item's epilogue stores have read the V ring, where dQ was staged (v_free);
  * the S issuer and the dP issuer run S = Q K^T and dP = dO V^T per chunk into one
    TMEM slot each, refilled once the softmax has loaded the previous chunk's;
  * the accumulate issuer runs dQ += dS K per chunk from one of two dS slots; the
    first of an item waits until the epilogue read the previous dQ (dq_free);
  * the softmax warps turn S / dP into dS, then read dQ, stage it in the V ring and
    store it.

Items without keys are skipped by every role. This test replays the roles in the
kernel's order under random interleavings (copies land in any order, the tensor
pipe runs in issue order) and checks every read of Q, dO, K, V, the TMEM slots, the
dQ accumulator and the staging area, and the ring hand-out. Planted faults must be
caught.
"""
import random

import pytest

from test_fwd_sync_model import MBarrier, ProtocolError

KST, VST, IRING = 3, 2, 4


def run_protocol(items, seed, wait_v_free=True, wait_dq_free=True, wait_q_rel=True,
                 wait_do_rel=True):
    """items: chunks per work item of this CTA (0 = no key). Raises on a violation."""
    rnd = random.Random(seed)
    mb = {}

    def M(name, count=1):
        if name not in mb:
            mb[name] = MBarrier(name, count)
        return mb[name]

    READERS = 4  # S issuer, dP issuer, accumulate issuer, softmax (all warps as one)
    for s in range(IRING):
        M(("ifull", s)), M(("iempty", s), READERS)
    ring = [None] * IRING
    smem_q, smem_do = [None], [None]
    smem_k, smem_v = [None] * KST, [None] * VST
    staged = set()            # V stages holding staged dQ not yet read by its stores
    tmem = {"S": None, "dP": None, "dS": [None, None], "acc": None}
    copies, pipe = [], []

    def commit(bar):
        pipe.append(bar.arrive)

    def land_into(buf, idx, tag, bar, busy):
        bar.arrive_expect_tx(1)

        def land():
            if busy():
                raise ProtocolError(f"copy of {tag} landed on a buffer still in use: {buf[idx]}")
            buf[idx] = tag
            bar.complete_tx(1)
        copies.append(land)

    reads = {"Q": set(), "dO": set(), "K": set(), "V": set()}  # tiles with MMAs pending

    def producer():
        j, g = 0, 0
        for k in range(len(items) + 1):
            s = k % IRING
            yield (lambda s=s, k=k: M(("iempty", s)).passed(((k // IRING) & 1) ^ 1))
            ring[s] = k if k < len(items) else None  # None: no further item
            M(("ifull", s)).arrive()
            if k == len(items):
                return
            n = items[k]
            if n == 0:
                continue
            for c in range(n):
                if c == 0:
                    if j > 0 and wait_q_rel:
                        yield (lambda j=j: M("qrel").passed((j - 1) & 1))
                    land_into(smem_q, 0, ("Q", k), M("q"), lambda: smem_q[0] in reads["Q"])
                ks = g % KST
                yield (lambda ks=ks, g=g: M(("kempty", ks)).passed(((g // KST) & 1) ^ 1))
                land_into(smem_k, ks, ("K", g), M(("kfull", ks)), lambda ks=ks: smem_k[ks] in reads["K"])
                if c == 0:
                    if j > 0 and wait_do_rel:
                        yield (lambda j=j: M("dorel").passed((j - 1) & 1))
                    land_into(smem_do, 0, ("dO", k), M("do"), lambda: smem_do[0] in reads["dO"])
                    if j > 0 and wait_v_free:
                        yield (lambda j=j: M("vfree").passed((j - 1) & 1))
                vs = g % VST
                yield (lambda vs=vs, g=g: M(("vempty", vs)).passed(((g // VST) & 1) ^ 1))
                land_into(smem_v, vs, ("V", g), M(("vfull", vs)),
                          lambda vs=vs: smem_v[vs] in reads["V"] or vs in staged)
                g += 1
            j += 1

    def take(k):
        s = k % IRING
        yield (lambda s=s, k=k: M(("ifull", s)).passed((k // IRING) & 1))
        w = ring[s]
        M(("iempty", s)).arrive()
        return w

    def score_issuer(kind):  # kind "S" (Q, K) or "dP" (dO, V)
        j, g, k = 0, 0, 0
        while True:
            w = yield from take(k)
            k += 1
            if w is None:
                return
            n = items[w]
            if n == 0:
                continue
            yield (lambda j=j: M("q" if kind == "S" else "do").passed(j & 1))
            j += 1
            for c in range(n):
                if kind == "S":
                    ks = g % KST
                    yield (lambda ks=ks, g=g: M(("kfull", ks)).passed((g // KST) & 1))
                else:
                    vs = g % VST
                    yield (lambda vs=vs, g=g: M(("vfull", vs)).passed((g // VST) & 1))
                if g > 0:
                    free = "sfree" if kind == "S" else "dpfree"
                    yield (lambda free=free, g=g: M(free).passed((g - 1) & 1))
                opnd = ("Q", w) if kind == "S" else ("dO", w)
                tile = ("K", g) if kind == "S" else ("V", g)
                reads[opnd[0]].add(opnd)
                reads[tile[0]].add(tile)

                def mma(g=g, opnd=opnd, tile=tile, last=c == n - 1):
                    res = smem_q[0] if kind == "S" else smem_do[0]
                    buf = smem_k[g % KST] if kind == "S" else smem_v[g % VST]
                    if res != opnd or buf != tile:
                        raise ProtocolError(f"{kind}({g}) read {res}, {buf}, wanted {opnd}, {tile}")
                    if tmem[kind] is not None and tmem[kind][1] != g - 1:
                        raise ProtocolError(f"{kind} slot refilled while holding {tmem[kind]}")
                    if tmem[kind] is not None and not tmem[kind][2]:
                        raise ProtocolError(f"{kind}({g}) overwrote {kind}({g - 1}) before the softmax read it")
                    tmem[kind] = (kind, g, False)
                    if kind == "dP":
                        reads["V"].discard(tile)
                    if last:  # the item's last S (dP) MMA has read Q (dO)
                        reads[opnd[0]].discard(opnd)
                pipe.append(mma)
                commit(M("s" if kind == "S" else "dp"))
                if kind == "dP":
                    commit(M(("vempty", g % VST)))
                g += 1
            commit(M("qrel" if kind == "S" else "dorel"))

    def acc_issuer():
        j, g, k = 0, 0, 0
        while True:
            w = yield from take(k)
            k += 1
            if w is None:
                return
            n = items[w]
            if n == 0:
                continue
            for c in range(n):
                pb, ks = g & 1, g % KST
                yield (lambda pb=pb, g=g: M(("ds", pb)).passed((g >> 1) & 1))
                if c == 0 and j > 0 and wait_dq_free:
                    yield (lambda j=j: M("dqfree").passed((j - 1) & 1))

                def mma(g=g, pb=pb, ks=ks, c=c, w=w):
                    if tmem["dS"][pb] != ("dS", g) or smem_k[ks] != ("K", g):
                        raise ProtocolError(f"dQ += dS K of chunk {g} read {tmem['dS'][pb]}, {smem_k[ks]}")
                    a = tmem["acc"]
                    if c == 0:
                        if a is not None and a[0] != "READ":
                            raise ProtocolError(f"dQ of item {w} overwrote an unread dQ {a}")
                    elif a != ("acc", w, g - 1):
                        raise ProtocolError(f"dQ accumulated onto {a}")
                    tmem["acc"] = ("acc", w, g)
                    tmem["dS"][pb] = ("USED", g)
                    reads["K"].discard(("K", g))
                pipe.append(mma)
                commit(M(("kempty", ks)))
                commit(M(("accdone", pb)))
                g += 1
            commit(M("done"))
            j += 1

    def softmax():
        j, g, k = 0, 0, 0
        while True:
            w = yield from take(k)
            k += 1
            if w is None:
                return
            n = items[w]
            if n == 0:
                continue
            for c in range(n):
                pb = g & 1
                yield (lambda g=g: M("s").passed(g & 1))
                if tmem["S"] != ("S", g, False):
                    raise ProtocolError(f"softmax read S {tmem['S']}, wanted chunk {g}")
                tmem["S"] = ("S", g, True)
                M("sfree").arrive()
                yield None
                yield (lambda g=g: M("dp").passed(g & 1))
                if tmem["dP"] != ("dP", g, False):
                    raise ProtocolError(f"softmax read dP {tmem['dP']}, wanted chunk {g}")
                tmem["dP"] = ("dP", g, True)
                M("dpfree").arrive()
                if g >= 2:
                    yield (lambda pb=pb, g=g: M(("accdone", pb)).passed(((g >> 1) - 1) & 1))
                if tmem["dS"][pb] is not None and tmem["dS"][pb] != ("USED", g - 2):
                    raise ProtocolError(f"dS slot {pb} overwritten while holding {tmem['dS'][pb]}")
                tmem["dS"][pb] = ("dS", g)
                M(("ds", pb)).arrive()
                g += 1
            # epilogue: dQ out of TMEM, staged in the V ring, TMA stores
            yield (lambda j=j: M("done").passed(j & 1))
            if tmem["acc"] != ("acc", w, g - 1):
                raise ProtocolError(f"epilogue of item {w} read {tmem['acc']}")
            tmem["acc"] = ("READ",)
            M("dqfree").arrive()
            for vs in range(VST):
                if smem_v[vs] in reads["V"]:
                    raise ProtocolError(f"dQ staged over V tile {smem_v[vs]} that an MMA still reads")
                staged.add(vs)
                smem_v[vs] = ("STAGE", w)

            def store_read(w=w):
                for vs in range(VST):
                    if smem_v[vs] != ("STAGE", w):
                        raise ProtocolError(f"dQ store of item {w} read {smem_v[vs]}")
                    staged.discard(vs)
            copies.append(store_read)
            yield (lambda: not staged)
            M("vfree").arrive()
            j += 1

    roles = {"tma": producer(), "S": score_issuer("S"), "dP": score_issuer("dP"),
             "acc": acc_issuer(), "softmax": softmax()}
    waiting = {r: None for r in roles}
    done = set()
    for _ in range(2_000_000):
        runnable = [r for r in roles if r not in done and (waiting[r] is None or waiting[r]())]
        choices = len(runnable) + (1 if copies else 0) + (1 if pipe else 0)
        if choices == 0:
            if len(done) == len(roles):
                return
            raise ProtocolError(f"deadlock: {sorted(set(roles) - done)} wait forever")
        c = rnd.randrange(choices)
        if c < len(runnable):
            r = runnable[c]
            try:
                waiting[r] = next(roles[r])
            except StopIteration:
                done.add(r)
                waiting[r] = None
        elif copies and c == len(runnable):
            copies.pop(rnd.randrange(len(copies)))()
        else:
            pipe.pop(0)()
    raise ProtocolError("no progress")


def random_items(rnd):
    return [rnd.choice([0, 1, 1, 2, 3, 4, 6]) for _ in range(rnd.randint(1, 8))]


def test_protocol_holds_under_random_interleavings():
    rnd = random.Random(20261205)
    for _ in range(1500):
        run_protocol(random_items(rnd), seed=rnd.randrange(10 ** 9))


def _caught(trials, **fault):
    rnd = random.Random(13)
    for _ in range(trials):
        try:
            run_protocol(random_items(rnd), seed=rnd.randrange(10 ** 9), **fault)
        except ProtocolError:
            return True
    return False


@pytest.mark.parametrize("fault", ["wait_v_free", "wait_q_rel", "wait_do_rel"])
def test_planted_fault_is_caught(fault):
    # dropping one of these per-item hand-offs must be detected
    assert _caught(3000, **{fault: False})


def test_dq_free_is_implied_by_the_next_ds_hand_off():
    # The accumulate issuer's first dQ MMA of an item also waits for that item's first
    # dS, which the softmax warps write only after they read the previous dQ out of
    # TMEM, so the dq_free wait never blocks (the kernel keeps it as a cheap guard).
    rnd = random.Random(17)
    for _ in range(1500):
        run_protocol(random_items(rnd), seed=rnd.randrange(10 ** 9), wait_dq_free=False)
