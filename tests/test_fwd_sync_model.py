"""A CPU model of the persistent forward kernel's synchronisation protocol.

fa_fwd_kernel (fa_fwd.cu) runs one CTA per SM over a sequence of work items; its
roles hand work to one another through mbarriers (phase / parity waits), named
barriers (bar.sync / bar.arrive, which count arrivals and cannot time out), an
in-order tensor pipe (MMAs and their commits) and TMA copies that land in any
order. Two races of that protocol were found with this model before the kernel ran:
a parity wait that passed on a phase two behind (the relay's first K wait with a
one-stage K ring), and epilogue stage grants arriving on the V full barriers, which
let the relay skip phases. This test replays the protocol -- role by role, in the
kernel's order -- under random interleavings and checks that

  * nobody deadlocks and every named-barrier generation pairs its roles exactly;
  * every MMA reads the operand tile it was meant to (Q, K, V, P in TMEM) and never
    one that a copy has already overwritten or not yet written;
  * no copy or epilogue stage overwrites a V stage that an MMA or a TMA store still
    has to read, and the epilogue reads each O accumulator before it is reused.

Item lists mix items with no key, one key tile and several, as the causal /
windowed schedules do. An item's epilogue stage goes to all its query tiles at once,
each staging through its own part; the last tile releases it after the others have
announced (EPI_JOIN) that their stores read their parts. The model must follow
fa_fwd_kernel: a change to the kernel's hand-offs has to be made here too. Three
planted faults (the races above, put back into the model, and a tile announcing its
part before its stores read it) must be caught.
"""
import random

import pytest


class ProtocolError(Exception):
    pass


class MBarrier:
    """mbarrier: arrival count + transaction bytes; try_wait.parity semantics."""

    def __init__(self, name, count=1):
        self.name, self.count, self.pending, self.tx, self.phase = name, count, count, 0, 0

    def _maybe_complete(self):
        if self.pending == 0 and self.tx == 0:
            self.phase += 1
            self.pending = self.count

    def arrive(self):
        self.pending -= 1
        if self.pending < 0:
            raise ProtocolError(f"too many arrivals on {self.name}")
        self._maybe_complete()

    def arrive_expect_tx(self, nbytes):
        self.tx += nbytes
        self.arrive()

    def complete_tx(self, nbytes):
        self.tx -= nbytes
        self._maybe_complete()

    def passed(self, parity):
        # try_wait.parity: true once the phase with this parity has completed, i.e.
        # while the current (incomplete) phase has the other parity
        return (self.phase & 1) != parity


class NamedBarrier:
    """bar.sync / bar.arrive: a generation completes when `count` threads arrived."""

    def __init__(self, name):
        self.name, self.arrived, self.generation, self.members = name, 0, 0, []

    def arrive(self, who, threads, count):
        if who in self.members:
            raise ProtocolError(f"{who} arrived twice in one generation of barrier {self.name}")
        self.members.append(who)
        self.arrived += threads
        gen = self.generation
        if self.arrived == count:
            self.arrived, self.members = 0, []
            self.generation += 1
        elif self.arrived > count:
            raise ProtocolError(f"barrier {self.name} overfilled")
        return gen


def run_protocol(items, NQ, KST, VST, seed, relay_observes_first_k=True,
                 release_after_reads=True, join_after_reads=True):
    """Play one CTA's item list; raises ProtocolError on any violation."""
    rnd = random.Random(seed)
    mb = {}

    def M(name, count=1):
        if name not in mb:
            mb[name] = MBarrier(name, count)
        return mb[name]

    nb = {}

    def N(i):
        if i not in nb:
            nb[i] = NamedBarrier(i)
        return nb[i]

    smem_q, smem_k, smem_v = [None] * NQ, [None] * KST, [None] * VST
    tmem_s, tmem_o = [None] * NQ, [None] * NQ
    copies = []      # TMA copies / stores in flight: completion callbacks, any order
    pipe = []        # tensor pipe: MMAs and commits, in issue order
    stores = set()   # epilogue stages whose TMA stores have not read them yet
    consumed = {}    # key tile -> number of PV MMAs that read it

    def tma(fn):
        copies.append(fn)

    def mma(fn):
        pipe.append(fn)

    def commit(bar):
        pipe.append(bar.arrive)

    def v_stage_free(s):
        c = smem_v[s]
        if c is None:
            return True
        if c[0] == "V":
            return consumed.get(c[1], 0) == NQ
        if c[0] == "STAGING":  # an item's epilogue: every tile's stores must have read it
            return all(("st", c[1], q) not in stores for q in range(NQ))
        return False

    def load_q(q, item):
        bar = M(("q", q))
        bar.arrive_expect_tx(1)

        def land():
            smem_q[q] = ("Q", item, q)
            bar.complete_tx(1)
        tma(land)

    def load_k(g):
        s = g % KST
        bar = M(("kfull", s))
        bar.arrive_expect_tx(1)

        def land():
            smem_k[s] = ("K", g)
            bar.complete_tx(1)
        tma(land)

    def load_v(pos, g):
        s = pos % VST
        bar = M(("vfull", s))
        if not v_stage_free(s):
            raise ProtocolError(f"V copy issued into a busy stage holding {smem_v[s]}")
        bar.arrive_expect_tx(1)

        def land():
            smem_v[s] = ("V", g)
            bar.complete_tx(1)
        tma(land)

    def nsync(i, who, threads, count):
        gen = N(i).arrive(who, threads, count)
        yield lambda: N(i).generation > gen

    key_tiles, g = [], 0  # global key-tile indices of each item
    for n in items:
        key_tiles.append(list(range(g, g + n)))
        g += n
    setup = len(items) > 0 and items[0] > 0
    for q in range(NQ):
        for name in ("q", "qfree", "s", "o", "grant"):
            M((name, q))
    for s in range(KST):
        M(("kfull", s)), M(("kempty", s))
    for s in range(VST):
        M(("vfull", s)), M(("vempty", s))
    if setup:  # the init thread's loads of the first item
        for q in range(NQ):
            load_q(q, 0)
        load_k(0)
        load_v(0, 0)

    def qk_producer():
        g, j = 0, 0
        for k, n in enumerate(items):
            if n == 0:
                continue
            for t in range(n):
                if k == 0 and t == 0:
                    g += 1
                    continue
                s = g % KST
                yield (lambda s=s, g=g: M(("kempty", s)).passed(((g // KST) & 1) ^ 1))
                load_k(g)
                if t == 0:
                    for q in range(NQ):
                        if j > 0:
                            yield (lambda q=q, j=j: M(("qfree", q)).passed((j - 1) & 1))
                        load_q(q, k)
                g += 1
            j += 1

    def v_producer():
        pos, seen, prev_stage = 0, [0] * VST, None

        def wait_release(p):
            s, u = p % VST, p // VST
            if seen[s] <= u:
                yield (lambda s=s, u=u: M(("vempty", s)).passed(u & 1))
                seen[s] = u + 1
        for k, n in enumerate(items):
            for t in range(n):
                if k == 0 and t == 0:
                    pos += 1
                    continue
                if pos >= VST:
                    yield from wait_release(pos - VST)
                load_v(pos, key_tiles[k][t])
                pos += 1
            if pos >= VST:
                yield from wait_release(pos - VST)
            if prev_stage is not None:
                yield from wait_release(prev_stage)
            if not v_stage_free(pos % VST):
                raise ProtocolError(f"epilogue stage granted while busy: {smem_v[pos % VST]}")
            for q in range(NQ):  # every tile at once, each staging through its own part
                M(("grant", q)).arrive()
            prev_stage = pos
            pos += 1

    def issuer():
        g, pos, j = 0, 0, 0
        for k, n in enumerate(items):
            if n == 0:
                pos += 1
                continue
            for q in range(NQ):  # item start: S_q(0) once the relay saw Q_q (and K_g)
                yield from nsync("relay", "issuer", 32, 64)

                def s0(q=q, k=k, g=g):
                    if smem_q[q] != ("Q", k, q) or smem_k[g % KST] != ("K", g):
                        raise ProtocolError(f"first S of item {k} read {smem_q[q]}, {smem_k[g % KST]}")
                    tmem_s[q] = ("S", k, q, g)
                mma(s0)
                commit(M(("s", q)))
                if n == 1:
                    commit(M(("qfree", q)))
            commit(M(("kempty", g % KST)))
            for t in range(n):
                vs, ks, more = pos % VST, (g + 1) % KST, t + 1 < n
                yield from nsync("relay", "issuer", 32, 64)
                for q in range(NQ):
                    yield from nsync(("P", q), "issuer", 32, 160)

                    def pv(q=q, k=k, g=g, vs=vs, t=t):
                        if tmem_s[q] != ("P", k, q, g):
                            raise ProtocolError(f"PV read P {tmem_s[q]}, wanted {('P', k, q, g)}")
                        if smem_v[vs] != ("V", g):
                            raise ProtocolError(f"PV read V {smem_v[vs]}, wanted {('V', g)}")
                        if t > 0 and tmem_o[q] != ("O", k, q, g - 1):
                            raise ProtocolError(f"PV accumulated onto {tmem_o[q]}")
                        if t == 0 and tmem_o[q] is not None and tmem_o[q][0] != "READ":
                            raise ProtocolError(f"PV overwrote an O not yet read: {tmem_o[q]}")
                        tmem_o[q] = ("O", k, q, g)
                        consumed[g] = consumed.get(g, 0) + 1
                    mma(pv)
                    if more:
                        def s(q=q, k=k, g=g, ks=ks):
                            if smem_q[q] != ("Q", k, q) or smem_k[ks] != ("K", g + 1):
                                raise ProtocolError(f"S read {smem_q[q]}, {smem_k[ks]}")
                            tmem_s[q] = ("S", k, q, g + 1)
                        mma(s)
                        commit(M(("s", q)))
                        if t + 2 == n:
                            commit(M(("qfree", q)))
                    else:
                        commit(M(("o", q)))
                commit(M(("vempty", vs)))
                if more:
                    commit(M(("kempty", ks)))
                g += 1
                pos += 1
            pos += 1
            j += 1

    def relay():
        g, j, pos, loads = 0, 0, 0, [0] * VST
        for k, n in enumerate(items):
            if n == 0:
                pos += 1
                continue
            for q in range(NQ):  # item start: Q_q and the first K tile
                yield (lambda q=q, j=j: M(("q", q)).passed(j & 1))
                if q == 0 and relay_observes_first_k:
                    yield (lambda g=g: M(("kfull", g % KST)).passed((g // KST) & 1))
                yield from nsync("relay", "relay", 32, 64)
            for t in range(n):
                more = t + 1 < n
                s = pos % VST
                yield (lambda s=s, c=loads[s]: M(("vfull", s)).passed(c & 1))
                loads[s] += 1
                if more:
                    ks, par = (g + 1) % KST, ((g + 1) // KST) & 1
                    yield (lambda ks=ks, par=par: M(("kfull", ks)).passed(par))
                yield from nsync("relay", "relay", 32, 64)
                g += 1
                pos += 1
            pos += 1
            j += 1

    def softmax(q):
        g, j, pos = 0, 0, 0
        pending = {"on": False, "slot": 0, "tag": None}

        def release():
            tag = pending["tag"]
            if release_after_reads:
                yield (lambda tag=tag: tag not in stores)
            # every tile's stores have read their part (the other tiles arrive on the join)
            yield from nsync(("join",), f"softmax{q}", 128, 128 * NQ)
            M(("vempty", pending["slot"])).arrive()
            pending["on"] = False

        for k, n in enumerate(items):
            for t in range(n):
                yield (lambda g=g: M(("s", q)).passed(g & 1))
                if tmem_s[q] != ("S", k, q, g):
                    raise ProtocolError(f"softmax read S {tmem_s[q]}, wanted {('S', k, q, g)}")
                yield None
                tmem_s[q] = ("P", k, q, g)
                N(("P", q)).arrive(f"softmax{q}", 128, 160)
                if pending["on"]:
                    yield from release()
                g += 1
            pos += n
            if n > 0:
                yield (lambda j=j: M(("o", q)).passed(j & 1))
                if tmem_o[q] != ("O", k, q, g - 1):
                    raise ProtocolError(f"epilogue read O {tmem_o[q]}")
                tmem_o[q] = ("READ",)
                j += 1
            if pending["on"]:
                yield from release()
            slot = pos % VST
            yield (lambda k=k: M(("grant", q)).passed(k & 1))
            if smem_v[slot] != ("STAGING", k):  # the first tile to start its stores
                if not v_stage_free(slot):
                    raise ProtocolError(f"staging into a busy stage: {smem_v[slot]}")
                smem_v[slot] = ("STAGING", k)
            tag = ("st", k, q)
            stores.add(tag)

            def store_read(slot=slot, k=k, tag=tag):
                if smem_v[slot] != ("STAGING", k):
                    raise ProtocolError(f"TMA store read an overwritten stage: {smem_v[slot]}")
                stores.discard(tag)
            tma(store_read)
            if q < NQ - 1:  # its part has been read: the last tile may release the stage
                if join_after_reads:
                    yield (lambda tag=tag: tag not in stores)
                N(("join",)).arrive(f"softmax{q}", 128, 128 * NQ)
            else:
                pending.update(on=True, slot=slot, tag=tag)
            yield None
            pos += 1
        if pending["on"]:
            yield from release()

    roles = {"qk": qk_producer(), "v": v_producer(), "issuer": issuer(), "relay": relay()}
    for q in range(NQ):
        roles[f"softmax{q}"] = softmax(q)
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


# (query tiles per CTA, K stages, V stages) of the kernel's configurations:
# bf16 D = 128, bf16 D = 64, fp32 D = 64
CONFIGS = [(2, 2, 3), (2, 3, 3), (1, 1, 1)]


def random_items(rnd):
    return [rnd.choice([0, 1, 1, 2, 2, 3, 4, 5, 7]) for _ in range(rnd.randint(1, 9))]


@pytest.mark.parametrize("cfg", CONFIGS)
def test_protocol_holds_under_random_interleavings(cfg):
    rnd = random.Random(20261203 + sum(cfg))
    for _ in range(1000):
        run_protocol(random_items(rnd), *cfg, seed=rnd.randrange(10 ** 9))


def _caught(cfg, trials, **fault):
    rnd = random.Random(7)
    for _ in range(trials):
        try:
            run_protocol(random_items(rnd), *cfg, seed=rnd.randrange(10 ** 9), **fault)
        except ProtocolError:
            return True
    return False


def test_planted_fault_relay_skips_first_k_is_caught():
    # with a one-stage K ring the relay's K_1 wait can pass on K_0's phase
    assert _caught((1, 1, 1), 3000, relay_observes_first_k=False)


def test_planted_fault_early_stage_release_is_caught():
    # giving the epilogue stage back before its TMA stores read it
    assert _caught((2, 2, 3), 3000, release_after_reads=False)


def test_planted_fault_join_before_the_stores_read_is_caught():
    # a tile that announces its part as read before its stores have read it lets the
    # last tile release the stage while those stores may still read it
    assert _caught((2, 2, 3), 400, join_after_reads=False)
