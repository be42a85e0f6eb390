"""A random-interleaving model of the persistent extend kernel's mbarrier protocol (host only).

Every role of one CTA is a coroutine -- the K and V producer warps, the two MMA issuers, the two
softmax groups -- and the asynchronous units are queues: the TMA engine completes gathers in any
order, and the tensor pipe executes each issuer's MMAs and commits in issue order.  A scheduler
advances them in random order over random item lists (items with one or two tiles, with and
without steps), with the phases, ring steps and S / P / turn counts running on across items as in
the kernel.  It checks what the hardware would not:

* parity aliasing: no wait ever tests a barrier two phases away from the one it means;
* deadlock: some role always makes progress;
* data hazards: an S MMA reads the K stage and Q buffer of its own step and item and never
  overwrites an S the softmax has not read or a P the PV MMA has not used; a PV MMA reads the V
  stage of its step and the P of its step; O is rescaled only when it holds PV(t-1), read out
  only when the item's last PV has run, and not overwritten by the next item before that; the
  next item's Q is copied in only once no S MMA of the current one is pending.

Barrier names follow the kernel: K_FULL / K_FREE / V_FULL / V_FREE per ring stage, S_FULL[x][b],
P_FULL[x][b], O_DONE[x], Q_FULL[x], TURN[x], DRAIN[x].
"""
import random

import pytest


class Barrier:
    def __init__(self, name, count):
        self.name, self.count = name, count
        self.arrived, self.tx, self.phases = 0, 0, 0

    def arrive(self, tx=0):
        self.arrived += 1
        self.tx += tx
        if self.arrived > self.count:
            raise RuntimeError(f"extra arrival on {self.name} phase {self.phases}")
        self._complete()

    def complete_tx(self, n):
        self.tx -= n
        if self.tx < 0:
            raise RuntimeError(f"transaction count below zero on {self.name}")
        self._complete()

    def _complete(self):
        if self.arrived == self.count and self.tx == 0:
            self.phases += 1
            self.arrived = 0


def simulate(items, stages, producer_warps, seed, p_rescale=0.3):
    """items: list of (steps, has_tile_B).  Raises RuntimeError on any violation."""
    rnd = random.Random(seed)
    bars = {}

    def make(key, count):
        bars[key] = Barrier(key, count)

    for i in range(stages):
        make(("K_FULL", i), 1)
        make(("K_FREE", i), 2)   # a commit from each issuer
        make(("V_FULL", i), 1)
        make(("V_FREE", i), 2)
    for x in range(2):
        for name in ("O_DONE", "TURN", "Q_FULL", "DRAIN"):
            make((name, x), 1)
        for b in range(2):
            make(("S_FULL", x, b), 1)
            make(("P_FULL", x, b), 1)
    tma = []                                   # gathers in flight
    pipe = {0: [], 1: []}                      # each issuer's MMAs and commits, in order
    ring = {"K": [None] * stages, "V": [None] * stages}     # ring step a stage was filled for
    landed = {"K": [None] * stages, "V": [None] * stages}   # ring step whose data has landed
    sbuf = {(x, b): None for x in range(2) for b in range(2)}  # ("S", id) or ("P", id)
    p_used = set()
    qbuf = {0: None, 1: None}
    qk_pending = {0: 0, 1: 0}
    o_state = {0: None, 1: None}               # (item, last PV step executed)
    o_read = {0: set(), 1: set()}

    def ready(key, phase):
        done = bars[key].phases
        if done == phase:
            return False
        if done == phase + 1:
            return True
        raise RuntimeError(f"parity alias on {key}: waiting for phase {phase}, {done} completed")

    steps_before = [0]
    for n, _ in items:
        steps_before.append(steps_before[-1] + n)

    def producer(op, w):
        # warp w fills ring steps w, w + PW, ... counted over all the CTA's items
        for i, (n, _) in enumerate(items):
            gs = steps_before[i]
            t0 = (w + producer_warps - gs % producer_warps) % producer_warps
            for t in range(t0, n, producer_warps):
                g = gs + t
                st = g % stages
                if g >= stages:
                    while not ready((op + "_FREE", st), g // stages - 1):
                        yield
                ring[op][st] = g
                landed[op][st] = None
                bars[(op + "_FULL", st)].arrive(tx=2)
                tma.append(((op + "_FULL", st), 1, op, st, g))  # two halves of the tile
                tma.append(((op + "_FULL", st), 1, op, st, g))
                yield

    def issuer(x):
        gs = sv = pb = nq = 0
        for i, (n, two) in enumerate(items):
            if n == 0:
                continue
            if x == 1 and not two:  # tile A only: release each stage with a plain arrival
                for t in range(n):
                    g = gs + t
                    while not ready(("K_FULL", g % stages), g // stages):
                        yield
                    bars[("K_FREE", g % stages)].arrive()
                    yield
                    while not ready(("V_FULL", g % stages), g // stages):
                        yield
                    bars[("V_FREE", g % stages)].arrive()
                    yield
                gs += n
                continue
            while not ready(("Q_FULL", x), nq):
                yield

            def qk(t):
                pipe[x].append(("QK", x, (sv + t) & 1, (i, t), (gs + t) % stages, gs + t))
                qk_pending[x] += 1

            def pv(t):
                pipe[x].append(("PV", x, (sv + t) & 1, (i, t), (gs + t) % stages, gs + t, t))

            for t in range(2):  # S(0), S(1); an item with fewer steps commits without an MMA
                if t < n:
                    g = gs + t
                    while not ready(("K_FULL", g % stages), g // stages):
                        yield
                    qk(t)
                    pipe[x].append(("S_FULL", x, (sv + t) & 1))
                    pipe[x].append(("K_FREE", g % stages))
                else:
                    pipe[x].append(("S_FULL", x, (sv + t) & 1))
            for t in range(n):
                g, g2 = gs + t, gs + t + 2
                more = t + 2 < n
                while not ready(("P_FULL", x, (pb + t) & 1), (pb + t) >> 1):
                    yield
                while not ready(("V_FULL", g % stages), g // stages):
                    yield
                if more:
                    while not ready(("K_FULL", g2 % stages), g2 // stages):
                        yield
                pv(t)
                if more:
                    qk(t + 2)  # into the buffer P(t) sits in, behind PV(t)
                pipe[x].append(("V_FREE", g % stages))
                pipe[x].append(("S_FULL", x, (sv + t) & 1))
                if more:
                    pipe[x].append(("K_FREE", g2 % stages))
                yield
            pipe[x].append(("O_DONE", x))
            gs += n
            sv += n + 2
            pb += n
            nq += 1
        pipe[x].append(("DRAIN", x))
        while not ready(("DRAIN", x), 0):
            yield

    def softmax(x):
        mine = [i for i, (n, two) in enumerate(items) if n > 0 and (x == 0 or two)]
        if not mine:
            return
        sv = pb = tb = nq = 0
        qbuf[x] = mine[0]
        bars[("Q_FULL", x)].arrive()
        yield
        for k, i in enumerate(mine):
            n, two = items[i]
            # the next item's query rows are copied in during this one only when the CTA's very
            # next item has tile x
            nxt = i + 1 if (i + 1 < len(items) and items[i + 1][0] > 0
                            and (x == 0 or items[i + 1][1])) else None
            if two and x == 1:
                bars[("TURN", 0)].arrive()  # tile A goes first
            for t in range(n):
                vs = sv + t
                while not ready(("S_FULL", x, vs & 1), vs >> 1):
                    yield
                if sbuf[(x, vs & 1)] != ("S", (i, t)):
                    raise RuntimeError(f"softmax {x} reads {sbuf[(x, vs & 1)]} for S{(i, t)}")
                if t == n - 1 and nxt is not None:
                    if qk_pending[x]:
                        raise RuntimeError(f"Q{x} overwritten with an S MMA pending")
                    qbuf[x] = ("loading", nxt)
                yield
                if two:
                    while not ready(("TURN", x), tb + t):
                        yield
                yield
                if two and (x == 0 or t + 1 < n):
                    bars[("TURN", 1 - x)].arrive()
                if t > 0 and rnd.random() < p_rescale:  # O rescaled: must hold PV(t-1)
                    vn = vs + 1
                    while not ready(("S_FULL", x, vn & 1), vn >> 1):
                        yield
                    if o_state[x] != (i, t - 1):
                        raise RuntimeError(f"rescale of O{x} at {o_state[x]} for step {(i, t)}")
                sbuf[(x, vs & 1)] = ("P", (i, t))
                bars[("P_FULL", x, (pb + t) & 1)].arrive()
                yield
            if nxt is not None:
                qbuf[x] = nxt
                bars[("Q_FULL", x)].arrive()
                yield
            while not ready(("O_DONE", x), nq):
                yield
            if o_state[x] != (i, n - 1):
                raise RuntimeError(f"epilogue of O{x} at {o_state[x]}, item {i}")
            o_read[x].add(i)
            yield
            sv += n + 2
            pb += n
            nq += 1
            if two:
                tb += n
            if nxt is None and k + 1 < len(mine):  # tile B after A-only items: its Q now
                if qk_pending[x]:
                    raise RuntimeError(f"Q{x} overwritten with an S MMA pending")
                qbuf[x] = mine[k + 1]
                bars[("Q_FULL", x)].arrive()
                yield

    def execute(x, op):
        if op[0] == "QK":
            _, x, b, sid, st, g = op
            if ring["K"][st] != g or landed["K"][st] != g:
                raise RuntimeError(f"S MMA {sid} reads K stage {st} holding {ring['K'][st]}")
            if qbuf[x] != sid[0]:
                raise RuntimeError(f"S MMA {sid} reads Q{x} = {qbuf[x]}")
            cur = sbuf[(x, b)]
            if cur is not None and cur[0] == "S":
                raise RuntimeError(f"S MMA {sid} overwrites unread {cur}")
            if cur is not None and cur[0] == "P" and cur[1] not in p_used:
                raise RuntimeError(f"S MMA {sid} overwrites unused {cur}")
            sbuf[(x, b)] = ("S", sid)
            qk_pending[x] -= 1
        elif op[0] == "PV":
            _, x, b, pid, st, g, t = op
            if ring["V"][st] != g or landed["V"][st] != g:
                raise RuntimeError(f"PV MMA {pid} reads V stage {st} holding {ring['V'][st]}")
            if sbuf[(x, b)] != ("P", pid):
                raise RuntimeError(f"PV MMA {pid} reads {sbuf[(x, b)]}")
            p_used.add(pid)
            if t == 0 and o_state[x] is not None and o_state[x][0] not in o_read[x]:
                raise RuntimeError(f"PV MMA {pid} overwrites O{x} before its epilogue")
            o_state[x] = pid
        else:
            bars[op].arrive()  # a commit

    alive = [producer("K", w) for w in range(producer_warps)]
    alive += [producer("V", w) for w in range(producer_warps)]
    alive += [issuer(0), issuer(1), softmax(0), softmax(1)]
    idle = 0
    while alive or tma or pipe[0] or pipe[1]:
        r = rnd.random()
        if r < 0.15 and tma:
            key, k, op, st, g = tma.pop(rnd.randrange(len(tma)))
            if ring[op][st] == g and not any(e[2] == op and e[3] == st and e[4] == g for e in tma):
                landed[op][st] = g
            bars[key].complete_tx(k)
            idle = 0
            continue
        if r < 0.3:
            x = rnd.randrange(2)
            if pipe[x]:
                execute(x, pipe[x].pop(0))
                idle = 0
                continue
        if not alive:
            continue
        a = rnd.choice(alive)
        try:
            next(a)
        except StopIteration:
            alive.remove(a)
        idle += 1
        if idle > 200000:
            raise RuntimeError("deadlock")


STAGES, PRODUCER_WARPS = 5, 3  # the kernel's kStages and kPW


def test_random_item_lists():
    rng = random.Random(7)
    for trial in range(1500):
        items = [(rng.choice([0, 1, 1, 2, 3, 4, 5, 7]), rng.random() < 0.7)
                 for _ in range(rng.randint(1, 6))]
        simulate(items, STAGES, PRODUCER_WARPS, trial)


@pytest.mark.parametrize("items", [
    [(1, True)] * 6,
    [(1, False)] * 6,
    [(2, False), (1, True), (1, False), (3, True)],
    [(26, True), (1, False), (11, True)],
])
def test_fixed_item_lists(items):
    for seed in range(100):
        simulate(items, STAGES, PRODUCER_WARPS, seed)


def test_a_ring_shallower_than_the_producer_warps_aliases_parity():
    """The kernel asserts kStages >= kPW at compile time: with fewer stages a producer warp can
    test a free barrier two phases early.  The model finds that."""
    found = 0
    for seed in range(50):
        rng = random.Random(seed)
        items = [(rng.choice([1, 2, 3, 5, 7]), rng.random() < 0.7)
                 for _ in range(rng.randint(1, 5))]
        try:
            simulate(items, 2, 3, seed)
        except RuntimeError as e:
            assert "parity alias" in str(e)
            found += 1
    assert found > 10
