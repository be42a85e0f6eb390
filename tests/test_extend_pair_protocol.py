"""A random-interleaving model of the SM-pair extend kernel's barrier protocol (host only).

Two CTAs (0 = even, 1 = odd) each have K and V producer warps and a softmax group; the even CTA
has the MMA issuer, the odd one the relay that forwards its landed ring stages to the even CTA.
The asynchronous units are queues: each CTA's TMA engine completes gathers in any order, and the
tensor pipe executes the issuer's MMAs and commits in issue order; a commit arrives on the
barriers of every CTA in its mask.  A scheduler advances everything in random order over random
item lists (items without steps included), with ring steps, S / P steps and items counted across
items as in the kernel.  It checks:

* parity aliasing: no wait ever tests a barrier two phases away from the one it means;
* deadlock: some role always makes progress;
* data hazards, in each CTA: an S MMA reads K stages (both CTAs' halves) of its own step that
  have landed and the Q rows of its own item, and never overwrites an S the softmax has not read
  or a P the PV MMA has not used; a PV MMA reads both CTAs' V halves of its step and both CTAs'
  P of its step; O is rescaled only when it holds PV(t-1), read out only after the item's last
  PV, and not overwritten by the next item before both CTAs read it; the next item's Q is copied
  in only once no S MMA of the current one is pending; a stage is refilled only after the MMAs
  that read it completed.

Barrier names follow the kernel: KL / VL (a CTA's own gathers landed), KP / VP (even CTA: the odd
CTA's half landed), KF / VF (stage free), SF[b], PF[b], QF, OD, DR.  PF and QF take one arrival
per CTA here (the kernel's four warps of each CTA arrive together).
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


def simulate(items, stages, producer_warps, seed, p_rescale=0.3, nbuf=3, q_in_order=True):
    """items: list of step counts; nbuf S buffers.  Raises RuntimeError on any violation.
    q_in_order=False drops the query-row copies' wait for the previous item's copy."""
    rnd = random.Random(seed)
    bars = {}

    def make(key, count):
        bars[key] = Barrier(key, count)

    for c in range(2):
        for s in range(stages):
            for name in ("KL", "VL", "KF", "VF"):
                make((c, name, s), 1)
        for b in range(nbuf):
            make((c, "SF", b), 1)
        make((c, "OD"), 1)
        for b in range(2):
            make((c, "MR", b), 1)   # a warpgroup's 128 threads, as one arrival here
            make((c, "ML", b), 2)   # both warpgroups
    for s in range(stages):
        make((0, "KP", s), 1)
        make((0, "VP", s), 1)
    for b in range(nbuf):
        make((0, "PF", b), 2)
    for c in range(2):
        for qb in range(2):
            make((c, "QF", qb), 1)  # the CTA's query rows of an item in Q buffer qb
        for qb in range(2):
            make((c, "QE", qb), 1)  # commit after the last S of an item that used Q buffer qb
    for qb in range(2):
        make((0, "QP", qb), 1)  # the relay: the odd CTA's query rows in buffer qb landed
    make((0, "DR"), 1)

    tma = {0: [], 1: []}                      # gathers in flight per CTA
    pipe = []                                 # the issuer's MMAs and commits, in order
    ring = {(c, op): [None] * stages for c in range(2) for op in "KV"}    # step a stage holds
    landed = {(c, op): [None] * stages for c in range(2) for op in "KV"}  # step landed there
    reading = {(c, op): [set() for _ in range(stages)] for c in range(2) for op in "KV"}
    sbuf = {(c, b): None for c in range(2) for b in range(nbuf)}  # ("S", id) or ("P", id)
    p_used = set()
    qbuf = {(c, qb): None for c in range(2) for qb in range(2)}  # item whose rows a buffer holds
    qk_pending = [0, 0]  # S MMAs issued, not yet executed, per Q buffer they read
    o_state = {0: None, 1: None}              # (item, last PV step executed)
    o_read = {0: set(), 1: set()}
    m_slot = {(c, b): None for c in range(2) for b in range(2)}  # (item, step) of a stored max
    m_read = set()

    def ready(key, phase):
        done = bars[key].phases
        if done == phase:
            return False
        if done == phase + 1:
            return True
        raise RuntimeError(f"parity alias on {key}: waiting for phase {phase}, {done} completed")

    work = [n for n in items if n > 0]        # every role skips items without steps
    steps_before = [0]
    for n in work:
        steps_before.append(steps_before[-1] + n)

    def producer(c, op, w):
        for i, n in enumerate(work):
            gs = steps_before[i]
            t0 = (w + producer_warps - gs % producer_warps) % producer_warps
            if op == "V" and t0 == 0:  # the V warp of an item's first step copies its Q rows
                yield from load_q(c, i)
            for t in range(t0, n, producer_warps):
                g = gs + t
                st = g % stages
                if g >= stages:
                    while not ready((c, op + "F", st), g // stages - 1):
                        yield
                if reading[(c, op)][st]:
                    raise RuntimeError(f"CTA {c} refills {op} stage {st} with MMAs reading it")
                ring[(c, op)][st] = g
                landed[(c, op)][st] = None
                bars[(c, op + "L", st)].arrive(tx=2)
                tma[c].append(((c, op + "L", st), 1, op, st, g))  # two halves / four gathers
                tma[c].append(((c, op + "L", st), 1, op, st, g))
                yield

    def relay():
        def fwd(op, g):
            st = g % stages
            while not ready((1, op + "L", st), g // stages):
                yield
            bars[(0, op + "P", st)].arrive()
        for i, n in enumerate(work):
            gs = steps_before[i]
            while not ready((1, "QF", i & 1), i >> 1):
                yield
            bars[(0, "QP", i & 1)].arrive()
            for t in range(min(nbuf, n)):
                yield from fwd("K", gs + t)
            for t in range(n):
                if t + nbuf < n:
                    yield from fwd("K", gs + t + nbuf)
                yield from fwd("V", gs + t)

    def issuer():
        sv = pb = nq = 0

        def landed_both(op, g):
            st = g % stages
            while not ready((0, op + "L", st), g // stages):
                yield
            while not ready((0, op + "P", st), g // stages):
                yield

        for i, n in enumerate(work):
            gs = steps_before[i]
            while not ready((0, "QF", nq & 1), nq >> 1):
                yield
            while not ready((0, "QP", nq & 1), nq >> 1):
                yield

            def qk(t):
                pipe.append(("QK", (sv + t) % nbuf, (i, t), (gs + t) % stages, gs + t))
                qk_pending[i & 1] += 1
                for c in range(2):
                    reading[(c, "K")][(gs + t) % stages].add((i, t))

            def pv(t):
                pipe.append(("PV", (sv + t) % nbuf, (i, t), (gs + t) % stages, gs + t, t))
                for c in range(2):
                    reading[(c, "V")][(gs + t) % stages].add((i, t))

            for t in range(nbuf):
                if t < n:
                    yield from landed_both("K", gs + t)
                    qk(t)
                    pipe.append(("SF", (sv + t) % nbuf))
                    pipe.append(("KF", (gs + t) % stages))
                    if t == n - 1:
                        pipe.append(("QE", i & 1))
                else:
                    pipe.append(("SF", (sv + t) % nbuf))  # a step without an MMA
            for t in range(n):
                g, g2 = gs + t, gs + t + nbuf
                more = t + nbuf < n
                if more:
                    yield from landed_both("K", g2)
                yield from landed_both("V", g)
                while not ready((0, "PF", (pb + t) % nbuf), (pb + t) // nbuf):
                    yield
                pv(t)
                if more:
                    qk(t + nbuf)
                pipe.append(("VF", g % stages))
                pipe.append(("SF", (sv + t) % nbuf))
                if more:
                    pipe.append(("KF", g2 % stages))
                if more and t + nbuf == n - 1:
                    pipe.append(("QE", i & 1))
                yield
            pipe.append(("OD",))
            sv += n + nbuf
            pb += n
            nq += 1
        pipe.append(("DR",))
        while not ready((0, "DR"), 0):
            yield

    q_loaded = {0: 0, 1: 0}  # the CTA's count of items whose query rows were copied in

    def load_q(c, i):
        """The CTA's query rows of item i into Q buffer i % 2, once item i-1's were copied in (so
        that the wait on QE is for its next phase) and the S MMAs of item i-2, the buffer's
        previous item, are done."""
        qb = i & 1
        if i > 0:
            while q_in_order and q_loaded[c] < i:
                yield
        if i > 1:
            while not ready((c, "QE", qb), (i - 2) >> 1):
                yield
            if qk_pending[qb]:
                raise RuntimeError(f"Q buffer {qb} of CTA {c} overwritten with an S MMA pending")
        qbuf[(c, qb)] = ("loading", i)
        yield
        qbuf[(c, qb)] = i
        bars[(c, "QF", qb)].arrive()
        q_loaded[c] = i + 1
        yield

    def softmax(c, w):
        """Warpgroup w of CTA c: the steps t = w (mod 2) of every item, a full row per thread.  It
        takes the running max of step t-1 from the other warpgroup (MR[(t-1) % 2]) and hands its
        own to step t+1; warpgroup 0 also copies the query rows in."""
        if not work:
            return
        sv = pb = nq = 0
        mr_done = [0, 0]  # phases of MR[b] this warpgroup has seen complete or produced
        for i, n in enumerate(work):
            nxt = i + 1 if i + 1 < len(work) else None
            for t in range(n):
                b = t % 2
                if t % 2 != w:
                    mr_done[b] += 1  # the other warpgroup's step: its MR phase
                    continue
                vs = sv + t
                while not ready((c, "SF", vs % nbuf), vs // nbuf):
                    yield
                if sbuf[(c, vs % nbuf)] != ("S", (i, t)):
                    raise RuntimeError(f"softmax {c}.{w} reads {sbuf[(c, vs % nbuf)]} for S{(i, t)}")
                if t > 0:  # the max of step t-1
                    pb_ = 1 - b
                    while not ready((c, "MR", pb_), mr_done[pb_] - 1):
                        yield
                    if m_slot[(c, pb_)] != (i, t - 1):
                        raise RuntimeError(f"softmax {c}.{w} step {(i, t)} reads max {m_slot[(c, pb_)]}")
                    m_read.add((c, i, t - 1))
                prev = m_slot[(c, b)]
                if prev is not None and prev[1] + 1 < work[prev[0]] and (c,) + prev not in m_read:
                    raise RuntimeError(f"max of {prev} in CTA {c} overwritten unread")
                m_slot[(c, b)] = (i, t)
                bars[(c, "MR", b)].arrive()
                mr_done[b] += 1
                yield
                if t > 0 and rnd.random() < p_rescale:  # O rescaled: must hold PV(t-1)
                    vn = vs + nbuf - 1
                    while not ready((c, "SF", vn % nbuf), vn // nbuf):
                        yield
                    if o_state[c] != (i, t - 1):
                        raise RuntimeError(f"rescale of O in CTA {c} at {o_state[c]}, step {(i, t)}")
                sbuf[(c, vs % nbuf)] = ("P", (i, t))
                bars[(0, "PF", (pb + t) % nbuf)].arrive()
                yield
            while not ready((c, "OD"), nq):
                yield
            if o_state[c] != (i, n - 1):
                raise RuntimeError(f"epilogue of O in CTA {c} at {o_state[c]}, item {i}")
            bars[(c, "ML", nq % 2)].arrive()  # the two warpgroups swap their sums
            while not ready((c, "ML", nq % 2), nq // 2):
                yield
            o_read[c].add(i)
            yield
            sv += n + nbuf
            pb += n
            nq += 1

    def execute(op):
        if op[0] == "QK":
            _, b, sid, st, g = op
            for c in range(2):
                if ring[(c, "K")][st] != g or landed[(c, "K")][st] != g:
                    raise RuntimeError(f"S MMA {sid} reads K stage {st} of CTA {c}: "
                                       f"{ring[(c, 'K')][st]}")
                if qbuf[(c, sid[0] & 1)] != sid[0]:
                    raise RuntimeError(f"S MMA {sid} reads Q of CTA {c} = "
                                       f"{qbuf[(c, sid[0] & 1)]}")
                cur = sbuf[(c, b)]
                if cur is not None and cur[0] == "S":
                    raise RuntimeError(f"S MMA {sid} overwrites unread {cur} in CTA {c}")
                if cur is not None and cur[0] == "P" and cur[1] not in p_used:
                    raise RuntimeError(f"S MMA {sid} overwrites unused {cur} in CTA {c}")
                sbuf[(c, b)] = ("S", sid)
                reading[(c, "K")][st].discard(sid)
            qk_pending[op[2][0] & 1] -= 1
        elif op[0] == "PV":
            _, b, pid, st, g, t = op
            for c in range(2):
                if ring[(c, "V")][st] != g or landed[(c, "V")][st] != g:
                    raise RuntimeError(f"PV MMA {pid} reads V stage {st} of CTA {c}")
                if sbuf[(c, b)] != ("P", pid):
                    raise RuntimeError(f"PV MMA {pid} reads {sbuf[(c, b)]} in CTA {c}")
                if t == 0 and o_state[c] is not None and o_state[c][0] not in o_read[c]:
                    raise RuntimeError(f"PV MMA {pid} overwrites O of CTA {c} before its epilogue")
                o_state[c] = pid
                reading[(c, "V")][st].discard(pid)
            p_used.add(pid)
        elif op[0] == "DR":
            bars[(0, "DR")].arrive()
        elif op[0] == "QE":
            for c in range(2):
                bars[(c, "QE", op[1])].arrive()
        else:  # a commit multicast to both CTAs
            for c in range(2):
                bars[(c,) + op].arrive()

    alive = [producer(c, op, w) for c in range(2) for op in "KV" for w in range(producer_warps)]
    alive += [issuer(), relay()] + [softmax(c, w) for c in range(2) for w in range(2)]
    idle = 0
    while alive or tma[0] or tma[1] or pipe:
        r = rnd.random()
        if r < 0.15:
            c = rnd.randrange(2)
            if tma[c]:
                key, k, op, st, g = tma[c].pop(rnd.randrange(len(tma[c])))
                if ring[(c, op)][st] == g and not any(e[2] == op and e[3] == st and e[4] == g
                                                        for e in tma[c]):
                    landed[(c, op)][st] = g
                bars[key].complete_tx(k)
                idle = 0
                continue
        if r < 0.3 and pipe:
            execute(pipe.pop(0))
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
    for c in range(2):
        if o_read[c] != set(range(len(work))):
            raise RuntimeError(f"CTA {c} wrote out items {sorted(o_read[c])}")


STAGES, PRODUCER_WARPS, S_BUFFERS = 4, 3, 3  # the kernel's kStages, kPW and kSBuf


def test_random_item_lists():
    rng = random.Random(11)
    for trial in range(1200):
        items = [rng.choice([0, 1, 1, 2, 3, 4, 5, 7, 9]) for _ in range(rng.randint(1, 6))]
        simulate(items, STAGES, PRODUCER_WARPS, trial, nbuf=S_BUFFERS)
        simulate(items, STAGES, PRODUCER_WARPS, trial, nbuf=2)  # and with two buffers


@pytest.mark.parametrize("items", [[1] * 6, [2, 0, 1, 3], [16, 1, 9], [0, 0, 4], [3, 3, 3]])
def test_fixed_item_lists(items):
    for seed in range(100):
        simulate(items, STAGES, PRODUCER_WARPS, seed, nbuf=S_BUFFERS)


def test_a_ring_shallower_than_the_producer_warps_aliases_parity():
    """The kernel asserts kStages >= kPW at compile time; with fewer stages a producer warp can
    test a free barrier two phases early, which the model finds."""
    found = 0
    for seed in range(60):
        rng = random.Random(seed)
        items = [rng.choice([2, 3, 5, 7, 9]) for _ in range(rng.randint(1, 5))]
        try:
            simulate(items, 2, 3, seed)
        except RuntimeError as e:
            assert "parity alias" in str(e)
            found += 1
    assert found > 10


def test_query_copies_out_of_order_alias_parity():
    """The V producer warps that copy query rows in run ahead of the issuer by up to a ring; the
    copy of item i must wait for item i-1's, or its wait on QE can pass on an earlier phase."""
    found = 0
    for seed in range(60):
        items = [1] * 6 if seed % 2 else [1, 2, 1, 1, 3, 1]
        try:
            simulate(items, STAGES, PRODUCER_WARPS, seed, nbuf=S_BUFFERS, q_in_order=False)
        except RuntimeError as e:
            assert "parity alias" in str(e) or "overwritten" in str(e)
            found += 1
    assert found > 10
