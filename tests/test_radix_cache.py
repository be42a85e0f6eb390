"""Host radix cache memory management: LRU eviction of unheld leaves, reference counts, a slot pool
shared with running requests (SGLang explainer, "LRU退避"; SGLang paper notes §3 and Figure 3).

The library (C ABI) is checked against oracle.radix.LRURadixCache, a plain list-based model
written separately from the pages, on random operation sequences, and both are replayed through
the nine steps of the pages' Figure 3 with run lengths chosen so that the evictions the pages
narrate are exactly what LRU with reference counts must do (the pages give no token counts).
"""
import numpy as np
import pytest

from oracle.radix import LRURadixCache
from prefix_shared_kv_gb300 import rx


class Cache:
    """Drives the library's tree + slot pool and the model side by side."""

    def __init__(self, pool_size):
        self.t, self.pool = rx.Radix(), rx.SlotPool(pool_size)
        self.m, self.m_free = LRURadixCache(), list(range(pool_size))
        self.P = pool_size

    def request(self, prompt, generated):
        """A request: hold its cached prefix, take slots for the rest (evicting if short), insert
        the whole sequence, release.  Returns the slots each side evicted."""
        seq = list(prompt) + list(generated)
        s_lib, sl_lib = self.t.acquire(prompt, lock=True)
        s_m, sl_m = self.m.acquire(prompt, lock=True)
        assert s_lib == s_m and list(sl_lib) == list(sl_m)
        need = len(seq) - s_lib
        ev_lib, ev_m = [], []
        if need > self.pool.free_count():
            ev_lib = list(self.t.evict(need - self.pool.free_count()))
            self.pool.release(ev_lib)
        if need > len(self.m_free):
            ev_m = self.m.evict(need - len(self.m_free))
            self.m_free += ev_m
        assert ev_lib == ev_m
        new_lib = self.pool.alloc(need)
        new_m, self.m_free = self.m_free[:need], self.m_free[need:]
        assert list(new_lib) == new_m
        slots = list(sl_lib) + list(new_lib)
        n_lib = self.t.insert(seq, slots)
        n_m = self.m.insert(seq, slots)
        assert n_lib == n_m == need
        self.t.release(prompt[:s_lib])
        self.m.release(prompt[:s_m])
        assert self.t.stats() == self.m.stats()
        assert self.t.stats()[0] + self.pool.free_count() == self.P
        return ev_lib, slots


def runs(*lengths, start):
    out, t = [], start
    for n in lengths:
        out.append(list(range(t, t + n)))
        t += n
    return out


def test_figure3_nine_steps():
    # run lengths: system prompt, chat 1 turn 1 (user + answer), chat 1 turn 2 ("c"), chat 2 turns
    # 1 and 2, few-shot examples, three few-shot queries (question + answer), a new chat-1 message
    S, T1, C2, H, G, E = runs(4, 4, 20, 16, 5, 4, start=1000)
    Q = [runs(2, 1, start=2000 + 10 * i) for i in range(3)]      # question, answer
    U5 = runs(4, start=3000)[0]
    c = Cache(45)
    # (1) empty; (2) chat 1 first turn: one new node
    c.request(S + T1[:2], T1[2:])
    assert c.t.stats() == (8, 1)
    # (3) chat 1 second turn: prefix reused, the new turn is a new node below it
    ev, _ = c.request(S + T1 + C2[:8], C2[8:])
    assert ev == [] and c.t.stats() == (28, 2)
    # (4) a second chat session: the first node splits so both share the system prompt
    ev, _ = c.request(S + H[:6], H[6:])
    assert ev == [] and c.t.stats() == (44, 4)
    assert c.t.match(S + [1])[0] == 4          # the system prompt is a node of its own now
    # (5) chat 2 continues; short of memory, the least recently used leaf (chat 1's second turn,
    #     "c") is evicted, and only it
    _, c2_slots = c.t.match(S + T1 + C2)
    ev, _ = c.request(S + H + G[:2], G[2:])
    assert ev == list(c2_slots[8:])
    assert c.t.stats() == (29, 4)
    # (6) a few-shot query shares nothing: a new branch at the root
    ev, _ = c.request(E + Q[0][0], Q[0][1])
    assert ev == [] and c.t.stats() == (36, 5)
    # (7) more few-shot queries on the same examples: the few-shot node splits at the examples
    for i in (1, 2):
        ev, _ = c.request(E + Q[i][0], Q[i][1])
        assert ev == []
    assert c.t.stats() == (42, 8)
    assert c.t.match(E + [0])[0] == 4
    # (8) a new message in chat 1 (its evicted turn is recomputed): the least recently used
    #     leaves are chat 2's two nodes, evicted leaf first, and nothing else
    _, g_slots = c.t.match(S + H + G)
    ev, _ = c.request(S + T1 + C2 + U5[:2], U5[2:])
    assert ev == list(g_slots[20:]) + list(g_slots[4:20])
    assert c.t.match(S + H)[0] == 4
    # (9) three sampled answers to the second few-shot question: the three least recently used
    #     unheld leaves go (the first query, the old answer, the third query); chat 1's node from
    #     (8) stays
    kept = c.t.match(S + T1 + C2 + U5)[0]
    evicted = []
    for k in range(3):
        ev, _ = c.request(E + Q[1][0], [4000 + 2 * k, 4001 + 2 * k])
        evicted += ev
    assert c.t.match(S + T1 + C2 + U5)[0] == kept == len(S + T1 + C2 + U5)
    assert c.t.match(E + Q[0][0])[0] == 4 and c.t.match(E + Q[2][0])[0] == 4
    assert c.t.match(E + Q[1][0] + Q[1][1])[0] == 6   # the old answer went
    assert len(evicted) == 3 + 1 + 3


@pytest.mark.parametrize("seed", range(6))
def test_random_operations_match_the_model(seed):
    rng = np.random.default_rng(seed)
    P = 400
    c = Cache(P)
    held = []                          # prompts currently held by running requests
    vocab = 12                         # few token values: many shared prefixes and splits
    for _ in range(160):
        op = rng.random()
        if op < 0.55 or not held:
            plen = int(rng.integers(1, 30))
            base = held[int(rng.integers(len(held)))] if held and rng.random() < 0.5 else []
            prompt = list(base[:int(rng.integers(0, len(base) + 1))]) + \
                [int(x) for x in rng.integers(0, vocab, size=plen)]
            gen = [int(x) for x in rng.integers(100, 200, size=int(rng.integers(1, 8)))]
            try:
                c.request(prompt, gen)
            except rx.RxError as e:    # pool exhausted with everything held: both sides agree
                assert e.status == rx.RX_ERR_WORKSPACE
                return
        elif op < 0.75:
            p = [int(x) for x in rng.integers(0, vocab, size=int(rng.integers(1, 20)))]
            unit = int(rng.integers(1, 4))
            a = c.t.acquire(p, match_unit=unit, lock=True)
            b = c.m.acquire(p, unit=unit, lock=True)
            assert a[0] == b[0] and list(a[1]) == b[1]
            held.append(p[:a[0]])
        elif op < 0.9:
            p = held.pop(int(rng.integers(len(held))))
            c.t.release(p)
            c.m.release(p)
        else:
            n = int(rng.integers(1, 60))
            a = list(c.t.evict(n))
            b = c.m.evict(n)
            assert a == b
            c.pool.release(a)
            c.m_free += b
        assert c.t.stats() == c.m.stats()


def test_release_checks_and_held_prefix_survives_eviction():
    t = rx.Radix()
    t.insert(list(range(10)), list(range(10)))
    saved, _ = t.acquire(list(range(6)) + [99], lock=True)
    assert saved == 6
    with pytest.raises(rx.RxError):
        t.release(list(range(5)))      # not a node boundary
    freed = t.evict(100)               # only the unheld tail can go
    assert list(freed) == [6, 7, 8, 9] and t.stats() == (6, 1)
    t.release(list(range(6)))
    assert list(t.evict(100)) == list(range(6))
    with pytest.raises(rx.RxError):
        t.release(list(range(6)))
    pool = rx.SlotPool(4)
    with pytest.raises(rx.RxError) as e:
        pool.alloc(5)
    assert e.value.status == rx.RX_ERR_WORKSPACE
    with pytest.raises(rx.RxError) as e:
        pool.release([7])
    assert e.value.status == rx.RX_ERR_RANGE
