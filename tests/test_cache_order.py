"""Cache-aware ordering (SGLang paper notes, §3 and App. A.3, Theorem 3.1): with a cache at least
as large as the longest request, the depth-first order of the batch's radix tree computes every
edge's KV once, the least any order can compute.  Checked by brute force over all orders of small
random batches, with the oracle's LRU radix cache; the library's rx_dfs_order gives the order."""
import itertools

import numpy as np
import pytest

from oracle import radix as R
from prefix_shared_kv_gb300 import rx


def random_batch(rng, n):
    # a few shared stems with branches, some requests a prefix of others
    stems = [list(rng.integers(0, 50, size=int(rng.integers(1, 6)))) for _ in range(3)]
    batch = []
    for _ in range(n):
        q = list(stems[int(rng.integers(0, 3))])
        for _ in range(int(rng.integers(0, 3))):
            q += list(rng.integers(0, 4, size=int(rng.integers(1, 4))))
        batch.append([int(x) for x in q])
    return batch


@pytest.mark.parametrize("seed", range(12))
def test_dfs_order_is_optimal_by_brute_force(seed):
    rng = np.random.default_rng(seed)
    batch = random_batch(rng, int(rng.integers(3, 7)))
    cap = max(len(q) for q in batch)                     # the theorem's smallest cache
    order = rx.dfs_order(batch)
    assert sorted(order.tolist()) == list(range(len(batch)))
    best = min(R.computed_tokens(batch, p, cap) for p in itertools.permutations(range(len(batch))))
    c_min = R.edge_tokens(batch)
    assert best == c_min                                 # every edge once is reachable ...
    assert R.computed_tokens(batch, order.tolist(), cap) == c_min   # ... and DFS reaches it
    # a bigger cache cannot do worse
    assert R.computed_tokens(batch, order.tolist(), 10 * cap) == c_min
    # longest-shared-prefix-first, run online, reaches it as well on these batches
    assert R.computed_tokens(batch, R.longest_prefix_first(batch, cap), cap) == c_min


def test_dfs_order_worked_example():
    batch = [[1, 2, 3, 4], [5, 6], [1, 2, 9], [1, 2], [5, 7, 8]]
    assert rx.dfs_order(batch).tolist() == [3, 0, 2, 1, 4]
    # 1-2 | 3-4 | 9 | 5 | 6 | 7-8: 9 edge tokens; cache hit rate 1 - 9 / 14 (App. A.3 formula)
    assert R.edge_tokens(batch) == 9
    assert R.computed_tokens(batch, [0, 1, 2, 3, 4], 4) > 9    # arrival order recomputes 1-2


def test_gain_rule_groups_worked_examples():
    # BatchLLM explainer's tree shape (system prompt -> few-shot sets -> queries), with counts of
    # our own: gain(A) = (4 - 1) * 50 = 150 > tokens(system) = 100 -> A is a group of its own;
    # gain(B) = (2 - 1) * 10 = 10 -> B's queries stay in the system prompt's group
    sysp, A, B = list(range(100)), list(range(1000, 1050)), list(range(2000, 2010))
    batch = [sysp + A + [3000 + i] for i in range(4)] + [sysp + B + [4000 + i] for i in range(2)]
    grp, gpl = rx.gain_groups(batch)
    assert gpl.tolist() == [100, 150]
    assert grp.tolist() == [1, 1, 1, 1, 0, 0]
    # gain equal to the penalty does not split ("exceeds"): (3 - 1) * 50 = 100
    batch = [sysp + A + [3000 + i] for i in range(3)] + [sysp + B + [4000 + i] for i in range(2)]
    grp, gpl = rx.gain_groups(batch)
    assert gpl.tolist() == [100] and grp.tolist() == [0] * 5
    # recursive: under A (50 tokens) a sub-stem C of 30 tokens with 3 requests: 2 * 30 = 60 > 50
    C = list(range(5000, 5030))
    batch = [sysp + A + C + [6000 + i] for i in range(3)] + \
        [sysp + A + [3000 + i] for i in range(2)] + [sysp + B + [4000 + i] for i in range(2)]
    grp, gpl = rx.gain_groups(batch)
    assert sorted(gpl.tolist()) == [100, 150, 180]
    g180 = gpl.tolist().index(180)
    assert grp.tolist()[:3] == [g180] * 3
    # a lone request and a root branch with one request form no group
    grp, gpl = rx.gain_groups([[1, 2, 3], [9, 9]])
    assert grp.tolist() == [-1, -1] and len(gpl) == 0


@pytest.mark.parametrize("seed", range(8))
def test_gain_groups_are_shared_prefixes(seed):
    rng = np.random.default_rng(100 + seed)
    batch = random_batch(rng, 12)
    grp, gpl = rx.gain_groups(batch)
    for g, plen in enumerate(gpl.tolist()):
        members = [batch[r] for r in range(len(batch)) if grp[r] == g]
        assert len(members) >= 1
        assert all(len(q) >= plen for q in members)
        assert all(q[:plen] == members[0][:plen] for q in members)
