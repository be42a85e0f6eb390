"""Host-side validation of the two contracts the attention and store calls trust (no GPU needed):
every row that declares a shared prefix really holds the same slots there (SGLang explainer,
RadixAttention: requests under one tree node share that node's KV pages; BatchLLM explainer,
Global Prefix Sharing: a group's common prefix is one KV context), and store slots are distinct
pool slots.  The table check is compared with a brute force over all pairs of requests below each
group, on random forests, and on the synthetic workloads the kernels are tested with."""
import numpy as np
import pytest

from prefix_shared_kv_gb300 import rx, workloads as W

RANGE, INVALID = 2, 1


def status_of(fn, *a, **k):
    try:
        fn(*a, **k)
        return 0, -1
    except rx.RxError as e:
        return e.status, e.bad


def brute_force_contract(table, req_idx, group_of_req, gpl, parent):
    """True when, for every group g, all requests whose path holds g agree on their first
    gpl[g] entries (all pairs compared)."""
    def path(g):
        while g >= 0:
            yield g
            g = parent[g] if parent is not None else -1
    members = {g: [] for g in range(len(gpl))}
    for b, g in enumerate(group_of_req):
        for a in path(g):
            members[a].append(b)
    for g, bs in members.items():
        n = gpl[g]
        for i in bs:
            for j in bs:
                if not np.array_equal(table[req_idx[i], :n], table[req_idx[j], :n]):
                    return False
    return True


def random_forest_case(rng):
    G = int(rng.integers(1, 6))
    parent = np.full(G, -1, np.int32)
    gpl = np.zeros(G, np.int32)
    for g in range(G):
        parent[g] = int(rng.integers(-1, g)) if g > 0 else -1
        base = gpl[parent[g]] if parent[g] >= 0 else 0
        gpl[g] = base + int(rng.integers(0, 6))
    B = int(rng.integers(1, 9))
    group_of_req = rng.integers(-1, G, B).astype(np.int32)
    stride = int(gpl.max()) + 8
    pool = 64
    table = rng.integers(0, pool, (B + 2, stride)).astype(np.int32)
    req_idx = rng.permutation(B + 2)[:B].astype(np.int32)
    # make the declared prefixes shared: copy each node's own keys from one source row
    for g in range(G):
        lo = gpl[parent[g]] if parent[g] >= 0 else 0
        src = rng.integers(0, pool, gpl[g] - lo)
        for b in range(B):
            a = group_of_req[b]
            while a >= 0 and a != g:
                a = parent[a]
            if a == g:
                table[req_idx[b], lo:gpl[g]] = src
    key_len = np.array([rng.integers(gpl[g] if g >= 0 else 0, stride + 1) for g in group_of_req],
                       np.int32)
    return table, pool, req_idx, key_len, group_of_req, gpl, parent


def test_check_tables_agrees_with_brute_force_on_random_forests(librx):
    rng = np.random.default_rng(0)
    seen = {0: 0, INVALID: 0}
    for _ in range(400):
        table, pool, req_idx, key_len, grp, gpl, parent = random_forest_case(rng)
        if rng.random() < 0.6:  # plant a change in some row's declared prefix
            b = int(rng.integers(0, len(req_idx)))
            if grp[b] >= 0 and gpl[grp[b]] > 0:
                j = int(rng.integers(0, gpl[grp[b]]))
                table[req_idx[b], j] = (table[req_idx[b], j] + 1) % pool
        st, bad = status_of(rx.check_tables, table, pool, req_idx, key_len, grp, gpl, parent)
        ok = brute_force_contract(table, req_idx, grp, gpl, parent)
        assert st == (0 if ok else INVALID), (st, ok)
        assert (bad == -1) == ok
        seen[st] += 1
    assert seen[0] > 50 and seen[INVALID] > 50


@pytest.mark.parametrize("kind", ["extend", "decode", "tree", "radix-mixed"])
def test_workload_tables_and_slots_pass(librx, kind):
    if kind == "extend":
        wl = W.extend_workload(1, 8, 2, n_groups=3, members=5, prefix=300, ext_lo=1, ext_hi=90,
                               own_cached_hi=30, ungrouped=2, ungrouped_prefix=50)
    elif kind == "decode":
        wl = W.decode_workload(2, 8, 2, n_groups=3, members=7, prefix=400, dist_lo=1,
                               dist_hi=100, ungrouped=2)
    elif kind == "tree":
        wl = W.tree_workload(3, 8, 8, depth=3, fanout=3, seg_lo=0, seg_hi=80, p_empty=0.2,
                             n_decode=20, tail_hi=30, n_extend=5, own_hi=20, ext_lo=1,
                             ext_hi=40)
    else:
        wl = W.radix_mixed(values=False)
    for st in wl.steps:
        rx.check_slots(st.store_slots, wl.pool_size)
        if st.extend is not None:
            e = st.extend
            rx.check_tables(wl.req_to_token, wl.pool_size, e.req_idx, e.prefix_len + e.extend_len,
                            e.group_of_req, e.group_prefix_len, e.group_parent)
        if st.decode is not None:
            d = st.decode
            rx.check_tables(wl.req_to_token, wl.pool_size, d.req_idx, d.seq_len, d.group_of_req,
                            d.group_prefix_len, d.group_parent)


def test_check_tables_names_the_request_that_breaks_a_shared_prefix(librx):
    wl = W.decode_workload(4, 8, 8, n_groups=2, members=4, prefix=100, dist_lo=1, dist_hi=20)
    d = wl.steps[0].decode
    t = wl.req_to_token.copy()
    members = np.flatnonzero(d.group_of_req == 1)
    victim = int(members[2])  # not the group's first request
    t[d.req_idx[victim], 57] = (t[d.req_idx[victim], 57] + 1) % wl.pool_size
    st, bad = status_of(rx.check_tables, t, wl.pool_size, d.req_idx, d.seq_len, d.group_of_req,
                        d.group_prefix_len)
    assert (st, bad) == (INVALID, victim)
    # the same change past the shared prefix (the request's own keys) breaks nothing
    t = wl.req_to_token.copy()
    j = int(d.group_prefix_len[1])
    t[d.req_idx[victim], j] = (t[d.req_idx[victim], j] + 1) % wl.pool_size
    assert status_of(rx.check_tables, t, wl.pool_size, d.req_idx, d.seq_len, d.group_of_req,
                     d.group_prefix_len) == (0, -1)


def test_check_tables_range_errors(librx):
    t = np.arange(40, dtype=np.int32).reshape(4, 10)  # row r holds slots 10r .. 10r+9
    ri = np.array([0, 3], np.int32)
    assert status_of(rx.check_tables, t, 40, ri, [10, 3]) == (0, -1)
    assert status_of(rx.check_tables, t, 39, ri, [10, 10]) == (RANGE, 1)  # slot 39 not in pool
    assert status_of(rx.check_tables, t, 40, ri, [11, 3]) == (RANGE, 0)   # longer than the row
    assert status_of(rx.check_tables, t, 40, [0, 4], [1, 1]) == (RANGE, 1)  # row outside table
    t2 = t.copy()
    t2[3, 2] = -5
    assert status_of(rx.check_tables, t2, 40, ri, [10, 3]) == (RANGE, 1)
    assert status_of(rx.check_tables, t2, 40, ri, [10, 2]) == (0, -1)  # not a key it reads
    # a request shorter than its group's prefix; a group out of range; a bad forest
    assert status_of(rx.check_tables, t, 40, ri, [10, 3], [0, 0], [5])[0] == RANGE
    assert status_of(rx.check_tables, t, 40, ri, [10, 3], [0, 1], [2])[0] == RANGE
    assert status_of(rx.check_tables, t, 40, ri, [10, 10], [0, 1], [2, 1], [-1, 0])[0] == RANGE


def test_check_slots(librx):
    assert status_of(rx.check_slots, np.zeros(0, np.int32), 10) == (0, -1)
    assert status_of(rx.check_slots, [3, 1, 2, 0], 4) == (0, -1)
    assert status_of(rx.check_slots, [3, 1, 4, 0], 4) == (RANGE, 2)
    assert status_of(rx.check_slots, [3, -1, 2], 4) == (RANGE, 1)
    # the earliest repeat is named: slot 1 at index 3 repeats index 1; slot 5 repeats later
    assert status_of(rx.check_slots, [5, 1, 7, 1, 5, 1], 8) == (INVALID, 3)
    rng = np.random.default_rng(3)
    for _ in range(200):
        n = int(rng.integers(1, 40))
        s = rng.integers(0, 50, n).astype(np.int32)
        first_rep = next((i for i in range(n) if s[i] in s[:i]), -1)
        st, bad = status_of(rx.check_slots, s, 50)
        assert (st, bad) == ((0, -1) if first_rep < 0 else (INVALID, first_rep))
