"""The benchmark's named workloads have the shapes their recipes state (head counts, request
counts, prefix / extend / distinct lengths, shared-prefix structure, pool slots), and the work the
benchmark divides by (extend FLOPs over unmasked pairs, unique decode KV bytes, store bytes) is
what those shapes give.  Host only.  The full-size workloads are built structure-only
(values=False: the same draws in the same order, cached KV not written into pools), which the
first test shows gives the same tables, slots, lengths and inputs as the full build."""
import os
import sys

import numpy as np
import pytest

from prefix_shared_kv_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def rows_share(table, rows, n):
    """All the given table rows hold the same first n slots."""
    return all(np.array_equal(table[rows[0], :n], table[r, :n]) for r in rows[1:])


def distinct_tokens_have_distinct_slots(wl):
    """Every slot is one token: a slot that appears in two rows appears at the same position of
    both (a shared prefix), never as two different tokens; and every slot is inside the pool."""
    lengths = {}
    for st in wl.steps:
        for b in (st.extend, st.decode):
            if b is None:
                continue
            n = (b.prefix_len + b.extend_len) if b is st.extend else b.seq_len
            for r, k in zip(b.req_idx, n):
                lengths[int(r)] = max(lengths.get(int(r), 0), int(k))
    slots = np.concatenate([wl.req_to_token[r, :k] for r, k in lengths.items()]).astype(np.int64)
    pos = np.concatenate([np.arange(k) for k in lengths.values()]).astype(np.int64)
    assert slots.min() >= 0 and slots.max() < wl.pool_size
    pairs = np.unique(slots * (1 << 32) + pos)  # distinct (slot, position) pairs
    assert np.unique(pairs >> 32).size == pairs.size  # each slot at one position only
    return True


def test_structure_only_builds_are_the_benchmarks_workloads():
    assert W.NAMED["extend"] is W.llama7b_extend and W.NAMED["decode"] is W.llama7b_decode_hf
    assert W.NAMED["gqa-decode"] is W.llama3_gqa_decode and W.NAMED["radix-mixed"] is W.radix_mixed
    assert W.NAMED["chunked-prefill"] is W.llama3_chunked_prefill
    for make in (W.tiny, lambda values: W.tree_workload(
            3, 8, 8, depth=3, fanout=2, seg_lo=0, seg_hi=60, p_empty=0.2, n_decode=12,
            tail_hi=9, n_extend=5, own_hi=7, ext_lo=1, ext_hi=20, values=values)):
        a, b = make(values=True), make(values=False)
        assert b.k_pool.shape[0] == 0 and np.array_equal(a.req_to_token, b.req_to_token)
        for sa, sb in zip(a.steps, b.steps):
            assert np.array_equal(sa.store_slots, sb.store_slots)
            assert np.array_equal(sa.k_new, sb.k_new) and np.array_equal(sa.v_new, sb.v_new)
            for xa, xb in ((sa.extend, sb.extend), (sa.decode, sb.decode)):
                assert (xa is None) == (xb is None)
                if xa is not None:
                    assert np.array_equal(xa.q, xb.q) and np.array_equal(xa.req_idx, xb.req_idx)


def test_tiny():
    wl = W.tiny()
    assert (wl.num_q_heads, wl.num_kv_heads, wl.pool_size) == (8, 2, 4096)
    e = wl.steps[0].extend
    assert list(e.prefix_len) == [1000] * 4 and list(e.extend_len) == [40] * 4
    assert rows_share(wl.req_to_token, list(e.req_idx), 1000)
    assert [list(st.decode.seq_len) for st in wl.steps[1:]] == [[1041 + s] * 4 for s in range(8)]
    used = {int(s) for st in wl.steps for s in st.store_slots} | set(
        int(s) for s in wl.req_to_token[e.req_idx[0], :1000])
    assert len(used) == 1192 and distinct_tokens_have_distinct_slots(wl)


def test_extend_workload():
    wl = W.llama7b_extend(values=False)
    e = wl.steps[0].extend
    assert (wl.num_q_heads, wl.num_kv_heads) == (32, 32) and len(e.req_idx) == 64
    assert (e.prefix_len == 2000).all() and e.extend_len.min() >= 40 and e.extend_len.max() <= 200
    for g in range(4):
        assert rows_share(wl.req_to_token, list(e.req_idx[e.group_of_req == g]), 2000)
    assert distinct_tokens_have_distinct_slots(wl)
    w = bench.work_counts(wl)
    pairs = float(np.sum(e.extend_len * 2000.0 + e.extend_len * (e.extend_len + 1) / 2.0))
    assert w["extend_flops"] == pytest.approx(4 * 128 * 32 * pairs)
    assert w["extend_flops"] == pytest.approx(2.604e11, rel=0.1)  # E ~ U[40, 200], mean 120


@pytest.mark.parametrize("name,hkv,prefix,lo,hi,tokens", [
    ("decode", 32, 2000, 100, 500, 108800),
    ("gqa-decode", 8, 16000, 200, 1000, 409600)])
def test_decode_workloads(name, hkv, prefix, lo, hi, tokens):
    wl = W.NAMED[name](values=False)
    d = wl.steps[0].decode
    assert (wl.num_q_heads, wl.num_kv_heads) == (32, hkv) and len(d.req_idx) == 256
    own = d.seq_len - prefix
    assert own.min() >= lo and own.max() <= hi
    for g in range(16):
        assert (d.group_of_req == g).sum() == 16
        assert rows_share(wl.req_to_token, list(d.req_idx[d.group_of_req == g]), prefix)
    if name == "gqa-decode":
        assert wl.pool_size >= 409600
    assert distinct_tokens_have_distinct_slots(wl)
    w = bench.work_counts(wl)
    unique = 16 * prefix + int(own.sum())
    assert w["decode_kv_bytes"] == unique * hkv * 128 * 2 * 2
    assert unique == pytest.approx(tokens, rel=0.05)


def test_radix_mixed():
    wl = W.radix_mixed(values=False)
    st = wl.steps[0]
    e, d = st.extend, st.decode
    assert (wl.num_q_heads, wl.num_kv_heads, wl.pool_size) == (32, 32, 32768)
    assert sorted(zip(e.prefix_len.tolist(), e.extend_len.tolist())) == \
        [(0, 1500)] * 8 + [(1700, 64)] * 16
    assert len(d.req_idx) == 40 and (d.seq_len - 1700).min() >= 1 and (d.seq_len - 1700).max() <= 32
    assert len(st.store_slots) == 16 * 64 + 8 * 1500 + 40
    # the tree: the 1000-token system prompt under every hit, a 500-token branch under four
    # leaves, a 200-token leaf under its requests
    hits = list(e.req_idx[e.prefix_len > 0]) + list(d.req_idx)
    assert rows_share(wl.req_to_token, hits, 1000)
    par, gpl = d.group_parent, d.group_prefix_len
    assert list(gpl[:1]) == [1000] and (gpl[1:9] == 1500).all() and (gpl[9:] == 1700).all()
    for leaf in range(9, 41):
        assert par[leaf] == 1 + (leaf - 9) // 4
        members = list(d.req_idx[d.group_of_req == leaf])
        assert rows_share(wl.req_to_token, members, 1700)
    assert distinct_tokens_have_distinct_slots(wl)
    w = bench.work_counts(wl)
    assert w["extend_flops"] == 4 * 128 * 32 * 10780080  # unmasked pairs, exactly
    tails = int((d.seq_len - 1700).sum())
    # tree-unique decode KV: 1,000 + 8 x 500 + the 32 leaves' 200 (every leaf has a request:
    # requests j and j + 32 share leaf j) + each request's own tail
    assert w["decode_kv_bytes"] == (1000 + 8 * 500 + 32 * 200 + tails) * 32 * 512
    assert w["store_bytes"] == 13064 * 32 * 256 * 2 * 2


def test_chunked_prefill():
    wl = W.llama3_chunked_prefill(values=False)
    assert (wl.num_q_heads, wl.num_kv_heads) == (32, 8) and len(wl.steps) == 3
    for i, st in enumerate(wl.steps):
        e, d = st.extend, st.decode
        assert list(e.extend_len) == [2048] and list(e.prefix_len) == [1024 + 2048 * i]
        assert len(d.req_idx) == 64
        own = d.seq_len - 1024 - i - 1  # own cached tail: U[200, 1000], one new token a step
        assert own.min() >= 200 and own.max() <= 1000
        if i:
            assert (own == wl.steps[0].decode.seq_len - 1024 - 1).all()
    assert distinct_tokens_have_distinct_slots(wl)


def test_paged():
    """The block-granular configuration: every key position p of a request sits in slot
    page * 16 + p % 16 of one of its pages, so every whole page is a run of 16 consecutive
    slots."""
    assert W.NAMED["paged"] is W.llama7b_paged
    a = W.paged_workload(5, 4, 2, page=16, prefix=90, n_req=3, ext_lo=1, ext_hi=40)
    b = W.paged_workload(5, 4, 2, page=16, prefix=90, n_req=3, ext_lo=1, ext_hi=40,
                         values=False)
    assert b.k_pool.shape[0] == 0 and np.array_equal(a.req_to_token, b.req_to_token)
    wl = W.NAMED["paged"](values=False)
    e = wl.steps[0].extend
    assert (wl.num_q_heads, wl.num_kv_heads) == (32, 32) and len(e.req_idx) == 64
    assert (e.prefix_len == 2000).all() and e.extend_len.min() >= 40 and e.extend_len.max() <= 200
    assert rows_share(wl.req_to_token, list(e.req_idx), 2000)
    assert distinct_tokens_have_distinct_slots(wl)
    for r, p, x in zip(e.req_idx, e.prefix_len, e.extend_len):
        s = wl.req_to_token[r, :p + x].astype(np.int64)
        assert (s % 16 == np.arange(p + x) % 16).all()          # position p in slot 16 k + p % 16
        full = (p + x) // 16 * 16
        assert (np.diff(s[:full].reshape(-1, 16), axis=1) == 1).all()  # whole pages are runs
