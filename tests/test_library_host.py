"""Host-side checks of the C ABI (no GPU needed): the library loads and exports every symbol the
header declares; the radix cache and the accounting agree with the oracle and the pages' values;
argument checks reject bad input before anything would be launched."""
import json
import os
import re

import numpy as np
import pytest

from oracle import accounting, radix as oradix
from prefix_shared_kv_gb300 import rx, workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = os.path.join(ROOT, "tests", "golden")


def declared_functions():
    text = open(os.path.join(ROOT, "include", "rx.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(rx_[a-z_0-9]+)\s*\(", text)))


def test_library_exports_every_declared_symbol(librx):
    names = declared_functions()
    assert len(names) >= 20
    for n in names:
        assert hasattr(librx, n), n
    assert sorted(rx.EXPORTED) == names


def test_noalloc_scratch_size_is_the_headers(librx):
    text = open(os.path.join(ROOT, "include", "rx.h")).read()
    m = re.search(r"#define RX_NOALLOC_SCRATCH_BYTES \(\(size_t\)(\d+) << (\d+)\)", text)
    assert m, "RX_NOALLOC_SCRATCH_BYTES not found in rx.h"
    assert rx.noalloc_scratch_bytes() == int(m.group(1)) << int(m.group(2))


def test_radix_matches_oracle_on_random_sequences(librx):
    rng = np.random.default_rng(0)
    for trial in range(60):
        tree, store = rx.Radix(), oradix.PrefixStore()
        next_slot = 0
        for _ in range(rng.integers(1, 12)):
            base = list(rng.integers(0, 4, rng.integers(0, 30)))
            slots = list(range(next_slot, next_slot + len(base)))
            next_slot += len(base)
            before = store.longest(base)
            added = tree.insert(base, slots)
            store.insert(base, slots)
            assert added == len(base) - before
        for _ in range(20):
            q = list(rng.integers(0, 4, rng.integers(0, 35)))
            for u in (1, 3, 16):
                saved, slots = tree.match(q, u)
                o_saved, o_slots = store.match(q, u)
                assert saved == o_saved
                assert list(slots) == list(o_slots)
        assert tree.stats()[0] == len(store)


def test_radix_worked_example(librx):
    g = json.load(open(os.path.join(GOLDEN, "prefix_cache_worked_example.json")))
    rng = np.random.default_rng(1)
    common = rng.integers(0, 16000, g["common_prefix_tokens"])
    tree = rx.Radix()
    first = np.concatenate([common, rng.integers(16000, 32000, g["question_tokens"])])
    tree.insert(first, np.arange(first.size))
    second = np.concatenate([common, rng.integers(16000, 32000, g["question_tokens"])])
    assert tree.match(second, 16)[0] == 992
    assert tree.match(second, 1)[0] == 1000
    ts = rng.integers(16000, 32000, 3)
    assert tree.match(np.concatenate([ts, second]), 1)[0] == 0
    assert tree.match(np.concatenate([ts, second]), 16)[0] == 0
    np.testing.assert_array_equal(tree.match(second, 1)[1], np.arange(1000))


def test_radix_split_keeps_first_slots_and_counts_nodes(librx):
    t = rx.Radix()
    assert t.insert([1, 2, 3, 4], [10, 11, 12, 13]) == 4
    assert t.insert([1, 2, 9], [20, 21, 22]) == 1
    assert t.stats() == (5, 3)          # root -> [1,2] -> {[3,4], [9]}
    assert list(t.match([1, 2, 9, 7])[1]) == [10, 11, 22]
    assert t.insert([1, 2], [30, 31]) == 0
    assert t.insert([5], [40]) == 1
    assert t.stats() == (6, 4)


def test_accounting_matches_oracle_and_pages(librx):
    g = json.load(open(os.path.join(GOLDEN, "closed_forms.json")))
    for c in g["token_saving_ratio"]["cases"]:
        logical = c["sharing"] * (c["prefix"] + c["distinct_inferred"])
        processed = c["prefix"] + c["sharing"] * c["distinct_inferred"]
        v = rx.token_saving(processed, logical)
        assert v == accounting.token_saving_ratio(processed, logical)
        assert round(v, 1) == c["printed_percent"]
    cr = g["compute_reduction"]
    assert rx.compute_reduction(cr["l_prefix"], cr["l_new"]) == accounting.compute_reduction(
        cr["l_prefix"], cr["l_new"])
    for m in range(0, 2000, 7):
        for u in (1, 16, 32):
            assert rx.saved_tokens(m, u) == oradix.PrefixStore().match([], 1)[0] + m // u * u
    assert np.isnan(rx.token_saving(1, 0))


def _desc(rows=4, stride=64, hq=8, hkv=2, pool=128):
    return rx.KVDesc(hq, hkv, 128, 128 ** -0.5, pool, 0x1000, rows, stride)


def test_plan_argument_checks(librx):
    p = rx.Plan()
    d = _desc()
    with pytest.raises(rx.RxError) as e:
        rx.decode_plan(p, d, [0, 9], [5, 5])            # row 9 outside a 4-row table
    assert e.value.status == rx.RX_ERR_RANGE
    with pytest.raises(rx.RxError) as e:
        rx.decode_plan(p, d, [0], [65])                 # longer than the stride
    assert e.value.status == rx.RX_ERR_RANGE
    with pytest.raises(rx.RxError) as e:
        rx.decode_plan(p, d, [0, 1], [5, 3], [0, 0], [4])  # group prefix > seq_len of a member
    assert e.value.status == rx.RX_ERR_RANGE
    with pytest.raises(rx.RxError) as e:
        rx.extend_plan(p, d, [0], [10], [-1])
    assert e.value.status == rx.RX_ERR_INVALID
    with pytest.raises(rx.RxError) as e:
        rx.extend_plan(p, _desc(hq=6, hkv=2), [0], [1], [1])
    assert e.value.status == rx.RX_ERR_UNSUPPORTED
    bad = _desc()
    bad.head_dim = 64
    with pytest.raises(rx.RxError) as e:
        rx.decode_plan(p, bad, [0], [1])
    assert e.value.status == rx.RX_ERR_UNSUPPORTED
    # a plan that was never built cannot size a workspace
    with pytest.raises(rx.RxError):
        rx.Plan().workspace_size()


def test_size_limits_are_refused_on_the_host(librx):
    """Limits of the int32 tables, refused by the planners before any row is built (planning only:
    no attention call is made with these descriptors)."""
    p = rx.Plan()
    big = _desc(rows=2, stride=1 << 30)
    with pytest.raises(rx.RxError) as e:  # 2^31 new rows in one batch
        rx.extend_plan(p, big, [0, 1], [0, 0], [1 << 30, 1 << 30])
    assert e.value.status == rx.RX_ERR_RANGE
    with pytest.raises(rx.RxError) as e:  # a pool of 2^31 slots
        rx.decode_plan(p, _desc(pool=1 << 31), [0], [1])
    assert e.value.status == rx.RX_ERR_INVALID
    with pytest.raises(rx.RxError) as e:  # a decode request must attend to its own token
        rx.decode_plan(p, _desc(), [0], [0])
    assert e.value.status in (rx.RX_ERR_INVALID, rx.RX_ERR_RANGE)
    with pytest.raises(rx.RxError) as e:  # more than 256 KV heads
        rx.decode_plan(p, _desc(hq=512, hkv=512), [0], [1])
    assert e.value.status == rx.RX_ERR_UNSUPPORTED


def test_plans_size_workspaces_without_a_gpu(librx):
    p = rx.Plan()
    d = _desc(rows=8, stride=4096, hq=32, hkv=8)
    rx.decode_plan(p, d, list(range(8)), [3000] * 8, [0] * 4 + [1] * 4, [2000, 1000])
    n_dec = p.workspace_size()
    # partials: every unit keeps one fp32 row of 128 + lse per (KV head, query row)
    assert n_dec > 8 * 32 * 129 * 4
    rx.extend_plan(p, d, list(range(8)), [2000] * 8, [100] * 8, [0] * 8, [2000])
    assert 256 < p.workspace_size() < n_dec
    # using an extend plan for decode is rejected before any launch
    with pytest.raises(rx.RxError) as e:
        rx.decode_attn(p, d, 16, 16, 16, 16, 16, None, stream=0)
    assert e.value.status == rx.RX_ERR_INVALID


def test_empty_batches_plan_to_no_work(librx):
    d = _desc(rows=1, stride=16, hq=4, hkv=2)
    p = rx.Plan()
    rx.extend_plan(p, d, [], [], [], [], [])
    assert p.workspace_size() == 256 and p.key_reads() == 0  # the header alone
    rx.decode_plan(p, d, [], [], [], [])
    assert p.key_reads() == 0 and p.launches() == 0


def test_binding_rejects_arrays_of_different_lengths(librx):
    p, d = rx.Plan(), _desc()
    with pytest.raises(ValueError):
        rx.extend_plan(p, d, [0], [10], [3], [])          # a group entry missing
    with pytest.raises(ValueError):
        rx.decode_plan(p, d, [0, 1], [5])                 # a length missing
    with pytest.raises(ValueError):
        rx.decode_plan(p, d, [0], [5], [0], [3, 4], [-1])  # a parent missing


def test_plan_launch_counts(librx):
    """What rx_plan_launches reports: one tensor-core launch for extend work; for decode, the
    tensor-core kernel only when a shared-prefix unit stacks >= 32 query rows per KV head, the
    mma.sync kernel for the rest, and the merge."""
    d = _desc(rows=40, stride=4096, hq=8, hkv=2)  # 4 query heads per KV head
    p = rx.Plan()
    rx.extend_plan(p, d, [0, 1], [100, 100], [10, 10], [0, 0], [100])
    assert p.launches() == 1
    rx.extend_plan(p, d, [0], [100], [0])  # nothing to extend
    assert p.launches() == 0
    rx.decode_plan(p, d, list(range(4)), [300] * 4, [0] * 4, [200])  # 16 rows: mma.sync only
    assert p.launches() == 2
    rx.decode_plan(p, d, list(range(8)), [200] * 8, [0] * 8, [200])  # 32 rows, no own keys
    assert p.launches() == 2
    rx.decode_plan(p, d, list(range(8)), [300] * 8, [0] * 8, [200])  # 32 rows and own keys
    assert p.launches() == 3
    wl = W.radix_mixed(values=False)  # tables and lengths only
    dc = wl.steps[0].decode
    dd = _desc(rows=wl.req_to_token.shape[0], stride=wl.req_to_token.shape[1],
               hq=wl.num_q_heads, hkv=wl.num_kv_heads, pool=wl.pool_size)
    rx.decode_plan(p, dd, dc.req_idx, dc.seq_len, dc.group_of_req, dc.group_prefix_len,
                   dc.group_parent)
    assert p.launches() == 3


def test_tree_plan_argument_checks(librx):
    p = rx.Plan()
    d = _desc()
    with pytest.raises(rx.RxError) as e:   # parent listed after its child
        rx.decode_plan(p, d, [0, 1], [20, 20], [0, 1], [5, 10], [1, -1])
    assert e.value.status == rx.RX_ERR_RANGE
    with pytest.raises(rx.RxError) as e:   # a child's prefix shorter than its parent's
        rx.decode_plan(p, d, [0, 1], [20, 20], [1, 1], [10, 5], [-1, 0])
    assert e.value.status == rx.RX_ERR_RANGE
    with pytest.raises(rx.RxError) as e:
        rx.extend_plan(p, d, [0], [10], [3], [1], [4, 12], [-1, 0])  # prefix 12 > prefix_len 10
    assert e.value.status == rx.RX_ERR_RANGE


def _tree_reads(wl, max_tok):
    """(key, KV head) rows a tree decode plan must read: each node's own keys once per member
    tile of the requests beneath it, each request's keys past its node's prefix once.  A node
    whose stacked query rows (members x gq) reach 32 runs on the tensor-core kernel: tiles of
    128 rows, two tiles per read."""
    dc = wl.steps[0].decode
    par, plen = dc.group_parent, dc.group_prefix_len
    members = np.zeros(len(par), np.int64)
    for g in dc.group_of_req:
        while g >= 0:
            members[g] += 1
            g = par[g]
    rows = 0
    for g in range(len(par)):
        lo = plen[par[g]] if par[g] >= 0 else 0
        if members[g]:
            gq = wl.num_q_heads // wl.num_kv_heads
            per_read = 2 * (128 // gq) if members[g] * gq >= 32 else max_tok
            rows += (plen[g] - lo) * -(-members[g] // per_read)
    rows += int(np.sum(dc.seq_len - plen[dc.group_of_req]))
    return rows * wl.num_kv_heads


def test_tree_decode_plan_reads_each_node_once(librx):
    from prefix_shared_kv_gb300 import workloads as W
    for seed, hq, hkv, n_dec in [(31, 8, 8, 40), (32, 8, 2, 12), (33, 32, 32, 100)]:
        wl = W.tree_workload(seed, hq, hkv, depth=4, fanout=3, seg_lo=1, seg_hi=200, p_empty=0.2,
                             n_decode=n_dec, tail_hi=50, n_extend=0, own_hi=0, ext_lo=1, ext_hi=1)
        dc = wl.steps[0].decode
        desc = rx.KVDesc(hq, hkv, 128, 128 ** -0.5, wl.pool_size, 0x1000, wl.req_to_token.shape[0],
                         wl.req_to_token.shape[1])
        p = rx.Plan()
        rx.decode_plan(p, desc, dc.req_idx, dc.seq_len, dc.group_of_req, dc.group_prefix_len,
                       dc.group_parent)
        max_tok = 64 // (hq // hkv)
        assert p.key_reads() == _tree_reads(wl, max_tok)
        # with every node's requests in one read this is the distinct slots, each read once
        slots = np.concatenate([wl.req_to_token[r, :n] for r, n in zip(dc.req_idx, dc.seq_len)])
        if n_dec <= max_tok or n_dec * (hq // hkv) <= 256:
            assert p.key_reads() == np.unique(slots).size * hkv
        one = rx.Plan()
        rx.decode_plan(one, desc, dc.req_idx, dc.seq_len)
        assert one.key_reads() == int(dc.seq_len.sum()) * hkv


def test_radix_mixed_tree_plans(librx):
    from prefix_shared_kv_gb300 import workloads as W
    wl, wl1 = W.radix_mixed(values=False), W.radix_mixed(tree=False, values=False)
    reads = []
    for w in (wl, wl1):
        dc, e = w.steps[0].decode, w.steps[0].extend
        desc = rx.KVDesc(32, 32, 128, 128 ** -0.5, w.pool_size, 0x1000, w.req_to_token.shape[0],
                         w.req_to_token.shape[1])
        p = rx.Plan()
        rx.decode_plan(p, desc, dc.req_idx, dc.seq_len, dc.group_of_req, dc.group_prefix_len,
                       dc.group_parent)
        pe = rx.Plan()
        rx.extend_plan(pe, desc, e.req_idx, e.prefix_len, e.extend_len, e.group_of_req,
                       e.group_prefix_len, e.group_parent)
        reads.append((p.key_reads(), pe.key_reads()))
    slots = np.concatenate([wl.req_to_token[r, :n] for r, n in zip(wl.steps[0].decode.req_idx,
                                                                 wl.steps[0].decode.seq_len)])
    # the tree plan reads the tree's distinct KV once: 1000 + 8 x 500 + 32 x 200 + tails
    assert reads[0][0] == np.unique(slots).size * 32
    assert reads[1][0] > 2 * reads[0][0]
    # extend: branch-level packing walks fewer keys than packing at the system prompt
    assert reads[0][1] < reads[1][1]


def test_block_granular_match_reuses_whole_pages(librx):
    from prefix_shared_kv_gb300 import workloads as W
    wl = W.paged_workload(77, 8, 2, page=16, prefix=1000, n_req=3, ext_lo=5, ext_hi=9)
    tokens, slots = wl.cached_sequences[0]
    assert len(tokens) == 992                      # 62 whole pages of the 1000-token prefix
    t = rx.Radix()
    t.insert(tokens, slots)
    e = wl.steps[0].extend
    for r in range(3):
        saved, got = t.match(e.tokens[r], match_unit=16)
        assert saved == 992 and np.array_equal(got, slots)
        assert np.all(got.reshape(-1, 16) // 16 == (got.reshape(-1, 16) // 16)[:, :1])  # pages


def _has_gpu():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


@pytest.mark.skipif(_has_gpu(), reason="fake device addresses: run where no GPU could be reached")
def test_attention_and_store_refuse_bad_pointers_before_any_launch(librx):
    """Host-side checks of the calls that launch kernels: each call below carries exactly one
    defect (a NULL or misaligned tensor, a missing, misaligned or short workspace, a plan of the
    other kind, a descriptor the plan was not built with) and must return its code before anything
    is enqueued.  The addresses are fake and never dereferenced."""
    import ctypes as C
    d = _desc(rows=4, stride=64, hq=8, hkv=2)
    p = rx.Plan()
    rx.extend_plan(p, d, [0], [10], [5])
    nb = p.workspace_size()
    good = dict(k=0x10000, v=0x20000, q=0x30000, o=0x40000, lse=0x50000, ws=0x100000, nb=nb)

    def call(fn, desc=d, **bad):
        assert len(bad) == 1  # never a call without a defect: that one would launch
        a = dict(good, **bad)
        return fn(p.handle, C.byref(desc), a["k"], a["v"], a["q"], a["o"], a["lse"], a["ws"],
                  a["nb"], None)

    ext, dec = librx.rx_extend_attn, librx.rx_decode_attn
    assert call(ext, q=0) == rx.RX_ERR_INVALID
    assert call(ext, k=0x10008) == rx.RX_ERR_INVALID
    assert call(ext, o=0x40008) == rx.RX_ERR_INVALID
    assert call(ext, lse=0x50004) == rx.RX_ERR_INVALID
    assert call(ext, ws=0) == rx.RX_ERR_WORKSPACE
    assert call(ext, ws=0x100010) == rx.RX_ERR_INVALID
    assert call(ext, nb=nb - 1) == rx.RX_ERR_WORKSPACE
    assert call(dec, q=0) == rx.RX_ERR_INVALID
    assert call(ext, desc=_desc(rows=4, stride=64, hq=8, hkv=2, pool=256),
                q=0x30000) == rx.RX_ERR_INVALID  # plan built for another pool size
    # the plan is an extend plan: the decode call refuses it whatever the pointers
    assert dec(p.handle, C.byref(d), 0x10000, 0x20000, 0x30000, 0x40000, 0x50000, 0x100000, nb,
               None) == rx.RX_ERR_INVALID
    st = librx.rx_store_kv
    assert st(C.byref(d), 0x10000, 0x20000, 0x60008, 0x70000, 0x80000, 3, None) == rx.RX_ERR_INVALID
    assert st(C.byref(d), 0x10000, 0x20000, 0x60000, 0x70000, None, 3, None) == rx.RX_ERR_INVALID
    assert st(C.byref(d), 0x10000, 0x20000, 0x60000, 0x70000, 0x80000, -1, None) == rx.RX_ERR_INVALID


def test_plan_rows_and_the_bindings_size_checks(librx):
    """rx_plan_rows is the q / o / lse row count a call touches (the sum of extend_len; the
    batch); the binding refuses tensors of another size or dtype before calling in (meta tensors:
    shapes and dtypes only, nothing that could reach a device)."""
    import torch
    for wl in (W.tiny(), W.extend_workload(2, 8, 2, n_groups=2, members=3, prefix=50, ext_lo=0,
                                           ext_hi=20, ungrouped=2, ungrouped_prefix=5),
               W.tree_workload(3, 8, 8, depth=2, fanout=2, seg_lo=0, seg_hi=40, p_empty=0.3,
                               n_decode=9, tail_hi=5, n_extend=4, own_hi=6, ext_lo=1, ext_hi=9)):
        d = _desc(rows=wl.req_to_token.shape[0], stride=wl.req_to_token.shape[1],
                  hq=wl.num_q_heads, hkv=wl.num_kv_heads, pool=wl.pool_size)
        for st in wl.steps:
            for b in (st.extend, st.decode):
                if b is None:
                    continue
                p = rx.Plan()
                if b is st.extend:
                    rx.extend_plan(p, d, b.req_idx, b.prefix_len, b.extend_len, b.group_of_req,
                                   b.group_prefix_len, b.group_parent)
                    n = int(b.extend_len.sum())
                else:
                    rx.decode_plan(p, d, b.req_idx, b.seq_len, b.group_of_req,
                                   b.group_prefix_len, b.group_parent)
                    n = len(b.req_idx)
                assert p.rows() == n
                hq = wl.num_q_heads
                q = torch.empty((n, hq, 128), dtype=torch.bfloat16, device="meta")
                lse = torch.empty((n, hq), dtype=torch.float32, device="meta")
                rx.check_io(p, d, q, q, lse)  # exact: accepted
                with pytest.raises(ValueError):
                    rx.check_io(p, d, q, torch.empty((n + 1, hq, 128), dtype=torch.bfloat16,
                                                     device="meta"), lse)
                with pytest.raises(ValueError):
                    rx.check_io(p, d, q, q, torch.empty((n, hq), dtype=torch.bfloat16,
                                                        device="meta"))
    p = rx.Plan()
    rx.decode_plan(p, _desc(), [], [])
    assert p.rows() == 0
    rx.check_io(p, _desc(), None, None, None)  # an empty batch may pass no tensors


def test_extend_kernel_choice_is_checked():
    p = rx.Plan()
    p.set_extend_kernel(rx.RX_EXTEND_PAIR)
    p.set_extend_kernel(rx.RX_EXTEND_TILES)
    for bad in (-1, 2, 7):
        with pytest.raises(rx.RxError) as e:
            p.set_extend_kernel(bad)
        assert e.value.status == rx.RX_ERR_INVALID
