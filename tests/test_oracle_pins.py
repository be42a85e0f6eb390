"""Pins for the fp64 oracle: it is checked against brute force, closed forms, invariants and the
values the pages print -- never against itself or the CUDA path."""
import json
import math
import os

import numpy as np
import pytest

from oracle import accounting, attention as A, radix
from prefix_shared_kv_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------------------------------------
# Brute force: pure-Python loops over keys with math.exp; independent of the numpy path.
# ---------------------------------------------------------------------------------------------

def _bf(bits):
    return float(A.bf16_to_f64(np.asarray([bits], np.uint16))[0])


def test_bf16_decoding_matches_torch_on_every_bit_pattern():
    """The oracle's bf16 -> float64 decoding (which the brute-force pins below use too) against
    torch's own bfloat16 -> float64 conversion, on all 65,536 bit patterns: zeros of both signs,
    subnormals, infinities and NaNs included."""
    torch = pytest.importorskip("torch")
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ours = A.bf16_to_f64(bits)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    nan = np.isnan(ref)
    assert (np.isnan(ours) == nan).all() and nan.sum() == 2 * 127  # exponent 255, mantissa != 0
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))  # -0.0 stays -0.0
    assert ours[0x3F80] == 1.0 and ours[0xC000] == -2.0 and ours[0x0001] == 2.0 ** -133
    assert ours[0x7F80] == np.inf and ours[0xFF80] == -np.inf


def brute_row(qrow_bits, keys_bits, vals_bits, scale):
    """Attention of one query over a list of key/value rows, written as plain loops."""
    d = len(qrow_bits)
    qv = [_bf(x) for x in qrow_bits]
    scores = []
    for k in keys_bits:
        scores.append(scale * sum(qv[c] * _bf(k[c]) for c in range(d)))
    big = max(scores)
    ws = [math.exp(s - big) for s in scores]
    tot = sum(ws)
    out = [0.0] * d
    for w, v in zip(ws, vals_bits):
        for c in range(d):
            out[c] += w * _bf(v[c])
    return [x / tot for x in out], big + math.log(tot)


def _tiny_extend(seed=7, hq=4, hkv=2):
    return W.extend_workload(seed, hq, hkv, n_groups=2, members=2, prefix=9, ext_lo=1,
                             ext_hi=6, own_cached_hi=4, ungrouped=1, ungrouped_prefix=3,
                             pool_size=256)


def _stored_pools(wl, step=0):
    st = wl.steps[step]
    return A.store_kv(wl.k_pool, wl.v_pool, st.k_new, st.v_new, st.store_slots)


@pytest.mark.parametrize("hq,hkv", [(4, 2), (2, 2), (4, 1)])
def test_extend_matches_brute_force(hq, hkv):
    wl = _tiny_extend(hq=hq, hkv=hkv)
    kp, vp = _stored_pools(wl)
    e = wl.steps[0].extend
    o, lse = A.extend(e.q, kp, vp, wl.req_to_token, e.req_idx, e.prefix_len, e.extend_len,
                      e.cu_q, wl.softmax_scale)
    gq = hq // hkv
    for r in range(len(e.req_idx)):
        p = int(e.prefix_len[r])
        for i in range(int(e.extend_len[r])):
            row = int(e.cu_q[r]) + i
            slots = wl.req_to_token[e.req_idx[r], :p + i + 1]
            for h in range(hq):
                bo, bl = brute_row(e.q[row, h], kp[slots, h // gq], vp[slots, h // gq],
                                   wl.softmax_scale)
                np.testing.assert_allclose(o[row, h], bo, rtol=0, atol=1e-12)
                assert abs(lse[row, h] - bl) < 1e-12


def test_decode_matches_brute_force():
    wl = W.decode_workload(3, 4, 2, n_groups=2, members=3, prefix=11, dist_lo=1, dist_hi=7,
                           ungrouped=2)
    kp, vp = _stored_pools(wl)
    dcd = wl.steps[0].decode
    o, lse = A.decode(dcd.q, kp, vp, wl.req_to_token, dcd.req_idx, dcd.seq_len, wl.softmax_scale)
    for b in range(len(dcd.req_idx)):
        slots = wl.req_to_token[dcd.req_idx[b], :dcd.seq_len[b]]
        for h in range(4):
            bo, bl = brute_row(dcd.q[b, h], kp[slots, h // 2], vp[slots, h // 2], wl.softmax_scale)
            np.testing.assert_allclose(o[b, h], bo, rtol=0, atol=1e-12)
            assert abs(lse[b, h] - bl) < 1e-12


def test_decode_is_an_extend_of_its_current_token():
    """Store-then-attend: a decode step is the extend of one new token (the current one) over a
    cached prefix of seq_len - 1 keys, so the two oracle functions agree on every request."""
    wl = W.decode_workload(5, 8, 2, n_groups=2, members=4, prefix=40, dist_lo=1, dist_hi=30,
                           ungrouped=2)
    kp, vp = _stored_pools(wl)
    d = wl.steps[0].decode
    B = len(d.req_idx)
    o, lse = A.decode(d.q, kp, vp, wl.req_to_token, d.req_idx, d.seq_len, wl.softmax_scale)
    oe, le = A.extend(d.q, kp, vp, wl.req_to_token, d.req_idx, d.seq_len - 1,
                      np.ones(B, np.int32), np.arange(B + 1, dtype=np.int32), wl.softmax_scale)
    np.testing.assert_allclose(oe, o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(le, lse, rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------------------------
# Closed forms of the softmax definition.
# ---------------------------------------------------------------------------------------------

def _rand(rng, *shape):
    return A.bf16_to_f64(W.normal_bf16(rng, shape))


def test_single_visible_key_returns_its_value():
    rng = np.random.default_rng(0)
    q, k, v = _rand(rng, 1, 128), _rand(rng, 1, 128), _rand(rng, 1, 128)
    scale = 1 / math.sqrt(128)
    o, lse = A.attend(q, k, v, np.ones((1, 1), bool), scale)
    np.testing.assert_array_equal(o[0], v[0])
    assert abs(lse[0] - scale * float(np.dot(q[0], k[0]))) < 1e-12


def test_zero_query_gives_mean_value_and_log_length():
    rng = np.random.default_rng(1)
    L = 37
    k, v = _rand(rng, L, 128), _rand(rng, L, 128)
    o, lse = A.attend(np.zeros((1, 128)), k, v, np.ones((1, L), bool), 0.3)
    np.testing.assert_allclose(o[0], v.mean(axis=0), atol=1e-13)
    assert abs(lse[0] - math.log(L)) < 1e-13


def test_identical_keys_give_mean_value_and_shifted_lse():
    rng = np.random.default_rng(2)
    L = 19
    q = _rand(rng, 1, 128)
    k = np.repeat(_rand(rng, 1, 128), L, axis=0)
    v = _rand(rng, L, 128)
    scale = 1 / math.sqrt(128)
    o, lse = A.attend(q, k, v, np.ones((1, L), bool), scale)
    np.testing.assert_allclose(o[0], v.mean(axis=0), atol=1e-13)
    assert abs(lse[0] - (scale * float(q[0] @ k[0]) + math.log(L))) < 1e-12


def test_unit_values_give_unit_output_and_rows_sum_to_one():
    rng = np.random.default_rng(3)
    L = 50
    q, k = _rand(rng, 5, 128) * 4, _rand(rng, L, 128)
    vis = np.tril(np.ones((5, L), bool), k=L - 5)
    o, _ = A.attend(q, k, np.ones((L, 128)), vis, 1 / math.sqrt(128))
    np.testing.assert_allclose(o, 1.0, atol=1e-14)


def test_masked_keys_do_not_contribute():
    rng = np.random.default_rng(4)
    L = 30
    q, k, v = _rand(rng, 1, 128), _rand(rng, L, 128), _rand(rng, L, 128)
    vis = np.zeros((1, L), bool)
    vis[0, :12] = True
    o1, l1 = A.attend(q, k, v, vis, 0.1)
    v2 = v.copy()
    v2[12:] = 1e6
    k2 = k.copy()
    k2[12:] = -k2[12:] * 50
    o2, l2 = A.attend(q, k2, v2, vis, 0.1)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)
    o3, l3 = A.attend(q, k[:12], v[:12], np.ones((1, 12), bool), 0.1)
    np.testing.assert_allclose(o1, o3, atol=1e-14)
    np.testing.assert_allclose(l1, l3, atol=1e-14)


# ---------------------------------------------------------------------------------------------
# Invariants the method rests on.
# ---------------------------------------------------------------------------------------------

def test_prefix_caching_equals_full_recompute():
    """Cached-prefix extend == the last rows of a from-scratch prefill over the same slots."""
    rng = np.random.default_rng(5)
    hq, hkv, P = 4, 2, 512
    b = W.Builder(rng, hq, hkv, P)
    pre = b.cached(70)
    new = b.new(23)
    row = b.row([pre, new])
    wl = b.finish("inv", [([new], ([row], [70], [23], [-1], [], []), None)], [], "")
    kp, vp = _stored_pools(wl)
    full_q = W.normal_bf16(rng, (93, hq, 128))
    r2t = wl.req_to_token
    ridx = wl.steps[0].extend.req_idx
    o_full, l_full = A.extend(full_q, kp, vp, r2t, ridx, np.array([0]), np.array([93]),
                              np.array([0, 93]), wl.softmax_scale)
    o_c, l_c = A.extend(full_q[70:], kp, vp, r2t, ridx, np.array([70]), np.array([23]),
                        np.array([0, 23]), wl.softmax_scale)
    np.testing.assert_allclose(o_c, o_full[70:], atol=1e-12)
    np.testing.assert_allclose(l_c, l_full[70:], atol=1e-12)
    # and a decode of the last row is the same as the last extend row
    o_d, l_d = A.decode(full_q[92:93], kp, vp, r2t, ridx, np.array([93]), wl.softmax_scale)
    np.testing.assert_allclose(o_d[0], o_full[92], atol=1e-12)
    np.testing.assert_allclose(l_d[0], l_full[92], atol=1e-12)


def test_merge_of_partitions_equals_softmax_over_union():
    rng = np.random.default_rng(6)
    L, n = 300, 7
    q, k, v = _rand(rng, n, 128) * 3, _rand(rng, L, 128), _rand(rng, L, 128)
    scale = 1 / math.sqrt(128)
    full = A.attend(q, k, v, np.ones((n, L), bool), scale)
    for nparts in (2, 3, 5):
        label = rng.integers(0, nparts, size=L)
        parts = [A.attend(q, k, v, np.broadcast_to(label == j, (n, L)), scale)
                 for j in range(nparts)]
        o, lse = A.merge(parts)
        np.testing.assert_allclose(o, full[0], atol=1e-12)
        np.testing.assert_allclose(lse, full[1], atol=1e-12)
        # associativity
        left = A.merge([A.merge(parts[:1] + parts[1:2]), *parts[2:]]) if nparts > 2 else (o, lse)
        np.testing.assert_allclose(left[0], o, atol=1e-12)
    # an empty partition is the identity
    empty = A.attend(q, k, v, np.zeros((n, L), bool), scale)
    assert np.all(np.isneginf(empty[1])) and np.all(empty[0] == 0)
    o, lse = A.merge([full, empty])
    np.testing.assert_allclose(o, full[0], atol=1e-15)
    np.testing.assert_allclose(lse, full[1], atol=1e-15)


def test_merge_prefix_and_distinct_partition_of_a_request():
    """The horizontal-fusion split: shared prefix keys and the request's own keys."""
    wl = W.decode_workload(11, 4, 4, n_groups=1, members=3, prefix=40, dist_lo=5, dist_hi=30)
    kp, vp = _stored_pools(wl)
    dcd = wl.steps[0].decode
    o, lse = A.decode(dcd.q, kp, vp, wl.req_to_token, dcd.req_idx, dcd.seq_len, wl.softmax_scale)
    gp = int(dcd.group_prefix_len[0])
    for b in range(3):
        L = int(dcd.seq_len[b])
        slots = wl.req_to_token[dcd.req_idx[b], :L]
        for h in range(4):
            q = A.bf16_to_f64(dcd.q[b, h])[None]
            K = A.bf16_to_f64(kp[slots, h])
            V = A.bf16_to_f64(vp[slots, h])
            pre = A.attend(q, K[:gp], V[:gp], np.ones((1, gp), bool), wl.softmax_scale)
            own = A.attend(q, K[gp:], V[gp:], np.ones((1, L - gp), bool), wl.softmax_scale)
            mo, ml = A.merge([pre, own])
            np.testing.assert_allclose(mo[0], o[b, h], atol=1e-12)
            assert abs(ml[0] - lse[b, h]) < 1e-12


# ---------------------------------------------------------------------------------------------
# Pool scatter.
# ---------------------------------------------------------------------------------------------

def test_store_kv_scatter_is_bit_exact_and_touches_only_its_slots():
    rng = np.random.default_rng(8)
    P, T = 200, 37
    sentinel = np.uint16(0x7FC1)
    kp = np.full((P, 2, 128), sentinel, np.uint16)
    vp = np.full((P, 2, 128), sentinel, np.uint16)
    slots = rng.permutation(P)[:T].astype(np.int32)
    kn = W.normal_bf16(rng, (T, 2, 128))
    vn = W.normal_bf16(rng, (T, 2, 128))
    k2, v2 = A.store_kv(kp, vp, kn, vn, slots)
    np.testing.assert_array_equal(k2[slots], kn)
    np.testing.assert_array_equal(v2[slots], vn)
    untouched = np.setdiff1d(np.arange(P), slots)
    assert np.all(k2[untouched] == sentinel) and np.all(v2[untouched] == sentinel)
    assert np.all(kp == sentinel)  # inputs not modified


# ---------------------------------------------------------------------------------------------
# Prefix match and token accounting: the pages' printed numbers.
# ---------------------------------------------------------------------------------------------

def test_worked_example_of_the_prefix_caching_page():
    g = json.load(open(os.path.join(GOLDEN, "prefix_cache_worked_example.json")))
    rng = np.random.default_rng(9)
    n, nq = g["common_prefix_tokens"], g["question_tokens"]
    common = list(rng.integers(0, 16000, n))

    def fresh(k):
        return list(rng.integers(16000, 32000, k))

    slot_iter = iter(range(10 ** 6))

    def store_of(seqs):
        s = radix.PrefixStore()
        for t in seqs:
            s.insert(t, [next(slot_iter) for _ in t])
        return s

    ts1, ts2 = fresh(3), fresh(3)
    situations = [
        (store_of([common + fresh(nq)]), common + fresh(nq)),
        (store_of([ts1 + common + fresh(nq)]), ts2 + common + fresh(nq)),
        (store_of([common + ts1 + fresh(nq)]), common + ts2 + fresh(nq)),
        # a long answer only adds decode tokens; what the next prompt reuses is unchanged
        (store_of([common + fresh(nq)]), common + fresh(nq)),
    ]
    for case, (store, prompt) in zip(g["cases"], situations):
        for unit, saved in case["saved"].items():
            assert store.match(prompt, int(unit))[0] == saved, case["situation"]
    # loss at unit 16 is at most 15 tokens, 1.5 % of a 1000-token prefix
    worst = max(m - (m // 16) * 16 for m in range(0, 5000))
    assert worst == g["max_loss_tokens_unit16"]
    assert worst / n == pytest.approx(g["max_loss_fraction_of_1000"])


def test_tiny_workload_prefix_saves_1000_and_992():
    wl = W.tiny()
    store = radix.PrefixStore()
    for toks, slots in wl.cached_sequences:
        store.insert(toks, slots)
    for toks in wl.steps[0].extend.tokens:
        saved1, slots1 = store.match(toks, 1)
        assert saved1 == 1000 and store.match(toks, 16)[0] == 992
        # the matched slots are the ones the request's table row starts with
    r2t = wl.req_to_token
    for r, toks in zip(wl.steps[0].extend.req_idx, wl.steps[0].extend.tokens):
        np.testing.assert_array_equal(store.match(toks, 1)[1], r2t[r, :1000])


def test_prefix_store_equals_brute_force_longest_common_prefix():
    rng = np.random.default_rng(10)
    for _ in range(200):
        seqs = [list(rng.integers(0, 3, rng.integers(0, 9))) for _ in range(rng.integers(1, 6))]
        s = radix.PrefixStore()
        for t in seqs:
            s.insert(t, list(range(len(t))))
        q = list(rng.integers(0, 3, rng.integers(0, 10)))
        best = 0
        for t in seqs:
            c = 0
            while c < min(len(t), len(q)) and t[c] == q[c]:
                c += 1
            best = max(best, c)
        assert s.longest(q) == best
        for u in (1, 2, 4):
            assert s.match(q, u)[0] == best // u * u


def test_first_stored_sequence_keeps_its_slots():
    s = radix.PrefixStore()
    s.insert([5, 6, 7], [10, 11, 12])
    s.insert([5, 6, 9], [20, 21, 22])
    assert s.match([5, 6, 9, 1])[1] == [10, 11, 22]


def test_compute_reduction_example():
    g = json.load(open(os.path.join(GOLDEN, "closed_forms.json")))["compute_reduction"]
    r = accounting.compute_reduction(g["l_prefix"], g["l_new"])
    assert round(100 * r) == g["printed_percent_approx"]
    # and it is the fraction of attended (query, key) prefill rows a hit skips: brute count
    assert r == pytest.approx(2000 / 2100)


def test_batchllm_token_saving_printed_values():
    g = json.load(open(os.path.join(GOLDEN, "closed_forms.json")))["token_saving_ratio"]
    for c in g["cases"]:
        logical = c["sharing"] * (c["prefix"] + c["distinct_inferred"])
        processed = c["prefix"] + c["sharing"] * c["distinct_inferred"]
        # processed tokens counted by brute force with a prefix store
        s = radix.PrefixStore()
        rng = np.random.default_rng(c["prefix"])
        pre = list(rng.integers(0, 16000, c["prefix"]))
        done = 0
        for _ in range(c["sharing"]):
            t = pre + list(rng.integers(16000, 32000, c["distinct_inferred"]))
            done += len(t) - s.match(t)[0]
            s.insert(t, list(range(len(t))))
        assert done == processed
        assert round(accounting.token_saving_ratio(processed, logical), 1) == c["printed_percent"]


def test_optimal_hit_rate_of_the_radix_mixed_tree_by_simulation():
    """1 - C / sum(prefill) equals the hit rate of running the tree's leaves in DFS order."""
    wl = W.radix_mixed(values=False)  # token sequences only
    leaves = wl.cached_sequences[:32]
    s = radix.PrefixStore()
    cached = total = 0
    for toks, slots in leaves:          # leaves are generated in DFS order
        cached += s.match(toks)[0]
        total += len(toks)
        s.insert(toks, slots)
    C = 1000 + 8 * 500 + 32 * 200
    assert total - cached == C
    assert accounting.hit_rate(cached, total) == pytest.approx(
        accounting.optimal_hit_rate(C, total), abs=1e-15)
    assert accounting.optimal_hit_rate(C, total) == pytest.approx(1 - 11400 / 54400)


def test_merge_gain_counts_tokens_saved_by_sharing_a_node():
    for leaves, tokens in [(1, 50), (4, 500), (16, 2000)]:
        s = radix.PrefixStore()
        node = list(range(tokens))
        processed = 0
        for j in range(leaves):
            t = node + [100000 + j]
            processed += len(t) - s.match(t)[0]
            s.insert(t, list(range(len(t))))
        unshared = leaves * (tokens + 1)
        assert unshared - processed == accounting.merge_gain(leaves, tokens)


def test_chunked_prefill_equals_one_prefill_of_the_whole_prompt():
    """Chunked prefill (each chunk an extend over the system prompt and the chunks before it,
    stored step by step) gives, row for row, what one extend of the whole prompt gives."""
    wl = W.chunked_prefill_workload(7, 4, 2, system=96, prompt=300, chunk=128, n_decode=2,
                                    tail_lo=5, tail_hi=20)
    kp, vp = wl.k_pool, wl.v_pool
    rows_o, rows_l, qs = [], [], []
    for st in wl.steps:
        kp, vp = A.store_kv(kp, vp, st.k_new, st.v_new, st.store_slots)
        e = st.extend
        o, l = A.extend(e.q, kp, vp, wl.req_to_token, e.req_idx, e.prefix_len, e.extend_len,
                        e.cu_q, wl.softmax_scale)
        rows_o.append(o)
        rows_l.append(l)
        qs.append(e.q)
    assert [int(s.extend.prefix_len[0]) for s in wl.steps] == [96, 224, 352]
    q = np.concatenate(qs)
    ridx = wl.steps[0].extend.req_idx
    o_full, l_full = A.extend(q, kp, vp, wl.req_to_token, ridx, np.array([96]), np.array([300]),
                              np.array([0, 300]), wl.softmax_scale)
    np.testing.assert_allclose(np.concatenate(rows_o), o_full, atol=1e-12)
    np.testing.assert_allclose(np.concatenate(rows_l), l_full, atol=1e-12)
