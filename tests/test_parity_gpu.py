"""Parity of the CUDA path (called through the C ABI) with the fp64 oracle.

Tolerances (bf16 in, fp32 accumulate, bf16 out): O max-abs <= 2e-2 and mean-abs <= 2e-3, LSE
within 1e-3; the pool scatter is bit-exact.  Small cases are compared element by element over every
row; the full-size workloads, run in the benchmark's launch configuration, are compared on every
row, except the two decode workloads, compared on a stratified set of requests.
"""
import numpy as np
import pytest
import torch

from oracle import attention as A
from prefix_shared_kv_gb300 import rx, workloads as W
from prefix_shared_kv_gb300.session import DeviceWorkload, bits_of, to_bf16, to_i32

pytestmark = pytest.mark.gpu

MAX_ABS, MEAN_ABS, LSE_ABS = 2e-2, 2e-3, 1e-3


def assert_close(o_gpu, lse_gpu, o_ref, lse_ref, rows=None, what=""):
    o = A.bf16_to_f64(bits_of(o_gpu))
    l = lse_gpu.double().cpu().numpy()
    if rows is not None:
        o, l, o_ref, lse_ref = o[rows], l[rows], o_ref[rows], lse_ref[rows]
    assert o.shape == o_ref.shape and l.shape == lse_ref.shape, what
    if o_ref.size == 0:  # an empty batch: nothing to compare
        return
    assert np.isfinite(o_ref).all()
    err = np.abs(o - o_ref)
    lerr = np.abs(l - lse_ref)
    assert err.max() <= MAX_ABS, f"{what}: O max-abs {err.max():.3e}"
    assert err.mean() <= MEAN_ABS, f"{what}: O mean-abs {err.mean():.3e}"
    assert lerr.max() <= LSE_ABS, f"{what}: LSE max-abs {lerr.max():.3e}"


def oracle_pools(wl, upto_step):
    kp, vp = wl.k_pool, wl.v_pool
    for s in range(upto_step + 1):
        st = wl.steps[s]
        kp, vp = A.store_kv(kp, vp, st.k_new, st.v_new, st.store_slots)
    return kp, vp


def stratified_decode_requests(d):
    """Decode requests that cover a batch's structure: in every group the members with the
    shortest and the longest own part, one request at every decile of the own lengths over the
    batch, and every request outside a group (a cache miss)."""
    grp = np.asarray(d.group_of_req)
    gpl = np.asarray(d.group_prefix_len)
    own = np.asarray(d.seq_len) - np.where(grp >= 0, gpl[np.maximum(grp, 0)], 0)
    pick = set(np.flatnonzero(grp < 0).tolist())
    for g in np.unique(grp[grp >= 0]):
        m = np.flatnonzero(grp == g)
        pick.add(int(m[np.argmin(own[m])]))
        pick.add(int(m[np.argmax(own[m])]))
    order = np.argsort(own, kind="stable")
    for q in range(11):
        pick.add(int(order[min(len(order) - 1, q * (len(order) - 1) // 10)]))
    return sorted(pick)


def run_and_check(wl, cuda, sample=None, seed=0, decode_pick=None,
                  extend_kernel=rx.RX_EXTEND_TILES):
    """Run every step of `wl` on the GPU and compare with the oracle: every row, or the rows of
    `sample` random requests per batch, or (decode only) the requests decode_pick(batch) names.
    Extend plans run on `extend_kernel`."""
    dw = DeviceWorkload(wl, cuda, extend_kernel=extend_kernel)
    rng = np.random.default_rng(seed)
    for i, st in enumerate(wl.steps):
        dw.run_step(i)
        torch.cuda.synchronize()
        kp, vp = oracle_pools(wl, i)
        if st.extend is not None:
            e = st.extend
            reqs = None
            rows = None
            if sample is not None and len(e.req_idx) > sample:
                reqs = sorted(rng.choice(len(e.req_idx), sample, replace=False))
                rows = np.concatenate([np.arange(e.cu_q[r], e.cu_q[r + 1]) for r in reqs])
            o, l = A.extend(e.q, kp, vp, wl.req_to_token, e.req_idx, e.prefix_len, e.extend_len,
                            e.cu_q, wl.softmax_scale, requests=reqs)
            if rows is None:
                rows = np.arange(e.q.shape[0])
            assert_close(dw.steps[i].ext_o, dw.steps[i].ext_lse, o, l, rows, f"{wl.name} extend")
        if st.decode is not None:
            d = st.decode
            reqs = None
            if decode_pick is not None:
                reqs = decode_pick(d)
            elif sample is not None and len(d.req_idx) > sample:
                reqs = sorted(rng.choice(len(d.req_idx), sample, replace=False))
            o, l = A.decode(d.q, kp, vp, wl.req_to_token, d.req_idx, d.seq_len, wl.softmax_scale,
                            requests=reqs)
            rows = np.arange(len(d.req_idx)) if reqs is None else np.asarray(reqs)
            assert_close(dw.steps[i].dec_o, dw.steps[i].dec_lse, o, l, rows, f"{wl.name} decode")
    return dw


# ---------------------------------------------------------------------------------------------
# rx_store_kv
# ---------------------------------------------------------------------------------------------

@pytest.mark.parametrize("hkv,T", [(2, 1), (8, 37), (32, 1000), (1, 0)])
def test_store_kv_bit_exact(cuda, hkv, T):
    rng = np.random.default_rng(T)
    P = 3000
    sentinel = np.uint16(0x7FC1)
    kp = np.full((P, hkv, 128), sentinel, np.uint16)
    vp = kp.copy()
    slots = rng.permutation(P)[:T].astype(np.int32)
    kn, vn = W.normal_bf16(rng, (T, hkv, 128)), W.normal_bf16(rng, (T, hkv, 128))
    dk, dv = to_bf16(kp, cuda), to_bf16(vp, cuda)
    r2t = to_i32(np.zeros((1, 16), np.int32), cuda)
    desc = rx.kv_desc(hkv, hkv, P, r2t)
    rx.store_kv(desc, dk, dv, to_bf16(kn, cuda), to_bf16(vn, cuda), to_i32(slots, cuda))
    torch.cuda.synchronize()
    ek, ev = A.store_kv(kp, vp, kn, vn, slots)
    np.testing.assert_array_equal(bits_of(dk), ek)
    np.testing.assert_array_equal(bits_of(dv), ev)


def test_store_kv_skips_out_of_range_slots(cuda):
    rng = np.random.default_rng(5)
    P, T = 100, 6
    kp = np.zeros((P, 2, 128), np.uint16)
    slots = np.array([3, -1, 50, 100, 99, 2 ** 30], np.int32)
    kn, vn = W.normal_bf16(rng, (T, 2, 128)), W.normal_bf16(rng, (T, 2, 128))
    dk, dv = to_bf16(kp, cuda), to_bf16(kp, cuda)
    desc = rx.kv_desc(2, 2, P, to_i32(np.zeros((1, 16), np.int32), cuda))
    rx.store_kv(desc, dk, dv, to_bf16(kn, cuda), to_bf16(vn, cuda), to_i32(slots, cuda))
    torch.cuda.synchronize()
    ok = [0, 2, 4]
    ek, _ = A.store_kv(kp, kp, kn[ok], vn[ok], slots[ok])
    np.testing.assert_array_equal(bits_of(dk), ek)


# ---------------------------------------------------------------------------------------------
# The tiny workload: 4 x 40 extend on a shared 1000-token prefix, then 8 decode steps.
# ---------------------------------------------------------------------------------------------

def test_tiny_workload_all_steps(cuda):
    run_and_check(W.tiny(), cuda)


# ---------------------------------------------------------------------------------------------
# Extend: head ratios, ragged tails, own cached parts, ungrouped requests, several tiles.
# ---------------------------------------------------------------------------------------------

@pytest.mark.parametrize("hq,hkv", [(4, 4), (8, 2), (16, 2), (8, 4)])
def test_extend_shapes(cuda, hq, hkv):
    wl = W.extend_workload(100 + hq + hkv, hq, hkv, n_groups=2, members=5, prefix=333,
                           ext_lo=1, ext_hi=150, own_cached_hi=70, ungrouped=2,
                           ungrouped_prefix=129)
    run_and_check(wl, cuda)


def test_extend_long_causal_and_empty(cuda):
    # prefix 0 full prefill longer than several tiles, and requests with nothing to extend
    wl = W.extend_workload(7, 8, 8, n_groups=1, members=3, prefix=65, ext_lo=0, ext_hi=3,
                           ungrouped=2, ungrouped_prefix=0)
    run_and_check(wl, cuda)
    wl = W.extend_workload(8, 8, 8, n_groups=0, members=0, prefix=0, ext_lo=300, ext_hi=700,
                           ungrouped=2, ungrouped_prefix=0)
    run_and_check(wl, cuda)


def test_extend_very_long_prefix(cuda):
    """Items of ~500 steps: a 32,000-token shared prefix (three members, GQA 4) and an ungrouped
    request on its own 20,000-token prefix."""
    wl = W.extend_workload(10, 8, 2, n_groups=1, members=3, prefix=32000, ext_lo=1, ext_hi=40,
                           ungrouped=1, ungrouped_prefix=20000)
    run_and_check(wl, cuda)


def test_empty_batches(cuda):
    """No requests at all: plans with no items, calls that launch nothing and return OK."""
    run_and_check(W.extend_workload(3, 4, 2, n_groups=0, members=3, prefix=100, ext_lo=1,
                                    ext_hi=30, ungrouped=0), cuda)
    run_and_check(W.decode_workload(3, 4, 2, n_groups=0, members=3, prefix=100, dist_lo=1,
                                    dist_hi=30, ungrouped=0), cuda)


def test_extend_peaky_softmax(cuda):
    wl = W.extend_workload(9, 8, 2, n_groups=1, members=4, prefix=200, ext_lo=30, ext_hi=90)
    for st in wl.steps:
        q = A.bf16_to_f64(st.extend.q) * 4.0
        st.extend.q = W.bf16_bits(q.astype(np.float32))
    run_and_check(wl, cuda)


def _unit_values(wl):
    one = np.uint16(0x3F80)  # bf16 1.0
    wl.v_pool = np.full_like(wl.v_pool, one)
    for st in wl.steps:
        st.v_new = np.full_like(st.v_new, one)
    return wl


def _within_one_ulp_of_one(o, what):
    # bf16 neighbours of 1.0: 1 - 2^-8 below, 1 + 2^-7 above
    v = A.bf16_to_f64(bits_of(o))
    assert v.size > 0 and ((v >= 1 - 2 ** -8) & (v <= 1 + 2 ** -7)).all(), \
        f"{what}: O in [{v.min()}, {v.max()}]"


@pytest.mark.parametrize("kind", ["extend", "decode", "tree"])
def test_unit_values_give_unit_output(cuda, kind):
    """With every V row equal to 1 the attention weights of a row sum to one, so each output is
    1.0 to one bf16 unit: this pins the kernels' own normalisation (P rounded to bf16 for the PV
    product against the fp32 row sum; partial rows merged by LSE), whatever the scores are."""
    if kind == "extend":
        wl = W.extend_workload(31, 16, 4, n_groups=2, members=6, prefix=900, ext_lo=1,
                               ext_hi=160, own_cached_hi=40, ungrouped=2, ungrouped_prefix=300)
    elif kind == "decode":
        # 24 members x gq 4 stack 96 rows: the shared prefix goes through the tensor-core units
        wl = W.decode_workload(32, 16, 4, n_groups=2, members=24, prefix=3000, dist_lo=1,
                               dist_hi=400, ungrouped=3)
    else:
        wl = W.tree_workload(33, 8, 8, depth=3, fanout=3, seg_lo=0, seg_hi=300, p_empty=0.2,
                             n_decode=30, tail_hi=60, n_extend=6, own_hi=40, ext_lo=1,
                             ext_hi=120)
    dw = run_and_check(_unit_values(wl), cuda)
    for i, st in enumerate(wl.steps):
        if st.extend is not None:
            _within_one_ulp_of_one(dw.steps[i].ext_o, f"{kind} extend")
        if st.decode is not None:
            _within_one_ulp_of_one(dw.steps[i].dec_o, f"{kind} decode")


def test_decode_calls_with_their_own_plans_on_two_streams(cuda):
    """Two callers, each with a plan of its own whose decode runs both partial kernels (a second
    stream per plan), issue their calls on two streams without waiting for each other, several
    times over; every result matches the oracle."""
    def make(seed):
        return W.tree_workload(seed, 8, 8, depth=2, fanout=3, seg_lo=50, seg_hi=300, p_empty=0.0,
                               n_decode=40, tail_hi=40, n_extend=1, own_hi=30, ext_lo=1,
                               ext_hi=10)
    wls = [make(41), make(43)]
    streams = [torch.cuda.Stream(cuda), torch.cuda.Stream(cuda)]
    dws = [DeviceWorkload(wl, cuda, stream=st) for wl, st in zip(wls, streams)]
    for dw in dws:
        assert dw.steps[0].dec_plan.launches() == 3
        with torch.cuda.stream(dw.stream):
            dw.store(0)
    torch.cuda.synchronize()
    for _ in range(4):
        for dw in dws:
            with torch.cuda.stream(dw.stream):
                dw.decode(0)
    torch.cuda.synchronize()
    for wl, dw in zip(wls, dws):
        st = wl.steps[0]
        kp, vp = A.store_kv(wl.k_pool, wl.v_pool, st.k_new, st.v_new, st.store_slots)
        d = st.decode
        o, l = A.decode(d.q, kp, vp, wl.req_to_token, d.req_idx, d.seq_len, wl.softmax_scale)
        assert_close(dw.steps[0].dec_o, dw.steps[0].dec_lse, o, l, what=wl.name)


def test_cuda_graph_replay_of_a_step(cuda):
    """A whole step -- store, extend, and a decode whose tensor-core and mma.sync units run on
    two streams (fork and join through events) before the merge -- captured once into a CUDA
    graph after a first eager run, then replayed: the results match the oracle, and a second
    replay gives the same bits as the first."""
    wl = W.tree_workload(41, 8, 8, depth=2, fanout=3, seg_lo=50, seg_hi=300, p_empty=0.0,
                         n_decode=40, tail_hi=40, n_extend=6, own_hi=30, ext_lo=1, ext_hi=100)
    dw = DeviceWorkload(wl, cuda)
    ds = dw.steps[0]
    assert ds.dec_plan.launches() == 3 and ds.ext_plan.launches() == 1
    dw.run_step(0)  # the first calls set kernel attributes and create the second stream
    torch.cuda.synchronize()
    eager = [t.clone() for t in (ds.ext_o, ds.ext_lse, ds.dec_o, ds.dec_lse)]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        dw.run_step(0)
    outs = (ds.ext_o, ds.ext_lse, ds.dec_o, ds.dec_lse)
    replays = []
    for _ in range(2):
        for t in outs:
            t.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        replays.append([t.clone() for t in outs])
    kp, vp = oracle_pools(wl, 0)
    st = wl.steps[0]
    e, d = st.extend, st.decode
    o, l = A.extend(e.q, kp, vp, wl.req_to_token, e.req_idx, e.prefix_len, e.extend_len, e.cu_q,
                    wl.softmax_scale)
    assert_close(replays[0][0], replays[0][1], o, l, what="graph extend")
    o, l = A.decode(d.q, kp, vp, wl.req_to_token, d.req_idx, d.seq_len, wl.softmax_scale)
    assert_close(replays[0][2], replays[0][3], o, l, what="graph decode")
    for a, b, c in zip(replays[0], replays[1], eager):
        assert torch.equal(a, b) and torch.equal(a, c)


def test_kernels_write_nothing_outside_their_outputs(cuda):
    """o and lse of both calls sit in buffers with 4,096 guard elements on each side, filled
    with a pattern: after a step (extend; decode with tensor-core units, mma.sync units and the
    merge) the guards are unchanged, and the outputs equal those of a run in plain buffers."""
    def make():
        return W.tree_workload(41, 8, 8, depth=2, fanout=3, seg_lo=50, seg_hi=300, p_empty=0.0,
                               n_decode=40, tail_hi=40, n_extend=6, own_hi=30, ext_lo=1,
                               ext_hi=100)
    plain = DeviceWorkload(make(), cuda)
    plain.run_step(0)
    dw = DeviceWorkload(make(), cuda)
    ds = dw.steps[0]
    assert ds.dec_plan.launches() == 3
    G = 4096
    guards = []

    def guarded(t):
        as_int = torch.int16 if t.element_size() == 2 else torch.int32
        pattern = 0x7FC1 if t.element_size() == 2 else 0x7F8A5A5A
        buf = torch.empty(t.numel() + 2 * G, dtype=t.dtype, device=cuda)
        buf.view(as_int).fill_(pattern)
        guards.append((buf.view(as_int), pattern))
        return buf[G:G + t.numel()].view(t.shape)

    ds.ext_o, ds.ext_lse = guarded(ds.ext_o), guarded(ds.ext_lse)
    ds.dec_o, ds.dec_lse = guarded(ds.dec_o), guarded(ds.dec_lse)
    dw.run_step(0)
    torch.cuda.synchronize()
    for b, pattern in guards:
        assert bool((b[:G] == pattern).all()) and bool((b[-G:] == pattern).all())
    p = plain.steps[0]
    for a, b in ((ds.ext_o, p.ext_o), (ds.ext_lse, p.ext_lse), (ds.dec_o, p.dec_o),
                 (ds.dec_lse, p.dec_lse)):
        assert torch.equal(a, b)


# ---------------------------------------------------------------------------------------------
# Decode: groups of many members, single-member groups, empty own parts, long prefixes.
# ---------------------------------------------------------------------------------------------

@pytest.mark.parametrize("hq,hkv", [(8, 8), (8, 2), (32, 4), (16, 8)])
def test_decode_shapes(cuda, hq, hkv):
    wl = W.decode_workload(200 + hq + hkv, hq, hkv, n_groups=3, members=21, prefix=777,
                           dist_lo=1, dist_hi=300, ungrouped=3)
    run_and_check(wl, cuda)


def test_decode_long_prefix_many_chunks(cuda):
    wl = W.decode_workload(11, 8, 8, n_groups=2, members=2, prefix=9000, dist_lo=1, dist_hi=3000)
    run_and_check(wl, cuda)
    wl = W.decode_workload(12, 32, 8, n_groups=1, members=1, prefix=5000, dist_lo=1, dist_hi=1)
    run_and_check(wl, cuda)


def test_decode_more_than_32_partials_per_request(cuda):
    """An 80,000-token GQA prefix read in ~2,048-key chunks: ~40 partial rows per request, more
    than one 32-partial chunk of the merge."""
    wl = W.decode_workload(14, 32, 8, n_groups=1, members=8, prefix=80000, dist_lo=1, dist_hi=50)
    run_and_check(wl, cuda, sample=3, seed=2)


def test_decode_group_prefix_zero_and_ungrouped_only(cuda):
    wl = W.decode_workload(13, 8, 4, n_groups=2, members=3, prefix=0, dist_lo=1, dist_hi=90,
                           ungrouped=5)
    run_and_check(wl, cuda)


def test_decode_grouping_does_not_change_the_result(cuda):
    wl = W.decode_workload(14, 16, 4, n_groups=2, members=9, prefix=400, dist_lo=20, dist_hi=200)
    dw = DeviceWorkload(wl, cuda)
    dw.run_step(0)
    d = wl.steps[0].decode
    plan = rx.Plan()
    rx.decode_plan(plan, dw.desc, d.req_idx, d.seq_len)          # no groups declared
    ws = torch.empty(plan.workspace_size(), dtype=torch.uint8, device=cuda)
    plan.upload(ws)
    o2 = torch.empty_like(dw.steps[0].dec_o)
    l2 = torch.empty_like(dw.steps[0].dec_lse)
    rx.decode_attn(plan, dw.desc, dw.k_pool, dw.v_pool, dw.steps[0].dec_q, o2, l2, ws)
    torch.cuda.synchronize()
    a = A.bf16_to_f64(bits_of(o2))
    b = A.bf16_to_f64(bits_of(dw.steps[0].dec_o))
    assert np.abs(a - b).max() <= MAX_ABS
    assert (l2 - dw.steps[0].dec_lse).abs().max().item() <= LSE_ABS


def test_extend_output_only_16_byte_aligned(cuda):
    """o at a 16-byte (not 32-byte) boundary: the kernel writes rows in 16-byte pieces there."""
    wl = W.extend_workload(15, 8, 2, n_groups=2, members=3, prefix=300, ext_lo=20, ext_hi=150)
    dw = DeviceWorkload(wl, cuda)
    dw.run_step(0)
    torch.cuda.synchronize()
    st = dw.steps[0]
    ref_o = st.ext_o.clone()
    ref_l = st.ext_lse.clone()
    n = ref_o.numel()
    buf = torch.empty(n + 64, dtype=torch.bfloat16, device=cuda)
    o16 = buf[8:8 + n].view_as(ref_o)  # 16 bytes past a 256-byte aligned base
    assert o16.data_ptr() % 32 == 16
    l2 = torch.empty_like(ref_l)
    rx.extend_attn(st.ext_plan, dw.desc, dw.k_pool, dw.v_pool, st.ext_q, o16, l2, st.ext_ws)
    torch.cuda.synchronize()
    assert torch.equal(o16, ref_o)
    assert torch.equal(l2, ref_l)
    e = wl.steps[0].extend
    kp, vp = oracle_pools(wl, 0)
    o, l = A.extend(e.q, kp, vp, wl.req_to_token, e.req_idx, e.prefix_len, e.extend_len, e.cu_q,
                    wl.softmax_scale)
    assert_close(o16, l2, o, l, None, "extend, o 16-byte aligned")


def test_plan_rebuilt_and_uploaded_again_while_the_first_copy_may_be_in_flight(cuda):
    """rx_plan_upload stages the tables in a pinned buffer the plan owns: rebuilding the plan and
    uploading it again on another stream must leave each workspace with its own tables."""
    wl = W.decode_workload(16, 16, 4, n_groups=2, members=6, prefix=300, dist_lo=20, dist_hi=120)
    dw = DeviceWorkload(wl, cuda)
    dw.run_step(0)
    torch.cuda.synchronize()
    d = wl.steps[0].decode
    half = len(d.req_idx) // 2
    plan = rx.Plan()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    outs = []
    for sel, st in ((np.arange(half), s1), (np.arange(half, len(d.req_idx)), s2)):
        rx.decode_plan(plan, dw.desc, d.req_idx[sel], d.seq_len[sel])
        ws = torch.empty(plan.workspace_size(), dtype=torch.uint8, device=cuda)
        q = dw.steps[0].dec_q[torch.as_tensor(sel, device=cuda)].contiguous()
        o = torch.empty_like(q)
        l = torch.empty((len(sel), wl.num_q_heads), dtype=torch.float32, device=cuda)
        with torch.cuda.stream(st):
            plan.upload(ws, stream=st)
            rx.decode_attn(plan, dw.desc, dw.k_pool, dw.v_pool, q, o, l, ws, stream=st)
        outs.append((sel, o, l, ws))
    torch.cuda.synchronize()
    kp, vp = oracle_pools(wl, 0)
    for sel, o, l, _ in outs:
        ro, rl = A.decode(d.q[sel], kp, vp, wl.req_to_token, d.req_idx[sel], d.seq_len[sel],
                          wl.softmax_scale)
        assert_close(o, l, ro, rl, None, "decode, plan rebuilt between uploads")


@pytest.mark.parametrize("hq,hkv,chunk", [(8, 2, 512), (16, 16, 256)])
def test_chunked_prefill_mixed_with_decode(cuda, hq, hkv, chunk):
    """A long prompt prefilled chunk by chunk (each chunk an extend over the system prompt and the
    earlier chunks) beside decode requests that share the system prompt, every step checked."""
    wl = W.chunked_prefill_workload(8, hq, hkv, system=256, prompt=1200, chunk=chunk,
                                    n_decode=6, tail_lo=20, tail_hi=120)
    run_and_check(wl, cuda)


# ---------------------------------------------------------------------------------------------
# Prefix trees (rx_decode_plan_tree / rx_extend_plan_tree): every node read once for the requests
# beneath it, partials of all levels merged; the result is the plain definition's.
# ---------------------------------------------------------------------------------------------

@pytest.mark.parametrize("seed,hq,hkv,depth,fanout,p_empty", [
    (21, 8, 8, 3, 3, 0.0),     # MHA, bushy
    (22, 8, 2, 4, 3, 0.3),     # GQA 4, empty node segments
    (23, 32, 8, 6, 1, 0.2),    # a chain six levels deep
    (24, 16, 2, 3, 4, 0.5),    # GQA 8, many empty nodes
])
def test_tree_decode_and_extend(cuda, seed, hq, hkv, depth, fanout, p_empty):
    wl = W.tree_workload(seed, hq, hkv, depth=depth, fanout=fanout, seg_lo=1, seg_hi=150,
                         p_empty=p_empty, n_decode=40, tail_hi=90, n_extend=10, own_hi=60,
                         ext_lo=1, ext_hi=140)
    run_and_check(wl, cuda)


def test_tree_decode_many_members_per_node(cuda):
    # 150 decode requests under a 3-node chain: the root has more members than one member tile
    wl = W.tree_workload(25, 32, 32, depth=3, fanout=1, seg_lo=200, seg_hi=1500, p_empty=0.0,
                         n_decode=150, tail_hi=40, n_extend=0, own_hi=0, ext_lo=1, ext_hi=1)
    run_and_check(wl, cuda)


def test_tree_and_one_level_plans_agree(cuda):
    wl = W.tree_workload(26, 16, 4, depth=4, fanout=2, seg_lo=30, seg_hi=300, p_empty=0.1,
                         n_decode=30, tail_hi=60, n_extend=0, own_hi=0, ext_lo=1, ext_hi=1)
    dw = DeviceWorkload(wl, cuda)
    dw.run_step(0)
    d = wl.steps[0].decode
    plan = rx.Plan()
    rx.decode_plan(plan, dw.desc, d.req_idx, d.seq_len)          # no groups declared
    assert plan.key_reads() > dw.steps[0].dec_plan.key_reads()
    ws = torch.empty(plan.workspace_size(), dtype=torch.uint8, device=cuda)
    plan.upload(ws)
    o2 = torch.empty_like(dw.steps[0].dec_o)
    l2 = torch.empty_like(dw.steps[0].dec_lse)
    rx.decode_attn(plan, dw.desc, dw.k_pool, dw.v_pool, dw.steps[0].dec_q, o2, l2, ws)
    torch.cuda.synchronize()
    a = A.bf16_to_f64(bits_of(o2))
    b = A.bf16_to_f64(bits_of(dw.steps[0].dec_o))
    assert np.abs(a - b).max() <= MAX_ABS
    assert (l2 - dw.steps[0].dec_lse).abs().max().item() <= LSE_ABS


# ---------------------------------------------------------------------------------------------
# Block-granular pools (prefix-caching comparison page: vLLM's 16-token blocks): the kernels index
# KV per token slot, so a paged pool is slots page * 16 + i; only whole pages of the prefix are
# reused and the rest is recomputed as part of the extend.
# ---------------------------------------------------------------------------------------------

@pytest.mark.parametrize("hq,hkv,prefix", [(8, 2, 1000), (32, 32, 517), (16, 16, 16)])
def test_block_granular_pool(cuda, hq, hkv, prefix):
    wl = W.paged_workload(40 + prefix, hq, hkv, page=16, prefix=prefix, n_req=5, ext_lo=1,
                          ext_hi=140)
    run_and_check(wl, cuda)


def test_block_granular_pool_odd_pages_and_mid_page_prefix(cuda):
    """Pages of 24 slots (a page boundary inside a kernel step, pages not aligned to 16 slots);
    pages of 16 with a declared shared prefix of 985 while the rows share 992 (the members' own
    keys start mid-page)."""
    run_and_check(W.paged_workload(61, 8, 2, page=24, prefix=1000, n_req=5, ext_lo=1,
                                   ext_hi=150), cuda)
    wl = W.paged_workload(62, 16, 4, page=16, prefix=1000, n_req=6, ext_lo=1, ext_hi=150)
    for st in wl.steps:
        for b in (st.extend, st.decode):
            if b is not None:
                b.group_prefix_len = np.asarray([985], dtype=b.group_prefix_len.dtype)
    run_and_check(wl, cuda)


# ---------------------------------------------------------------------------------------------
# Full-size workloads in the benchmark's configuration.  Every extend and decode row of the
# extend, radix-mixed (tree and one-level) and chunked-prefill workloads; for the two decode
# workloads, whose oracle reads up to 17,000 keys per request, a stratified set of requests
# (every group's shortest and longest member, every own-length decile, every ungrouped request).
# ---------------------------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["extend", "radix-mixed", "radix-mixed-1level",
                                  "chunked-prefill", "paged"])
def test_full_size_workloads_every_row(cuda, name):
    run_and_check(W.NAMED[name](), cuda)


@pytest.mark.parametrize("name", ["decode", "gqa-decode"])
def test_full_size_decode_workloads_stratified(cuda, name):
    wl = W.NAMED[name]()
    picked = stratified_decode_requests(wl.steps[0].decode)
    assert len(picked) >= 2 * 16  # both ends of every group at least
    run_and_check(wl, cuda, decode_pick=stratified_decode_requests)


# ---------------------------------------------------------------------------------------------
# Failure detection on the GPU without a fault: a bounded wait that nothing completes gives up,
# records RX_ERR_TIMEOUT in the status word and leaves the context usable.
# ---------------------------------------------------------------------------------------------

def test_bounded_wait_times_out_and_the_context_stays_usable(cuda):
    import time
    status = torch.zeros(1, dtype=torch.int32, device=cuda)
    t0 = time.perf_counter()
    rx.selftest_wait_timeout(status, 20_000_000)        # 20 ms
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    assert status.item() == rx.RX_ERR_TIMEOUT
    assert 0.015 < waited < 1.5
    status.zero_()
    rx.selftest_wait_timeout(status, 5_000_000)
    torch.cuda.synchronize()
    assert status.item() == rx.RX_ERR_TIMEOUT
    run_and_check(W.tiny(), cuda)                        # kernels still run and agree


@pytest.mark.parametrize("hq,hkv", [(32, 32), (32, 8)])
def test_table_entry_outside_the_pool_is_flagged(cuda, hq, hkv):
    """An entry of req_to_token outside the pool is not read (the kernels read zeros instead) and
    sets RX_ERR_RANGE in the workspace status word; rx_read_status reports and clears it.  Checked
    for the extend kernel and, in a shared prefix (tensor-core units at gq = 4, mma.sync units at
    gq = 1) and in a request's own keys, for the decode kernels."""
    ext = W.extend_workload(60 + hkv, hq, hkv, n_groups=2, members=4, prefix=600, ext_lo=10,
                            ext_hi=90, ungrouped=1, ungrouped_prefix=300)
    dec = W.decode_workload(70 + hkv, hq, hkv, n_groups=2, members=9, prefix=900, dist_lo=20,
                            dist_hi=300, ungrouped=2)
    for wl, kind in ((ext, "extend"), (dec, "decode")):
        dw = DeviceWorkload(wl, cuda)
        dw.store(0)
        ds = dw.steps[0]
        b = wl.steps[0].extend if kind == "extend" else wl.steps[0].decode
        run = dw.extend if kind == "extend" else dw.decode
        ws = ds.ext_ws if kind == "extend" else ds.dec_ws
        grp = np.asarray(b.group_of_req)
        for where in ("shared prefix", "own keys"):
            saved = dw.r2t.clone()
            if where == "shared prefix":
                for r in np.flatnonzero(grp == 0):  # every member's row, so they stay equal
                    dw.r2t[int(b.req_idx[r]), 123] = wl.pool_size + 3
            else:
                r = int(np.flatnonzero(grp < 0)[0])
                n = int(b.prefix_len[r] + b.extend_len[r]) if kind == "extend" else int(b.seq_len[r])
                dw.r2t[int(b.req_idx[r]), n // 2] = wl.pool_size + 3
            run(0)
            assert rx.read_status(ws) == rx.RX_ERR_RANGE, (kind, where)
            assert rx.read_status(ws) == rx.RX_OK
            dw.r2t.copy_(saved)
            run(0)
            assert rx.read_status(ws) == rx.RX_OK
    run_and_check(W.tiny(), cuda)  # the context still runs and agrees


# ---------------------------------------------------------------------------------------------
# Random shapes: extend, decode and tree workloads with random head ratios, group sizes, prefix
# and tail lengths (empty parts included), each checked against the oracle.
# ---------------------------------------------------------------------------------------------

def _random_workload(rng, i):
    hkv = int(rng.choice([1, 2, 4, 8]))
    hq = hkv * int(rng.choice([1, 2, 4, 8]))
    seed = int(rng.integers(0, 1 << 30))
    kind = i % 3
    if kind == 0:
        return W.extend_workload(seed, hq, hkv, n_groups=int(rng.integers(0, 4)),
                                 members=int(rng.integers(1, 9)),
                                 prefix=int(rng.integers(0, 1500)),
                                 ext_lo=int(rng.integers(0, 30)), ext_hi=int(rng.integers(30, 300)),
                                 own_cached_hi=int(rng.integers(0, 100)),
                                 ungrouped=int(rng.integers(0, 4)),
                                 ungrouped_prefix=int(rng.integers(0, 700)))
    if kind == 1:
        return W.decode_workload(seed, hq, hkv, n_groups=int(rng.integers(1, 4)),
                                 members=int(rng.integers(1, 40)),
                                 prefix=int(rng.integers(0, 5000)), dist_lo=1,
                                 dist_hi=int(rng.integers(1, 800)),
                                 ungrouped=int(rng.integers(0, 4)))
    return W.tree_workload(seed, hq, hkv, depth=int(rng.integers(1, 5)),
                           fanout=int(rng.integers(1, 4)), seg_lo=0,
                           seg_hi=int(rng.integers(1, 600)), p_empty=float(rng.random() * 0.4),
                           n_decode=int(rng.integers(1, 40)), tail_hi=int(rng.integers(0, 80)),
                           n_extend=int(rng.integers(1, 12)), own_hi=int(rng.integers(0, 60)),
                           ext_lo=int(rng.integers(1, 20)), ext_hi=int(rng.integers(20, 200)))


@pytest.mark.parametrize("seed", [301, 302, 303])
def test_random_workloads(cuda, seed):
    rng = np.random.default_rng(seed)
    for i in range(10):
        run_and_check(_random_workload(rng, i), cuda)
