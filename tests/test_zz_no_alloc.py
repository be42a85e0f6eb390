"""rx_decode_attn_noalloc: decode for callers that cannot allocate device memory.

Such a caller (for example a custom operator that a host framework hands only its input and
output buffers, or a runtime that forbids allocation while serving under a fixed memory budget)
cannot provide a workspace.  The entry point keeps the plan tables and partial results in the
library's own scratch instead.  These tests call it through the C ABI twice in a row and compare
each result with the fp64 oracle and with the workspace-based rx_decode_attn on the same inputs;
check that a table entry outside the pool is reported through rx_noalloc_read_status; and check
that a plan larger than the scratch is refused before anything runs.  The file is collected last
so that a failure here does not stop the rest of the suite from running first.
"""
import numpy as np
import pytest
import torch

from oracle import attention as A
from prefix_shared_kv_gb300 import rx, workloads as W
from prefix_shared_kv_gb300.session import DeviceWorkload, bits_of

pytestmark = pytest.mark.gpu

MAX_ABS, MEAN_ABS, LSE_ABS = 2e-2, 2e-3, 1e-3


def _close(o_a, lse_a, o_ref, lse_ref):
    """o_a, lse_a: device results; o_ref, lse_ref: float64 arrays of the same shapes."""
    a = A.bf16_to_f64(bits_of(o_a))
    err = np.abs(a - o_ref)
    assert np.isfinite(a).all() and np.isfinite(o_ref).all()
    assert err.max() <= MAX_ABS and err.mean() <= MEAN_ABS
    assert np.abs(lse_a.double().cpu().numpy() - lse_ref).max() <= LSE_ABS


def _workload(hq, hkv):
    # 4 groups of 9 on a 1500-token prefix (36 stacked rows per KV head at gq = 4: the shared
    # units go to the tensor-core kernel; 9 rows at gq = 1: to the mma.sync kernel) + 5 ungrouped
    return W.decode_workload(301 + hkv, hq, hkv, n_groups=4, members=9, prefix=1500, dist_lo=20,
                             dist_hi=600, ungrouped=5)


@pytest.mark.parametrize("hq,hkv", [(32, 32), (32, 8)])
def test_noalloc_decode_matches_the_oracle_and_the_workspace_decode_on_two_calls(cuda, hq, hkv):
    wl = _workload(hq, hkv)
    dw = DeviceWorkload(wl, cuda)
    dw.run_step(0)  # stores the step's KV and runs the workspace-based decode
    ds = dw.steps[0]
    assert ds.dec_plan.workspace_size() <= rx.noalloc_scratch_bytes()
    st = wl.steps[0]
    kp, vp = A.store_kv(wl.k_pool, wl.v_pool, st.k_new, st.v_new, st.store_slots)
    d = st.decode
    o_ref, lse_ref = A.decode(d.q, kp, vp, wl.req_to_token, d.req_idx, d.seq_len,
                              wl.softmax_scale)
    torch.cuda.synchronize()
    ws_o, ws_lse = ds.dec_o.clone(), ds.dec_lse.clone()
    _close(ws_o, ws_lse, o_ref, lse_ref)
    for _ in range(2):
        o = torch.full_like(ws_o, float("nan"))
        lse = torch.full_like(ws_lse, float("nan"))
        rx.decode_attn_noalloc(ds.dec_plan, dw.desc, dw.k_pool, dw.v_pool, ds.dec_q, o, lse)
        assert rx.noalloc_read_status() == rx.RX_OK
        _close(o, lse, o_ref, lse_ref)
        _close(o, lse, A.bf16_to_f64(bits_of(ws_o)), ws_lse.double().cpu().numpy())


@pytest.mark.parametrize("hq,hkv", [(32, 32), (32, 8)])
def test_noalloc_reports_a_table_entry_outside_the_pool(cuda, hq, hkv):
    wl = _workload(hq, hkv)
    dw = DeviceWorkload(wl, cuda)
    dw.store(0)
    ds = dw.steps[0]
    d = wl.steps[0].decode
    o = torch.empty_like(ds.dec_o)
    lse = torch.empty_like(ds.dec_lse)
    grp = np.asarray(d.group_of_req)
    for where in ("shared prefix", "own keys"):
        saved = dw.r2t.clone()
        if where == "shared prefix":
            # key 700 of group 0's prefix, in every member's row (the rows stay equal there)
            for b in np.flatnonzero(grp == 0):
                dw.r2t[int(d.req_idx[b]), 700] = wl.pool_size + 3
        else:
            b = int(np.flatnonzero(grp < 0)[0])  # an ungrouped request: its own keys only
            dw.r2t[int(d.req_idx[b]), int(d.seq_len[b]) // 2] = wl.pool_size + 3
        rx.decode_attn_noalloc(ds.dec_plan, dw.desc, dw.k_pool, dw.v_pool, ds.dec_q, o, lse)
        assert rx.noalloc_read_status() == rx.RX_ERR_RANGE, where
        assert rx.noalloc_read_status() == rx.RX_OK  # the read cleared it
        dw.r2t.copy_(saved)
        rx.decode_attn_noalloc(ds.dec_plan, dw.desc, dw.k_pool, dw.v_pool, ds.dec_q, o, lse)
        assert rx.noalloc_read_status() == rx.RX_OK


def test_noalloc_refuses_a_plan_larger_than_its_scratch(cuda):
    # a plan for 4096 requests of 60000 keys: its partial results exceed the scratch
    rows, stride = 4096, 65536
    desc = rx.KVDesc(32, 32, 128, 128 ** -0.5, 1 << 20, 0x1000, rows, stride)
    plan = rx.Plan()
    rx.decode_plan(plan, desc, np.arange(rows), np.full(rows, 60000))
    assert plan.workspace_size() > rx.noalloc_scratch_bytes()
    with pytest.raises(rx.RxError) as e:
        rx.decode_attn_noalloc(plan, desc, 256, 256, 256, 256, 256)
    assert e.value.status == rx.RX_ERR_WORKSPACE
    assert "scratch" in str(e.value)
