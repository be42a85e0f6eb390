"""rx_decode_attn_noalloc: decode for callers that cannot allocate device memory.

Such a caller (for example a custom operator that a host framework hands only its input and
output buffers, or a runtime that forbids allocation while serving under a fixed memory budget)
cannot provide a workspace.  The entry point keeps the plan tables and partial results in the
library's own scratch instead.  These tests call it through the C ABI twice in a row and compare
each result with the workspace-based rx_decode_attn on the same inputs, and check that a plan
larger than the scratch is refused before anything runs.  The file is collected last so that a
failure here does not stop the rest of the suite from running first.
"""
import ctypes

import numpy as np
import pytest
import torch

from oracle import attention as A
from prefix_shared_kv_gb300 import rx, workloads as W
from prefix_shared_kv_gb300.session import DeviceWorkload, bits_of

pytestmark = pytest.mark.gpu

MAX_ABS, MEAN_ABS, LSE_ABS = 2e-2, 2e-3, 1e-3


def _close(o_a, lse_a, o_b, lse_b):
    a = A.bf16_to_f64(bits_of(o_a))
    b = A.bf16_to_f64(bits_of(o_b))
    err = np.abs(a - b)
    assert np.isfinite(a).all()
    assert err.max() <= MAX_ABS and err.mean() <= MEAN_ABS
    assert (lse_a.double() - lse_b.double()).abs().max().item() <= LSE_ABS


@pytest.mark.parametrize("hq,hkv", [(32, 32), (32, 8)])
def test_noalloc_decode_matches_workspace_decode_on_two_calls(cuda, hq, hkv):
    wl = W.decode_workload(301 + hkv, hq, hkv, n_groups=4, members=9, prefix=1500, dist_lo=20,
                           dist_hi=600, ungrouped=5)
    dw = DeviceWorkload(wl, cuda)
    dw.run_step(0)  # stores the step's KV and runs the workspace-based decode
    ds = dw.steps[0]
    assert ds.dec_plan.workspace_size() <= rx.NOALLOC_SCRATCH_BYTES
    ref_o, ref_lse = ds.dec_o.clone(), ds.dec_lse.clone()
    for _ in range(2):
        o = torch.full_like(ref_o, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        rx.decode_attn_noalloc(ds.dec_plan, dw.desc, dw.k_pool, dw.v_pool, ds.dec_q, o, lse)
        torch.cuda.synchronize()
        _close(o, lse, ref_o, ref_lse)


def test_noalloc_refuses_a_plan_larger_than_its_scratch(cuda):
    # a plan for 4096 requests of 60000 keys: its partial results exceed the scratch
    rows, stride = 4096, 65536
    desc = rx.KVDesc(32, 32, 128, 128 ** -0.5, 1 << 20, 0x1000, rows, stride)
    plan = rx.Plan()
    rx.decode_plan(plan, desc, np.arange(rows), np.full(rows, 60000))
    assert plan.workspace_size() > rx.NOALLOC_SCRATCH_BYTES
    with pytest.raises(rx.RxError) as e:
        rx.decode_attn_noalloc(plan, desc, 256, 256, 256, 256, 256)
    assert e.value.status == rx.RX_ERR_WORKSPACE
    assert "scratch" in str(e.value)
