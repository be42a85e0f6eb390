"""Parity of the SM-pair extend kernel (rx_plan_set_extend_kernel(RX_EXTEND_PAIR): a cluster of
two CTAs per item, tcgen05 cta_group::2, 128-key steps) with the fp64 oracle, at the tolerances
of the default kernel: the small extend cases element by element, the full-size extend workloads
on every row, random extend and tree workloads, and the status word on a table entry outside
the pool.  Decode plans are not affected by the choice; the tree workloads run them too."""
import numpy as np
import pytest

from prefix_shared_kv_gb300 import rx, workloads as W
from prefix_shared_kv_gb300.session import DeviceWorkload

from test_parity_gpu import _random_workload, run_and_check

pytestmark = pytest.mark.gpu

PAIR = rx.RX_EXTEND_PAIR


def check(wl, cuda):
    return run_and_check(wl, cuda, extend_kernel=PAIR)


@pytest.mark.parametrize("hq,hkv", [(4, 4), (8, 2), (16, 2), (8, 4), (32, 4)])
def test_shapes(cuda, hq, hkv):
    check(W.extend_workload(200 + hq + hkv, hq, hkv, n_groups=2, members=5, prefix=333, ext_lo=1,
                            ext_hi=150, own_cached_hi=70, ungrouped=2, ungrouped_prefix=129),
          cuda)


def test_one_step_items_and_empty_requests(cuda):
    """Items of one to three steps back to back (the query rows of one item are copied in while
    the previous item's last steps run), and requests with nothing to extend."""
    check(W.extend_workload(17, 8, 8, n_groups=3, members=6, prefix=65, ext_lo=0, ext_hi=3,
                            ungrouped=3, ungrouped_prefix=0), cuda)
    check(W.extend_workload(18, 8, 2, n_groups=6, members=2, prefix=129, ext_lo=1, ext_hi=20,
                            ungrouped=4, ungrouped_prefix=40), cuda)


def test_long_causal_and_long_prefix(cuda):
    check(W.extend_workload(8, 8, 8, n_groups=0, members=0, prefix=0, ext_lo=300, ext_hi=700,
                            ungrouped=2, ungrouped_prefix=0), cuda)
    check(W.extend_workload(10, 8, 2, n_groups=1, members=3, prefix=32000, ext_lo=1, ext_hi=40,
                            ungrouped=1, ungrouped_prefix=20000), cuda)


def test_empty_batch(cuda):
    check(W.extend_workload(3, 4, 2, n_groups=0, members=3, prefix=100, ext_lo=1, ext_hi=30,
                            ungrouped=0), cuda)


def test_peaky_softmax(cuda):
    from oracle import attention as A
    wl = W.extend_workload(9, 8, 2, n_groups=1, members=4, prefix=200, ext_lo=30, ext_hi=90)
    for st in wl.steps:
        q = A.bf16_to_f64(st.extend.q) * 4.0
        st.extend.q = W.bf16_bits(q.astype(np.float32))
    check(wl, cuda)


@pytest.mark.parametrize("name", ["extend", "radix-mixed", "radix-mixed-1level",
                                  "chunked-prefill"])
def test_full_size_workloads_every_row(cuda, name):
    check(W.NAMED[name](), cuda)


@pytest.mark.parametrize("seed", [401, 402])
def test_random_extend_and_tree_workloads(cuda, seed):
    rng = np.random.default_rng(seed)
    for i in range(12):
        wl = _random_workload(rng, i)
        if i % 3 != 1:  # the decode-only kind does not reach the extend kernel
            check(wl, cuda)


def test_table_entry_outside_the_pool_is_flagged(cuda):
    wl = W.extend_workload(61, 32, 8, n_groups=2, members=4, prefix=600, ext_lo=10, ext_hi=90,
                           ungrouped=1, ungrouped_prefix=300)
    dw = DeviceWorkload(wl, cuda, extend_kernel=PAIR)
    dw.store(0)
    b = wl.steps[0].extend
    grp = np.asarray(b.group_of_req)
    saved = dw.r2t.clone()
    for r in np.flatnonzero(grp == 0):
        dw.r2t[int(b.req_idx[r]), 123] = wl.pool_size + 3
    dw.extend(0)
    assert rx.read_status(dw.steps[0].ext_ws) == rx.RX_ERR_RANGE
    assert rx.read_status(dw.steps[0].ext_ws) == rx.RX_OK
    dw.r2t.copy_(saved)
    dw.extend(0)
    assert rx.read_status(dw.steps[0].ext_ws) == rx.RX_OK
    check(W.tiny(), cuda)

