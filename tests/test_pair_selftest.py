"""The tensor-core steps of the extend kernel that runs on a pair of SMs (tcgen05 .cta_group::2),
checked on one cluster against plain fp32 matrix products of the same bf16 operands: S = Q K^T with
M = 256 query rows split over the two CTAs and the 128 keys of a step split into halves, and
O = P V with P read from tensor memory and V's columns split into halves."""
import pytest
import torch

from prefix_shared_kv_gb300 import rx

pytestmark = pytest.mark.gpu


def test_pair_mma_matches_a_plain_product(cuda):
    g = torch.Generator().manual_seed(5)
    q, k, v = (torch.randn(n, 128, generator=g).to(torch.bfloat16) for n in (256, 128, 128))
    p = torch.rand(256, 128, generator=g).to(torch.bfloat16)
    dq, dk, dv, dp = (t.to(cuda) for t in (q, k, v, p))
    s_out = torch.full((256, 128), float("nan"), device=cuda)
    o_out = torch.full((256, 128), float("nan"), device=cuda)
    for _ in range(2):
        info = torch.tensor([0, -7, -7], dtype=torch.int32, device=cuda)  # status starts at OK
        rx.selftest_pair_mma(dq, dk, dv, dp, s_out, o_out, info)
        torch.cuda.synchronize()
        st, a0, a1 = info.tolist()
        assert st == rx.RX_OK
        assert a0 == a1 == 0, f"tensor-memory addresses of the pair: {a0:#x}, {a1:#x}"
        s_ref = q.double() @ k.double().T
        o_ref = p.double() @ v.double()
        es = (s_out.double().cpu() - s_ref).abs()
        eo = (o_out.double().cpu() - o_ref).abs()
        for name, e, ref in (("S", es, s_ref), ("O", eo, o_ref)):
            for half in (0, 1):  # rows of each CTA of the pair
                err = e[128 * half:128 * (half + 1)]
                assert err.max().item() < 1e-3 * ref.abs().max().item(), \
                    f"{name} rows of CTA {half}: max error {err.max().item():.4g}"
