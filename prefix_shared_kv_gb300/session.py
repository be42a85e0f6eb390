"""Device-side driver of a workload through the C ABI.

Holds the device tensors of a seeded workload (pools, request->slot table, per-step new KV, query
rows, outputs, plans and workspaces) and runs its steps: rx_store_kv, then rx_extend_attn and/or
rx_decode_attn.  Torch provides the device memory and the stream; every step of the path runs in
librx's kernels.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import List, Optional

import numpy as np
import torch

from . import rx
from .workloads import Workload


def to_bf16(a: np.ndarray, device) -> torch.Tensor:
    """uint16 bf16 bit patterns -> bf16 tensor on `device` (bit copy)."""
    t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16))
    return t.to(device).view(torch.bfloat16)


def to_i32(a: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)


def bits_of(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> uint16 bit patterns on the host."""
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)


@dataclass
class DevStep:
    slots: torch.Tensor
    k_new: torch.Tensor
    v_new: torch.Tensor
    ext_plan: Optional[rx.Plan] = None
    ext_ws: Optional[torch.Tensor] = None
    ext_q: Optional[torch.Tensor] = None
    ext_o: Optional[torch.Tensor] = None
    ext_lse: Optional[torch.Tensor] = None
    dec_plan: Optional[rx.Plan] = None
    dec_ws: Optional[torch.Tensor] = None
    dec_q: Optional[torch.Tensor] = None
    dec_o: Optional[torch.Tensor] = None
    dec_lse: Optional[torch.Tensor] = None


def fill_normal_bf16(t: torch.Tensor, seed: int) -> None:
    """Fill a bf16 device tensor with fp32 N(0,1) draws rounded to bf16 (round-to-nearest-even)
    from a seeded torch generator on the tensor's device, a chunk at a time."""
    g = torch.Generator(device=t.device)
    g.manual_seed(seed)
    flat = t.view(-1)
    step = 1 << 26
    for s in range(0, flat.numel(), step):
        n = min(step, flat.numel() - s)
        flat[s:s + n] = torch.randn(n, generator=g, device=t.device,
                                    dtype=torch.float32).to(torch.bfloat16)


def workspace(nbytes: int, device) -> torch.Tensor:
    # torch's caching allocator returns 512-byte aligned blocks
    return torch.empty(max(256, nbytes), dtype=torch.uint8, device=device)


class DeviceWorkload:
    """`pool_seed`: for a workload built structure-only (values=False, no cached KV drawn on the
    host), the pools are allocated on the device and every slot is filled with N(0,1) bf16 values
    from this seed (K with pool_seed, V with pool_seed + 1).  Used where only timing matters;
    parity checks use host-drawn pools, which the oracle reads too.  `extend_kernel`: the
    tensor-core kernel the extend plans run on (rx.RX_EXTEND_TILES or rx.RX_EXTEND_PAIR)."""

    def __init__(self, wl: Workload, device="cuda", stream=None, pool_seed=None,
                 extend_kernel=rx.RX_EXTEND_TILES):
        self.wl = wl
        self.device = torch.device(device)
        self.stream = stream
        if wl.k_pool.shape[0] == 0 and wl.pool_size > 0:
            if pool_seed is None:
                raise ValueError("structure-only workload: pass pool_seed to fill its pools")
            shape = (wl.pool_size, wl.num_kv_heads, wl.head_dim)
            self.k_pool = torch.empty(shape, dtype=torch.bfloat16, device=self.device)
            self.v_pool = torch.empty(shape, dtype=torch.bfloat16, device=self.device)
            fill_normal_bf16(self.k_pool, pool_seed)
            fill_normal_bf16(self.v_pool, pool_seed + 1)
        else:
            self.k_pool = to_bf16(wl.k_pool, self.device)
            self.v_pool = to_bf16(wl.v_pool, self.device)
        self.r2t = to_i32(wl.req_to_token, self.device)
        self.desc = rx.kv_desc(wl.num_q_heads, wl.num_kv_heads, wl.pool_size, self.r2t,
                               wl.softmax_scale)
        self.steps: List[DevStep] = []
        hq, d = wl.num_q_heads, wl.head_dim
        for st in wl.steps:
            ds = DevStep(to_i32(st.store_slots, self.device), to_bf16(st.k_new, self.device),
                         to_bf16(st.v_new, self.device))
            if st.extend is not None:
                e = st.extend
                ds.ext_plan = rx.Plan()
                ds.ext_plan.set_extend_kernel(extend_kernel)
                rx.extend_plan(ds.ext_plan, self.desc, e.req_idx, e.prefix_len, e.extend_len,
                               e.group_of_req, e.group_prefix_len, e.group_parent)
                ds.ext_ws = workspace(ds.ext_plan.workspace_size(), self.device)
                ds.ext_plan.upload(ds.ext_ws, stream=stream)
                ds.ext_q = to_bf16(e.q, self.device)
                n = e.q.shape[0]
                ds.ext_o = torch.empty((n, hq, d), dtype=torch.bfloat16, device=self.device)
                ds.ext_lse = torch.empty((n, hq), dtype=torch.float32, device=self.device)
            if st.decode is not None:
                dc = st.decode
                ds.dec_plan = rx.Plan()
                rx.decode_plan(ds.dec_plan, self.desc, dc.req_idx, dc.seq_len, dc.group_of_req,
                               dc.group_prefix_len, dc.group_parent)
                ds.dec_ws = workspace(ds.dec_plan.workspace_size(), self.device)
                ds.dec_plan.upload(ds.dec_ws, stream=stream)
                ds.dec_q = to_bf16(dc.q, self.device)
                n = dc.q.shape[0]
                ds.dec_o = torch.empty((n, hq, d), dtype=torch.bfloat16, device=self.device)
                ds.dec_lse = torch.empty((n, hq), dtype=torch.float32, device=self.device)
            self.steps.append(ds)

    def store(self, i: int):
        ds = self.steps[i]
        rx.store_kv(self.desc, self.k_pool, self.v_pool, ds.k_new, ds.v_new, ds.slots, self.stream)

    def extend(self, i: int):
        ds = self.steps[i]
        if ds.ext_plan is not None:
            rx.extend_attn(ds.ext_plan, self.desc, self.k_pool, self.v_pool, ds.ext_q, ds.ext_o,
                           ds.ext_lse, ds.ext_ws, self.stream)

    def decode(self, i: int):
        ds = self.steps[i]
        if ds.dec_plan is not None:
            rx.decode_attn(ds.dec_plan, self.desc, self.k_pool, self.v_pool, ds.dec_q, ds.dec_o,
                           ds.dec_lse, ds.dec_ws, self.stream)

    def run_step(self, i: int):
        self.store(i)
        self.extend(i)
        self.decode(i)

    def run_all(self):
        for i in range(len(self.steps)):
            self.run_step(i)
