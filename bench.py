#!/usr/bin/env python3
"""Benchmark of the prefix-shared KV attention path on one GB300 per rank.

One step = one pass of the whole hot path over one batch: host prefix match of the batch's
requests (radix cache), rx_store_kv of the step's new tokens, rx_extend_attn and rx_decode_attn.
The default workload is the radix-tree mixed batch (1000-token system prompt -> 8 x 500 -> 32 x
200 leaves; 16 leaf requests extend 64 tokens, 8 cache misses prefill 1500 tokens, 40 decode
requests), the one batch that exercises every part of the path.

Printed metric (one JSON line on rank 0): `value` = extend FLOPs of the batch divided by the device
time of the whole step (store + extend + decode), in TFLOP/s; `parts` gives each part against its
own roofline (decode: unique KV bytes / time vs HBM; extend: FLOPs / time vs bf16 tensor peak;
store: bytes moved / time).  Decode-only workloads report decode GB/s instead.  `per_workload`
adds the extend, decode and gqa-decode configurations, each timed the same way in the same
process (their pools filled with N(0,1) bf16 on the device, so that the host does not draw
gigabytes of KV), with its own parts and clock record.

Timing: W warm-up steps, then K steps, each bracketed by CUDA events on the launch stream with an
L2 flush between steps (outside the events: a 256 MiB buffer written, then another read, so no
dirty flush lines are left for the step to write back); barrier + synchronize on both sides; max
over ranks.  `--impl reference` times the fp64 oracle on host cores on a bounded sample instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "prefix-shared attn: decode KV GB/s (% HBM peak); extend TFLOP/s (% BF16 peak)"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# nominal GB300 figures, reported beside the measured denominators (context only)
NOMINAL_HBM_GBS, NOMINAL_BF16_TFLOPS = 8000.0, 2250.0


# ---------------------------------------------------------------------------------------------
# Algorithmic work of a workload (what the method must compute / move, nothing more)
# ---------------------------------------------------------------------------------------------

def work_counts(wl, step=0):
    st = wl.steps[step]
    d, hq, hkv = wl.head_dim, wl.num_q_heads, wl.num_kv_heads
    out = {"extend_flops": 0.0, "decode_kv_bytes": 0.0, "store_bytes": 0.0,
           "extend_rows": 0, "decode_rows": 0}
    out["store_bytes"] = float(len(st.store_slots)) * hkv * d * 2 * 2 * 2  # K,V x read+write
    if st.extend is not None:
        e = st.extend
        p = e.prefix_len.astype(np.float64)
        E = e.extend_len.astype(np.float64)
        out["extend_flops"] = float(4.0 * d * hq * np.sum(E * p + E * (E + 1) / 2))
        out["extend_rows"] = int(E.sum())
    if st.decode is not None:
        dc = st.decode
        # the least the method must read: every distinct pool slot the batch attends to, once
        slots = np.concatenate([wl.req_to_token[r, :n] for r, n in zip(dc.req_idx, dc.seq_len)])
        tokens = float(np.unique(slots).size)
        out["decode_kv_bytes"] = tokens * hkv * d * 2 * 2
        out["decode_rows"] = int(len(dc.req_idx))
    return out


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return {k: float(pk[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


# ---------------------------------------------------------------------------------------------
# Clocks during the timed region
# ---------------------------------------------------------------------------------------------

class ClockSampler:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        try:
            with open(self.path) as f:
                return self.parse(f.readlines())
        finally:
            os.unlink(self.path)

    @staticmethod
    def parse(lines):
        """Lines of the query above (csv, no header, no units) -> median SM clock, the largest
        maximum clock, the sample count and the slowdown reasons seen active; None without a
        usable sample."""
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------------------------
# Oracle (CPU) timing on a bounded sample -- the reference arm and the cpu_baseline
# ---------------------------------------------------------------------------------------------

def oracle_sample_rate(wl, budget_s=12.0):
    """Time the fp64 oracle on a bounded sample of the step and scale it to the whole step.
    Returns (extend TFLOP/s equivalent, decode GB/s equivalent, est. step seconds, sample text,
    threads)."""
    from oracle import attention as A
    st = wl.steps[0]
    kp, vp = A.store_kv(wl.k_pool, wl.v_pool, st.k_new, st.v_new, st.store_slots)
    w = work_counts(wl)
    d, hq = wl.head_dim, wl.num_q_heads
    t_ext = t_dec = 0.0
    f_done = b_done = 0.0
    n_ext = n_dec = 0
    if st.extend is not None:
        e = st.extend
        order = np.argsort(-(e.extend_len.astype(np.int64)))  # mix long and short requests
        order = np.concatenate([order[::2], order[1::2]])
        t0 = time.perf_counter()
        for r in order:
            if e.extend_len[r] == 0:
                continue
            A.extend(e.q, kp, vp, wl.req_to_token, e.req_idx, e.prefix_len, e.extend_len, e.cu_q,
                     wl.softmax_scale, requests=[int(r)])
            E, p = float(e.extend_len[r]), float(e.prefix_len[r])
            f_done += 4.0 * d * hq * (E * p + E * (E + 1) / 2)
            n_ext += 1
            if time.perf_counter() - t0 > budget_s * (0.7 if st.decode is not None else 1.0):
                break
        t_ext = time.perf_counter() - t0
    if st.decode is not None:
        dc = st.decode
        t0 = time.perf_counter()
        gp_of = lambda b: dc.group_prefix_len[dc.group_of_req[b]] if dc.group_of_req[b] >= 0 else 0
        for b in range(len(dc.req_idx)):
            A.decode(dc.q, kp, vp, wl.req_to_token, dc.req_idx, dc.seq_len, wl.softmax_scale,
                     requests=[b])
            # the oracle reads every key of the request; count the bytes the method must move
            b_done += float(dc.seq_len[b]) * wl.num_kv_heads * d * 4
            n_dec += 1
            if time.perf_counter() - t0 > budget_s * (0.3 if st.extend is not None else 1.0):
                break
        t_dec = time.perf_counter() - t0
    est = 0.0
    if f_done > 0:
        est += t_ext * w["extend_flops"] / f_done
    if b_done > 0:
        naive_bytes = float(np.sum(st.decode.seq_len)) * wl.num_kv_heads * d * 4
        est += t_dec * naive_bytes / b_done
    ext_rate = w["extend_flops"] / est / 1e12 if est > 0 else 0.0
    dec_rate = w["decode_kv_bytes"] / est / 1e9 if est > 0 else 0.0
    try:
        import threadpoolctl
        threads = max(i.get("num_threads", 1) for i in threadpoolctl.threadpool_info()) or 1
    except Exception:
        threads = os.cpu_count() or 1
    sample = (f"{n_ext} extend + {n_dec} decode requests of the batch in fp64 numpy "
              f"({t_ext + t_dec:.1f} s), scaled to the whole step by FLOPs / KV bytes")
    return ext_rate, dec_rate, est, sample, threads


# ---------------------------------------------------------------------------------------------

def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["rx", "reference"], default="rx")
    from prefix_shared_kv_gb300 import workloads as W
    ap.add_argument("--workload", default="radix-mixed", choices=sorted(W.NAMED))
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-workload", action="store_true",
                    help="skip timing the extend / decode / gqa-decode configurations beside "
                         "the main workload")
    ap.add_argument("--only", choices=["store", "extend", "decode"], default=None,
                    help="time one part alone (profiling runs)")
    ap.add_argument("--extend-kernel", choices=["tiles", "pair"], default="tiles",
                    help="the extend kernel: one SM per item (tiles, the default) or an SM pair")
    return ap.parse_args()


def ext_kernel(args):
    from prefix_shared_kv_gb300 import rx
    return rx.RX_EXTEND_PAIR if args.extend_kernel == "pair" else rx.RX_EXTEND_TILES


def dist_init():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
        pg = dist
    return rank, world, local, pg


def barrier(pg, dev=None):
    if pg is not None:
        if dev is not None:
            pg.barrier(device_ids=[dev.index])
        else:
            pg.barrier()


def allreduce_max(pg, x, dev):
    if pg is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def kernel_source_hash(name):
    """sha1 of the kernel's source file followed by the planner's (rx_api.cpp: the order in which
    items run decides what is re-read from DRAM)."""
    h = hashlib.sha1()
    try:
        for f in (name, "rx_api.cpp"):
            h.update(open(os.path.join(ROOT, "prefix_shared_kv_gb300", "csrc", f), "rb").read())
    except OSError:
        return None
    return h.hexdigest()[:12]


def recorded_traffic(kernel_file, workload):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on this exact
    kernel source (hash) and workload; else None."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    h = kernel_source_hash(kernel_file)
    try:
        for line in open(path):
            f = line.split()
            if len(f) >= 4 and f[0] == kernel_file and f[1] == workload and f[3] == h:
                return float(f[2])
    except OSError:
        pass
    return None


def main():
    args = parse_args()
    from prefix_shared_kv_gb300 import workloads as W

    if args.impl == "reference":
        # the oracle on host cores; under torchrun only rank 0 runs it
        if int(os.environ.get("RANK", "0")) != 0:
            return 0
        wl = W.NAMED[args.workload]()
        w = work_counts(wl)
        rates = []
        t0 = time.perf_counter()
        per = max(2.0, min(12.0, 150.0 / max(1, args.steps)))
        for _ in range(args.steps):
            er, dr, est, sample, threads = oracle_sample_rate(wl, budget_s=per)
            rates.append((er, dr, est))
        er = statistics.mean(r[0] for r in rates)
        dr = statistics.mean(r[1] for r in rates)
        est = statistics.mean(r[2] for r in rates)
        primary = er if w["extend_flops"] > 0 else dr
        unit = "TFLOP/s" if w["extend_flops"] > 0 else "GB/s"
        line = {"impl": "reference", "metric": METRIC, "value": primary, "unit": unit,
                "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": est * 1e3, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": {"workload": wl.name, "recipe": wl.recipe},
                "cpu_baseline": {"value": primary, "unit": unit, "cores": threads,
                                 "kind": "oracle", "sample": sample},
                "e2e": {"value": primary, "unit": unit, "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0},
                "wall_s": time.perf_counter() - t0}
        print(json.dumps(line), flush=True)
        return 0

    rank, world, local, pg = dist_init()
    import torch
    from prefix_shared_kv_gb300 import rx
    from prefix_shared_kv_gb300.session import DeviceWorkload

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    rx.lib()
    wl = W.NAMED[args.workload]()
    w = work_counts(wl)
    peaks, peak_src = load_peaks()
    dw = DeviceWorkload(wl, dev, extend_kernel=ext_kernel(args))
    # L2 flush between steps, outside the timed region: write a 256 MiB buffer (twice the L2), then
    # read another one, so that the written lines are back in DRAM before the next step starts
    # (left dirty in L2, their write-back would be timed inside the step's first kernel)
    flush_w = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    flush_r = torch.zeros(256 << 20, dtype=torch.uint8, device=dev)

    def flush_l2():
        flush_w.zero_()
        flush_r.max()

    only = [args.only] if args.only else None
    m = measure(dw, w, args, dev, pg, flush_l2, peaks, only)
    ms_max, part_ms, pdesc, clk, t_wall = m["ms_max"], m["part_ms"], m["parts"], m["clocks"], m["wall"]
    has_ext, has_dec = m["has_ext"], m["has_dec"]
    units_per_step = w["extend_flops"] if has_ext else (w["decode_kv_bytes"] if has_dec else w["store_bytes"])
    scale = 1e12 if has_ext else 1e9
    unit = "TFLOP/s" if has_ext else "GB/s"
    value = world * units_per_step / (ms_max * 1e-3) / scale
    value_is = ("the batch's extend FLOPs (unmasked causal pairs x 4 d Hq) / device time of the "
                "whole step (store + extend + decode); each part against its own roofline is in "
                "'parts'" if has_ext else
                "unique decode KV bytes / device time of the whole step (store + decode); each "
                "part against its own roofline is in 'parts'")

    if has_ext:
        dom = ("extend", "extend_attn.cu")
        roof = {"bound": "tensor", "achieved": pdesc["extend"]["TFLOP/s"],
                "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": pdesc["extend"]["frac_bf16"]}
    elif has_dec:
        dom = ("decode", "decode_attn.cu")
        roof = {"bound": "hbm", "achieved": pdesc["decode"]["GB/s"], "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": pdesc["decode"]["frac_hbm"]}
    else:
        dom = ("store", "store_kv.cu")
        roof = {"bound": "hbm", "achieved": pdesc["store"]["GB/s"], "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": pdesc["store"]["frac_hbm"]}
    roof["kernel"] = dom[0]
    roof["peak_source"] = f"{peak_src} (burst)" if roof["unit"] == "TFLOP/s" else peak_src
    roof["traffic"] = recorded_traffic(dom[1], wl.name)
    roof["traffic_source"] = (
        "recorded: dram__bytes_read.sum + dram__bytes_write.sum per launch from an earlier ncu "
        "capture of this kernel and planner source (hash) on this workload, profiles/dram_traffic.txt; not "
        "measured in this run" if roof["traffic"] is not None else
        "none: no ncu capture recorded for this kernel source and workload")

    gpu_launches = args.steps * m["launches_per_step"]

    # ---- the other configurations, timed the same way in this process ---------------------
    per_workload = None
    if not args.only and not args.no_per_workload:
        per_workload = {}
        del dw
        torch.cuda.empty_cache()
        for name in ("extend", "decode", "gqa-decode", "paged"):
            if name == args.workload:
                continue
            # structure-only build (slots, lengths, new tokens' KV, queries drawn on the host as
            # for the parity tests); every pool slot filled with N(0,1) bf16 on the device
            pwl = W.NAMED[name](values=False)
            pw = work_counts(pwl)
            pdw = DeviceWorkload(pwl, dev, pool_seed=7000 + len(name),
                                 extend_kernel=ext_kernel(args))
            pm = measure(pdw, pw, args, dev, pg, flush_l2, peaks, None)
            per_workload[name] = {"workload": pwl.name, "recipe": pwl.recipe,
                                  "ms_per_step": pm["ms_max"], "parts": pm["parts"],
                                  "clocks": pm["clocks"],
                                  "pools": "every slot N(0,1) bf16, filled on the device"}
            gpu_launches += args.steps * pm["launches_per_step"]
            del pdw
            torch.cuda.empty_cache()
        dw = DeviceWorkload(wl, dev, extend_kernel=ext_kernel(args))

    # ---- end to end through the public API with host buffers -----------------------------
    e2e = None
    if not args.no_e2e and not args.only:
        e2e = run_e2e(wl, dw, dev, args, pg, world, w, unit, scale, has_ext)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not args.only:  # N = 1 only
        er, dr, est, sample, threads = oracle_sample_rate(wl, budget_s=12.0)
        cpu = {"value": er if has_ext else dr, "unit": unit, "cores": threads, "kind": "oracle",
               "sample": sample}

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": unit, "value_is": value_is,
                "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "bf16", "data": "synthetic",
                "config": {"workload": wl.name, "recipe": wl.recipe,
                           "parallelism": f"replicas x{world}",
                           "extend_kernel": args.extend_kernel,
                           "l2": "between timed steps a 256 MiB buffer written, then another "
                                 "256 MiB buffer read (outside the timed region)"},
                "parts": pdesc, "roofline": roof, "gpu_launches": gpu_launches,
                "clocks": clk, "e2e": e2e, "cpu_baseline": cpu, "wall_timed_s": t_wall,
                "per_workload": per_workload}
        if args.only:
            line["only"] = args.only
        print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()
    return 0


def measure(dw, w, args, dev, pg, flush_l2, peaks, only):
    """W warm-up steps, then K timed steps of the workload's parts (CUDA events on the launch
    stream around every part, the L2 flush between steps outside the events, nvidia-smi clock
    samples during the timed steps); the step time is the maximum over ranks."""
    import torch
    wl = dw.wl
    stream = torch.cuda.current_stream(dev)
    parts = [("store", dw.store), ("extend", dw.extend), ("decode", dw.decode)]
    if only:
        parts = [p for p in parts if p[0] in only]
    for _ in range(max(args.warmup, 0)):
        flush_l2()
        for _, f in parts:
            f(0)
    torch.cuda.synchronize(dev)
    barrier(pg, dev)
    torch.cuda.synchronize(dev)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(parts) + 1)]
          for _ in range(args.steps)]
    clocks = ClockSampler(dev.index if dev.index is not None else 0)
    clocks.start()
    t_wall = time.perf_counter()
    for k in range(args.steps):
        flush_l2()
        ev[k][0].record(stream)
        for j, (_, f) in enumerate(parts):
            f(0)
            ev[k][j + 1].record(stream)
    torch.cuda.synchronize(dev)
    t_wall = time.perf_counter() - t_wall
    barrier(pg, dev)
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    step_ms = [ev[k][0].elapsed_time(ev[k][-1]) for k in range(args.steps)]
    part_ms = {name: statistics.mean(ev[k][j].elapsed_time(ev[k][j + 1]) for k in range(args.steps))
               for j, (name, _) in enumerate(parts)}
    ms_max = allreduce_max(pg, statistics.mean(step_ms), dev)
    has_ext = w["extend_flops"] > 0 and "extend" in part_ms
    has_dec = w["decode_kv_bytes"] > 0 and "decode" in part_ms
    pdesc = {}
    if "store" in part_ms:
        a = w["store_bytes"] / (part_ms["store"] * 1e-3) / 1e9
        pdesc["store"] = {"ms": part_ms["store"], "GB/s": a, "frac_hbm": a / peaks["hbm_gbs"],
                          "frac_hbm_nominal": a / NOMINAL_HBM_GBS, "bytes": w["store_bytes"]}
    if has_ext:
        a = w["extend_flops"] / (part_ms["extend"] * 1e-3) / 1e12
        pdesc["extend"] = {"ms": part_ms["extend"], "TFLOP/s": a,
                           "frac_bf16": a / peaks["bf16_tflops"],
                           "frac_bf16_sustained": a / peaks.get("bf16_tflops_sustained",
                                                                peaks["bf16_tflops"]),
                           "frac_bf16_nominal": a / NOMINAL_BF16_TFLOPS,
                           "flops": w["extend_flops"]}
    if has_dec:
        a = w["decode_kv_bytes"] / (part_ms["decode"] * 1e-3) / 1e9
        pdesc["decode"] = {"ms": part_ms["decode"], "GB/s": a, "frac_hbm": a / peaks["hbm_gbs"],
                           "frac_hbm_nominal": a / NOMINAL_HBM_GBS,
                           "unique_kv_bytes": w["decode_kv_bytes"],
                           # what the plan's kernels read (a prefix read for two member tiles of
                           # a group counts twice): the kernel's own bandwidth is plan bytes / ms
                           "plan_kv_bytes": float(dw.steps[0].dec_plan.key_reads())
                           * wl.head_dim * 2 * 2}
    # kernels of ours per step, as the plans report them
    st0 = dw.steps[0]
    per = {"store": int(wl.steps[0].store_slots.shape[0] > 0),
           "extend": st0.ext_plan.launches() if st0.ext_plan is not None else 0,
           "decode": st0.dec_plan.launches() if st0.dec_plan is not None else 0}
    return {"ms_max": ms_max, "part_ms": part_ms, "parts": pdesc, "clocks": clk, "wall": t_wall,
            "has_ext": has_ext, "has_dec": has_dec,
            "launches_per_step": sum(per[n] for n, _ in parts)}


def run_e2e(wl, dw, dev, args, pg, world, w, unit, scale, has_ext):
    """Same step through the public API with host buffers, as a serving loop runs it: per step the
    host radix match of the extend requests, plan builds + uploads, H2D of the step's inputs from
    pinned memory, the three calls, D2H of O and LSE.  Steps are pipelined over two buffer sets and
    three streams (H2D, kernels, D2H), so step k+1's inputs travel while step k computes; every
    step's copies are inside the timed region (wall clock over all steps, synchronize at the end)."""
    import torch
    from prefix_shared_kv_gb300 import rx
    from prefix_shared_kv_gb300.session import workspace

    st = wl.steps[0]
    ds = dw.steps[0]
    SETS = 2
    pin = lambda t: t.cpu().pin_memory()
    h_in = {"slots": pin(ds.slots), "k_new": pin(ds.k_new), "v_new": pin(ds.v_new)}
    if ds.ext_q is not None:
        h_in["ext_q"] = pin(ds.ext_q)
    if ds.dec_q is not None:
        h_in["dec_q"] = pin(ds.dec_q)
    outs = {}
    if ds.ext_o is not None:
        outs.update(ext_o=ds.ext_o, ext_lse=ds.ext_lse)
    if ds.dec_o is not None:
        outs.update(dec_o=ds.dec_o, dec_lse=ds.dec_lse)
    d_in = [{k: torch.empty_like(v, device=dev) for k, v in h_in.items()} for _ in range(SETS)]
    d_out = [{k: torch.empty_like(v) for k, v in outs.items()} for _ in range(SETS)]
    h_out = [{k: torch.empty_like(v, device="cpu").pin_memory() for k, v in outs.items()}
             for _ in range(SETS)]
    tree = rx.Radix()
    for toks, slots in wl.cached_sequences:
        tree.insert(toks, slots)
    eplan = [rx.Plan() for _ in range(SETS)]
    dplan = [rx.Plan() for _ in range(SETS)]
    ews = dws = None
    if st.extend is not None:
        e = st.extend
        rx.extend_plan(eplan[0], dw.desc, e.req_idx, e.prefix_len, e.extend_len, e.group_of_req,
                       e.group_prefix_len, e.group_parent)
        ews = [workspace(eplan[0].workspace_size(), dev) for _ in range(SETS)]
        # the cache hit of every extend request must be the prefix the workload cached
        for r, toks in enumerate(e.tokens):
            assert tree.match(toks, 1, want_slots=False) == int(e.prefix_len[r])
    if st.decode is not None:
        dc = st.decode
        rx.decode_plan(dplan[0], dw.desc, dc.req_idx, dc.seq_len, dc.group_of_req,
                       dc.group_prefix_len, dc.group_parent)
        dws = [workspace(dplan[0].workspace_size(), dev) for _ in range(SETS)]
    h2d = sum(v.numel() * v.element_size() for v in h_in.values())
    d2h = sum(v.numel() * v.element_size() for v in outs.values())
    s_in, s_cmp, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    ev_in = [torch.cuda.Event() for _ in range(SETS)]
    ev_cmp = [torch.cuda.Event() for _ in range(SETS)]
    ev_out = [torch.cuda.Event() for _ in range(SETS)]
    issued = [False] * SETS

    def one(i):
        b = i % SETS
        # host side of the step: a2 prefix match of the extend requests, then the plans
        if st.extend is not None:
            e = st.extend
            pl = np.fromiter((tree.match(t, 1, want_slots=False) for t in e.tokens), np.int32,
                             count=len(e.tokens))
            rx.extend_plan(eplan[b], dw.desc, e.req_idx, pl, e.extend_len, e.group_of_req,
                           e.group_prefix_len, e.group_parent)
        if st.decode is not None:
            dc = st.decode
            rx.decode_plan(dplan[b], dw.desc, dc.req_idx, dc.seq_len, dc.group_of_req,
                           dc.group_prefix_len, dc.group_parent)
        # H2D into set b once the kernels of the step that last used it are done: the plans first,
        # then the inputs, all on the input stream (a plan upload queued on the kernel stream would
        # wait behind the next step's input copy on the same copy engine)
        if issued[b]:
            s_in.wait_event(ev_cmp[b])
        if st.extend is not None:
            eplan[b].upload(ews[b], stream=s_in)
        if st.decode is not None:
            dplan[b].upload(dws[b], stream=s_in)
        with torch.cuda.stream(s_in):
            for k in h_in:
                d_in[b][k].copy_(h_in[k], non_blocking=True)
        ev_in[b].record(s_in)
        # kernels: after the inputs landed and the previous D2H of set b's outputs finished
        s_cmp.wait_event(ev_in[b])
        if issued[b]:
            s_cmp.wait_event(ev_out[b])
        rx.store_kv(dw.desc, dw.k_pool, dw.v_pool, d_in[b]["k_new"], d_in[b]["v_new"],
                    d_in[b]["slots"], stream=s_cmp)
        if st.extend is not None:
            rx.extend_attn(eplan[b], dw.desc, dw.k_pool, dw.v_pool, d_in[b]["ext_q"],
                           d_out[b]["ext_o"], d_out[b]["ext_lse"], ews[b], stream=s_cmp)
        if st.decode is not None:
            rx.decode_attn(dplan[b], dw.desc, dw.k_pool, dw.v_pool, d_in[b]["dec_q"],
                           d_out[b]["dec_o"], d_out[b]["dec_lse"], dws[b], stream=s_cmp)
        ev_cmp[b].record(s_cmp)
        # D2H of the step's results
        s_out.wait_event(ev_cmp[b])
        with torch.cuda.stream(s_out):
            for k in outs:
                h_out[b][k].copy_(d_out[b][k], non_blocking=True)
        ev_out[b].record(s_out)
        issued[b] = True

    for i in range(max(3, args.warmup)):
        one(i)
    torch.cuda.synchronize(dev)
    barrier(pg, dev)
    t0 = time.perf_counter()
    for i in range(args.steps):
        one(i)
    torch.cuda.synchronize(dev)
    ms_total = (time.perf_counter() - t0) * 1e3
    barrier(pg, dev)
    ms = allreduce_max(pg, ms_total / max(1, args.steps), dev)
    units = w["extend_flops"] if has_ext else w["decode_kv_bytes"]
    return {"value": world * units / (ms * 1e-3) / scale, "unit": unit, "ms_per_step": ms,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "note": "per step: host radix match, plan builds + uploads, H2D, kernels, D2H; steps "
                    "pipelined over two buffer sets and three streams"}


if __name__ == "__main__":
    sys.exit(main())
