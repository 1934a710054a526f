#!/usr/bin/env python
"""Benchmark of the tile-centric communication-overlapped GEMM path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step = one fused AllGather+GEMM call (the mover, per-chunk signals and the
rank-swizzled persistent tcgen05 GEMM: every row of the AG+GEMM hot path) on the
Llama-70B-MLP-like workload: W=8 emulated ranks, A_r 1024x8192, B 8192x3584 bf16
(481.0 GFLOP).  Inputs are seeded synthetic data resident in HBM; L2 is flushed
(a 256 MiB write) between timed steps, outside the timed events.  Each step is
timed with CUDA events on the launching stream; K steps are bracketed by a
barrier and a device synchronise; the max over ranks is reported.  Under
torchrun (N > 1) every rank runs an independent replica (the path is one GPU's
work; there is no data-path collective), so scaling is weak.

The JSON line also carries the other workloads of the path (tiny AG+GEMM,
GEMM+ReduceScatter, the MLP chain, the MoE layer) measured the same way, the
overlap efficiency of the AG+GEMM fusion, the roofline of the dominant kernel,
an end-to-end number through host buffers, SM clocks sampled during the timed
region, and the CPU oracle timed on a bounded sample of the same workload.

--impl reference times the fp64 CPU oracle itself (the only reference this
path has) on bounded samples of the same workload and prints the same line
with "impl": "reference"; under torchrun only rank 0 runs it.
"""
from __future__ import annotations

import argparse
import glob
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "ag_70b"
METRIC = "fused AG+GEMM / GEMM+RS TFLOP/s on 1 GB300 (W emulated ranks); % BF16 peak"
UNIT = "TFLOP/s"
L2_FLUSH_BYTES = 256 << 20  # > 129 MB L2
MOE_LAUNCHES = 3  # routing, permutation, the persistent expert-GEMM + combine kernel

# DRAM bytes per launch of the dominant kernel from ncu (dram__bytes_read.sum +
# dram__bytes_write.sum), keyed by the hash of the kernel's sources (AG_KERNEL_SOURCES) they
# were taken on.
# A kernel changed since the capture reports traffic null.
NCU_TRAFFIC = {"ag_70b": {"fe1bb8d7778bd175": 587978240,   # profiles/ag_70b_persistent_kernel_ncu.md
                           "33004dd266fe890c": 587501056,   # its traffic re-captures
                           "c63981ffce7b1bcf": 612093952,
                           "06013d50fb65ebef": 612273152,
                           "abcbff1dabca23fc": 612214528},
               # GEMM+RS, owner-slot chain and ring order, captured back to back on one box
               # (profiles/rs_70b_ring_persistent_kernel_pair_ncu.md)
               "rs_70b": {"c63981ffce7b1bcf": 5608278016, "06013d50fb65ebef": 5641131520,
                          "abcbff1dabca23fc": 5573654528},
               "rs_70b_ring": {"c63981ffce7b1bcf": 8656728064, "06013d50fb65ebef": 7760482816,
                               "abcbff1dabca23fc": 9909475584}}


# The sources the AllGather+GEMM kernel is compiled from: its translation unit and every
# header it includes (the ABI header too).
AG_KERNEL_SOURCES = ["communication_overlapped_gemm_gb300/csrc/tl_gemm_ops.cu",
                     "communication_overlapped_gemm_gb300/csrc/tl_engine.cuh",
                     "communication_overlapped_gemm_gb300/csrc/tl_engine2.cuh",
                     "communication_overlapped_gemm_gb300/csrc/tl_ptx.cuh",
                     "communication_overlapped_gemm_gb300/csrc/tl_sched.h",
                     "communication_overlapped_gemm_gb300/csrc/tl_host.h",
                     "include/tl.h"]


def _code_only(text: str) -> str:
    """C/C++/CUDA source without its comments and with whitespace runs collapsed: a change of
    documentation does not change the code a profile was taken of.  (String literals in these
    sources hold no comment markers.)"""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def src_hash(files=None) -> str:
    """Hash of the code (comments stripped) of the given source files (paths from the
    repository root), by default of every file of the CUDA sources."""
    if files is None:
        paths = sorted(glob.glob(os.path.join(ROOT, "communication_overlapped_gemm_gb300", "csrc", "*")))
    else:
        paths = [os.path.join(ROOT, f) for f in sorted(files)]
    h = hashlib.sha256()
    for f in paths:
        with open(f, encoding="utf-8") as fh:
            h.update(os.path.basename(f).encode())
            h.update(_code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return dict(hbm=float(d["hbm_gbs"]), bf16=float(d["bf16_tflops"]),
                    bf16_sus=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), src="measured")
    except Exception:
        return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, src="fallback")


# ----------------------------------------------------------------------------- distributed
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def init_dist(world, backend):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist if world > 1 else None


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(dist, x: float, device=None) -> float:
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clock / throttle-reason samples taken while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.out = None

    def start(self):
        try:
            self.out = open(os.devnull, "w") if False else None
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return dict(sm_mhz=None, sm_max_mhz=None, reasons=["clock sampling unavailable"], samples=0)
        time.sleep(0.15)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        sm, smax, reasons, n = [], [], set(), 0
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            n += 1
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return dict(sm_mhz=statistics.median(sm) if sm else None, sm_max_mhz=max(smax) if smax else None,
                    reasons=sorted(reasons), samples=n)


def gpu_id_for(device: int) -> str:
    import torch
    try:
        u = str(torch.cuda.get_device_properties(device).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        if vis:
            return vis.split(",")[device]
        return str(device)


# ----------------------------------------------------------------------------- helpers
def dev_bf16(bits, device):
    import numpy as np
    import torch
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.to(device)


def pinned_bf16(bits):
    import numpy as np
    import torch
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.pin_memory()


def timed_steps(fn, steps, flush, stream):
    """Per-step CUDA-event times (ms) on `stream`, L2 flushed before each step (outside the events)."""
    import torch
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for e0, e1 in evs:
        flush.zero_()
        e0.record(stream)
        fn()
        e1.record(stream)
    torch.cuda.synchronize()
    return [e0.elapsed_time(e1) for e0, e1 in evs]


def ag_flops(W, mpr, n, k):
    return 2.0 * W * mpr * n * k


# ----------------------------------------------------------------------------- our arm
def run_ours(args):
    import numpy as np
    import torch

    import __graft_entry__ as ge
    ge.build()
    import communication_overlapped_gemm_gb300 as tl
    from seeded_inputs import WORKLOADS, workload_inputs

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist = init_dist(world, "nccl")
    pk = peaks()
    stream = torch.cuda.current_stream()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    ctx = tl.Context(local)

    d = WORKLOADS[WORKLOAD].dims
    W, mpr, n, k = d["W"], d["m_per_rank"], d["n"], d["k"]
    inp = workload_inputs(WORKLOAD)
    a = [dev_bf16(x, device) for x in inp["a_shards"]]
    b = dev_bf16(inp["b"], device)
    c = torch.empty((W * mpr, n), dtype=torch.bfloat16, device=device)
    ws = torch.zeros(tl.tl_ag_gemm_workspace_bytes(W, mpr, n, k), dtype=torch.uint8, device=device)
    flops = ag_flops(W, mpr, n, k)

    def step():
        tl.tl_ag_gemm(ctx, a, b, c, ws, rank=0, stream=stream)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    if ctx.check() != tl.TL_OK:
        raise RuntimeError("device status not OK after warm-up")

    sampler = ClockSampler(gpu_id_for(local))
    barrier(dist)
    torch.cuda.synchronize()
    sampler.start()
    times = timed_steps(step, args.steps, flush, stream)
    torch.cuda.synchronize()
    barrier(dist)
    clocks = sampler.stop()
    if ctx.check() != tl.TL_OK:
        raise RuntimeError("device status not OK after the timed steps")
    total_ms = max_over_ranks(dist, sum(times), device)
    value = flops * args.steps * world / (total_ms * 1e-3) / 1e12
    launch_ms = statistics.mean(times)
    achieved = flops / (launch_ms * 1e-3) / 1e12
    h = src_hash(AG_KERNEL_SOURCES)
    traffic = NCU_TRAFFIC.get(WORKLOAD, {}).get(h)

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD, "W": W, "m_per_rank": mpr, "n": n, "k": k, "rank": 0,
                   "parallelism": f"replicas x{world} (each GPU runs the W={W} emulated-rank workload)",
                   "l2": "flushed between timed steps (256 MiB write outside the events)"},
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": pk["bf16"], "unit": "TFLOP/s",
                     "frac": round(achieved / pk["bf16"], 4), "traffic": traffic,
                     "peak_src": f"bf16 burst, {pk['src']} (MEASURED_PEAKS.json)" if pk["src"] == "measured"
                     else "bf16 burst, fallback 1.9 PFLOP/s",
                     "kernel": "tl::persistent_kernel<tl::AgOp>", "algorithmic": f"{flops/1e9:.1f} GFLOP per launch",
                     "src_hash": h},
        "gpu_launches": args.steps,
        "clocks": clocks,
    }

    if not args.quick:
        line["overlap"] = overlap_ag(tl, ctx, a, b, c, ws, flush, stream, device, times, W, mpr, n, k, pk)
        line["workloads"] = sub_workloads(tl, ctx, flush, stream, device, pk, args)
        line["e2e"] = e2e_ag(tl, ctx, inp, device, stream, W, mpr, n, k, args)
        line["baselines"] = {"cublas_plus_copy_ms": cublas_plus_copy(a, b, flush, stream, device)}
    if rank == 0 and not args.no_cpu:
        line["cpu_baseline"] = cpu_baseline_ag(inp, args.cpu_seconds)
        line["cpu_baseline"]["single_thread"] = cpu_single_thread_ag(args.cpu_seconds / 2)
    ctx.close()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


def overlap_ag(tl, ctx, a, b, c, ws, flush, stream, device, fused_times, W, mpr, n, k, pk):
    """(t_copy_alone + t_gemm_alone - t_fused) / min(t_copy_alone, t_gemm_alone)."""
    import torch
    reps = 30
    # communication alone: the same mover, standalone
    for _ in range(3):
        tl.tl_allgather(ctx, a, ws, rank=0, stream=stream)
    t_copy = statistics.median(timed_steps(lambda: tl.tl_allgather(ctx, a, ws, rank=0, stream=stream), reps,
                                           flush, stream))
    # the same AllGather on the TMA units (bulk copies, one thread per SM): the copy-engine mover
    with tl.Context(ctx.device, mover_tma=1) as ct:
        for _ in range(3):
            tl.tl_allgather(ct, a, ws, rank=0, stream=stream)
        t_copy_tma = statistics.median(timed_steps(lambda: tl.tl_allgather(ct, a, ws, rank=0, stream=stream), reps,
                                                   flush, stream))
        if ct.check() != tl.TL_OK:
            raise RuntimeError("tl_allgather (mover_tma): device status not OK")
    # GEMM alone: the same engine on the already-gathered operand (W = 1, no signals)
    gath = ws[: W * mpr * k * 2].view(torch.bfloat16).view(W * mpr, k)
    ws1 = torch.zeros(tl.tl_ag_gemm_workspace_bytes(1, W * mpr, n, k), dtype=torch.uint8, device=device)
    g = lambda: tl.tl_ag_gemm(ctx, [gath], b, c, ws1, rank=0, stream=stream)
    for _ in range(3):
        g()
    t_gemm = statistics.median(timed_steps(g, reps, flush, stream))
    t_fused = statistics.median(fused_times)
    moved = 2.0 * (W - 1 + 1) * mpr * k * 2  # bytes read + written by the mover (all W shards)
    return {
        "t_copy_alone_us": round(t_copy * 1e3, 2), "t_gemm_alone_us": round(t_gemm * 1e3, 2),
        "t_fused_us": round(t_fused * 1e3, 2),
        "efficiency": round((t_copy + t_gemm - t_fused) / min(t_copy, t_gemm), 4),
        "copy_alone_gbs": round(moved / (t_copy * 1e-3) / 1e9, 1),
        "copy_alone_hbm_frac": round(moved / (t_copy * 1e-3) / 1e9 / pk["hbm"], 4),
        "copy_alone_tma_us": round(t_copy_tma * 1e3, 2),
        "copy_alone_tma_hbm_frac": round(moved / (t_copy_tma * 1e-3) / 1e9 / pk["hbm"], 4),
        "gemm_alone_tflops": round(ag_flops(W, mpr, n, k) / (t_gemm * 1e-3) / 1e12, 2),
        "gemm_alone_frac": round(ag_flops(W, mpr, n, k) / (t_gemm * 1e-3) / 1e12 / pk["bf16"], 4),
    }


def cublas_plus_copy(a, b, flush, stream, device):
    """Non-overlapped context baseline: serial gather (torch.cat) then cuBLAS (torch.matmul)."""
    import torch
    f = lambda: torch.matmul(torch.cat(a, dim=0), b)
    for _ in range(3):
        f()
    return round(statistics.median(timed_steps(f, 20, flush, stream)), 5)


def sub_workloads(tl, ctx, flush, stream, device, pk, args):
    import torch
    from seeded_inputs import WORKLOADS, workload_inputs
    out = {}
    reps = args.sub_steps

    def gemm_alone(r, fn, flops):
        for _ in range(2):
            fn()
        torch.cuda.synchronize()
        if ctx.check() != tl.TL_OK:
            raise RuntimeError("plain GEMMs: device status not OK")
        t = statistics.median(timed_steps(fn, max(3, reps // 2), flush, stream))
        r["gemm_alone_us"] = round(t * 1e3, 2)
        r["gemm_alone_tflops"] = round(flops / (t * 1e-3) / 1e12, 2)
        r["fused_over_gemm_alone"] = round(r["us"] / (t * 1e3), 4)

    def rs_alone(r, fn, nbytes, extra=None):
        """t_copy_alone of a fused GEMM+RS: its communication (and, for the MLP chain, its
        AllGathers) alone; with t_gemm_alone and t_fused gives the overlap efficiency
        (t_copy + t_gemm - t_fused) / min(t_copy, t_gemm)."""
        for _ in range(2):
            fn()
        torch.cuda.synchronize()
        if ctx.check() != tl.TL_OK:
            raise RuntimeError("communication alone: device status not OK")
        t = statistics.median(timed_steps(fn, max(5, reps), flush, stream))
        tg, tf = r["gemm_alone_us"] * 1e-3, r["us"] * 1e-3
        r["copy_alone_us"] = round(t * 1e3, 2)
        r["copy_alone_gbs"] = round(nbytes / (t * 1e-3) / 1e9, 1)
        r["copy_alone_hbm_frac"] = round(nbytes / (t * 1e-3) / 1e9 / pk["hbm"], 4)
        r["overlap_efficiency"] = round((t + tg - tf) / min(t, tg), 4)
        if extra:
            r["copy_alone"] = extra

    def cublas_leg(r, fn, flops):
        """Context: the same products through cuBLAS (torch.matmul into preallocated bf16
        outputs), timed like the fused call: the library GEMM under the same tensor load."""
        for _ in range(2):
            fn()
        torch.cuda.synchronize()
        t = statistics.median(timed_steps(fn, max(3, reps // 2), flush, stream))
        r["cublas_gemms_us"] = round(t * 1e3, 2)
        r["cublas_gemms_tflops"] = round(flops / (t * 1e-3) / 1e12, 2)
        r["fused_over_cublas_gemms"] = round(r["us"] / (t * 1e3), 4)

    def rec(name, fn, flops, bytes_alg, bound, launches):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        if ctx.check() != tl.TL_OK:
            raise RuntimeError(f"{name}: device status not OK")
        t = statistics.median(timed_steps(fn, reps, flush, stream))
        tf = flops / (t * 1e-3) / 1e12
        gbs = bytes_alg / (t * 1e-3) / 1e9
        r = {"us": round(t * 1e3, 2), "tflops": round(tf, 2), "gpu_launches_per_call": launches,
             "bound": bound}
        if bound == "tensor":
            r["frac"] = round(tf / pk["bf16"], 4)
        else:
            r["hbm_gbs"] = round(gbs, 1)
            r["frac"] = round(gbs / pk["hbm"], 4)
            r["tensor_frac"] = round(tf / pk["bf16"], 4)
        out[name] = r

    # tiny AG+GEMM
    d = WORKLOADS["ag_tiny"].dims
    inp = workload_inputs("ag_tiny")
    a = [dev_bf16(x, device) for x in inp["a_shards"]]
    b = dev_bf16(inp["b"], device)
    c = torch.empty((d["W"] * d["m_per_rank"], d["n"]), dtype=torch.bfloat16, device=device)
    ws = torch.zeros(tl.tl_ag_gemm_workspace_bytes(d["W"], d["m_per_rank"], d["n"], d["k"]), dtype=torch.uint8,
                     device=device)
    rec("ag_tiny", lambda: tl.tl_ag_gemm(ctx, a, b, c, ws, stream=stream),
        ag_flops(d["W"], d["m_per_rank"], d["n"], d["k"]), 0, "latency", 1)
    out["ag_tiny"]["gather"] = "pull: mover chunks, one release signal each"
    # the same call with the low-latency push gather (LL words carry the call's signal)
    with tl.Context(ctx.device, ag_ll=1) as cl:
        rec("ag_tiny_ll", lambda: tl.tl_ag_gemm(cl, a, b, c, ws, stream=stream),
            ag_flops(d["W"], d["m_per_rank"], d["n"], d["k"]), 0, "latency", 1)
        if cl.check() != tl.TL_OK:
            raise RuntimeError("ag_tiny_ll: device status not OK")
        out["ag_tiny_ll"]["gather"] = "low-latency push: flag-in-payload LL words, no separate signal"
    del a, b, c, ws

    # GEMM + ReduceScatter
    d = WORKLOADS["rs_70b"].dims
    inp = workload_inputs("rs_70b")
    a = [dev_bf16(x, device) for x in inp["a"]]
    b = [dev_bf16(x, device) for x in inp["b"]]
    W, m, n, kr = d["W"], d["m"], d["n"], d["k_r"]
    o = [torch.empty((m // W, n), dtype=torch.bfloat16, device=device) for _ in range(W)]
    ws = torch.zeros(tl.tl_gemm_rs_workspace_bytes(W, m, n, kr), dtype=torch.uint8, device=device)
    rec("rs_70b", lambda: tl.tl_gemm_rs(ctx, a, b, o, ws, stream=stream), 2.0 * W * m * n * kr, 0, "tensor", 1)
    # the same W products with a plain bf16 store (the AG engine with nothing to gather)
    cp = torch.empty((m, n), dtype=torch.bfloat16, device=device)
    ws1 = torch.zeros(tl.tl_ag_gemm_workspace_bytes(1, m, n, kr), dtype=torch.uint8, device=device)
    gemm_alone(out["rs_70b"], lambda: [tl.tl_ag_gemm(ctx, [a[p]], b[p], cp, ws1, stream=stream) for p in range(W)],
               2.0 * W * m * n * kr)
    del ws1
    cublas_leg(out["rs_70b"], lambda: [torch.matmul(a[p], b[p], out=cp) for p in range(W)], 2.0 * W * m * n * kr)
    del cp
    # the communication alone: the ReduceScatter of the W ranks' fp32 partials (m x n each)
    parts = [torch.randn((m, n), dtype=torch.float32, device=device) for _ in range(W)]
    rs_alone(out["rs_70b"], lambda: tl.tl_reduce_scatter(ctx, parts, o, stream=stream), W * m * n * 4 + m * n * 2)
    del ws
    # the ring reduction ([TL] §5): the same products, partials passed rank to rank
    with tl.Context(ctx.device, rs_ring=1) as cr:
        wsr = torch.zeros(tl.tl_gemm_rs_ring_workspace_bytes(W, m, n, kr), dtype=torch.uint8, device=device)
        rec("rs_70b_ring", lambda: tl.tl_gemm_rs(cr, a, b, o, wsr, stream=stream), 2.0 * W * m * n * kr, 0, "tensor", 1)
        if cr.check() != tl.TL_OK:
            raise RuntimeError("rs_70b_ring: device status not OK")
        del wsr
    for key in ("gemm_alone_us", "gemm_alone_tflops"):
        out["rs_70b_ring"][key] = out["rs_70b"][key]
    h = src_hash(AG_KERNEL_SOURCES)
    for key in ("rs_70b", "rs_70b_ring"):
        out[key]["ncu_dram_bytes"] = NCU_TRAFFIC[key].get(h)  # null once the kernel changed
    out["rs_70b_ring"]["fused_over_gemm_alone"] = round(out["rs_70b_ring"]["us"] / out["rs_70b"]["gemm_alone_us"], 4)
    rs_alone(out["rs_70b_ring"], lambda: tl.tl_reduce_scatter(ctx, parts, o, stream=stream), W * m * n * 4 + m * n * 2)
    del parts
    oracle_time(out["rs_70b"], "rs_70b", inp, args)
    del a, b, o

    # MLP chain
    d = WORKLOADS["mlp2_8b"].dims
    inp = workload_inputs("mlp2_8b")
    W, T, hdim, f = d["W"], d["tokens"], d["hidden"], d["f_r"]
    x = [dev_bf16(v, device) for v in inp["x_shards"]]
    w1 = [dev_bf16(v, device) for v in inp["w1"]]
    w2 = [dev_bf16(v, device) for v in inp["w2"]]
    o = [torch.empty((T // W, hdim), dtype=torch.bfloat16, device=device) for _ in range(W)]
    ws = torch.zeros(tl.tl_mlp2_workspace_bytes(W, T, hdim, f), dtype=torch.uint8, device=device)
    rec("mlp2_8b", lambda: tl.tl_mlp2(ctx, x, w1, w2, o, ws, stream=stream), 2.0 * W * T * hdim * f * 2, 0,
        "tensor", 1)
    # the same 2 W products as plain GEMMs (no gather, GELU, chaining or reduction)
    xg = torch.cat(x, dim=0)
    hbuf = torch.empty((T, f), dtype=torch.bfloat16, device=device)
    ybuf = torch.empty((T, hdim), dtype=torch.bfloat16, device=device)
    ws1 = torch.zeros(max(tl.tl_ag_gemm_workspace_bytes(1, T, f, hdim), tl.tl_ag_gemm_workspace_bytes(1, T, hdim, f)),
                      dtype=torch.uint8, device=device)

    def mlp_plain():
        for r in range(W):
            tl.tl_ag_gemm(ctx, [xg], w1[r], hbuf, ws1, stream=stream)
            tl.tl_ag_gemm(ctx, [hbuf], w2[r], ybuf, ws1, stream=stream)
    gemm_alone(out["mlp2_8b"], mlp_plain, 2.0 * W * T * hdim * f * 2)

    def mlp_cublas():
        for r in range(W):
            torch.matmul(xg, w1[r], out=hbuf)
            torch.matmul(hbuf, w2[r], out=ybuf)
    cublas_leg(out["mlp2_8b"], mlp_cublas, 2.0 * W * T * hdim * f * 2)
    del xg, hbuf, ybuf, ws1
    # the communication alone: every rank's AllGather of X, then the ReduceScatter of the W
    # ranks' fp32 layer-2 partials (T x hidden each)
    ws_ag = torch.zeros(tl.tl_ag_gemm_workspace_bytes(W, T // W, 8, hdim), dtype=torch.uint8, device=device)
    parts = [torch.randn((T, hdim), dtype=torch.float32, device=device) for _ in range(W)]

    def mlp_comm():
        for r in range(W):
            tl.tl_allgather(ctx, x, ws_ag, rank=r, stream=stream)
        tl.tl_reduce_scatter(ctx, parts, o, stream=stream)
    rs_alone(out["mlp2_8b"], mlp_comm, W * 2 * T * hdim * 2 + W * T * hdim * 4 + T * hdim * 2,
             f"{W} AllGathers of X (tl_allgather, rank r each) + tl_reduce_scatter of {W} fp32 partials")
    # the same chain with the push-mode AllGather ([TD] §3.2 Algorithm 1)
    with tl.Context(ctx.device, ag_push=1) as cp_:
        rec("mlp2_8b_push", lambda: tl.tl_mlp2(cp_, x, w1, w2, o, ws, stream=stream), 2.0 * W * T * hdim * f * 2, 0,
            "tensor", 1)
        if cp_.check() != tl.TL_OK:
            raise RuntimeError("mlp2_8b_push: device status not OK")
    del ws_ag, parts
    oracle_time(out["mlp2_8b"], "mlp2_8b", inp, args)
    del x, w1, w2, o, ws

    # MoE layer
    d = WORKLOADS["moe_64e"].dims
    inp = workload_inputs("moe_64e")
    T, H, E, F, kk = d["T"], d["H"], d["E"], d["F"], d["topk"]
    xx = dev_bf16(inp["x"], device)
    lg = torch.from_numpy(inp["logits"]).to(device)
    wg, wu, wd = (dev_bf16(inp[q], device) for q in ("w_gate", "w_up", "w_down"))
    oo = torch.empty((T, H), dtype=torch.float32, device=device)
    ws = torch.zeros(tl.tl_moe_workspace_bytes(T, H, E, F, kk), dtype=torch.uint8, device=device)
    moe_flops = 2.0 * T * kk * H * F * 3
    # algorithmic bytes: the expert weights, x, logits and out once; the intermediates the
    # layer materialises (the gathered rows Xp, h and y, all bf16) written once and read once
    moe_bytes = 3.0 * E * H * F * 2 + T * H * 2 + T * E * 4 + T * H * 4 + 2.0 * T * kk * (H * 2 + F * 2 + H * 2)
    rec("moe_64e", lambda: tl.tl_moe_combine(ctx, xx, lg, kk, wg, wu, wd, oo, ws, stream=stream), moe_flops,
        moe_bytes, "hbm", MOE_LAUNCHES)
    out["moe_64e"]["combine_sms"] = ctx.config.combine_ctas  # the workload as stated: 8 reserved SMs
    # the same layer with a 16-SM combine partition, for comparison
    with tl.Context(ctx.device, combine_ctas=16) as c16:
        rec("moe_64e_16sm", lambda: tl.tl_moe_combine(c16, xx, lg, kk, wg, wu, wd, oo, ws, stream=stream), moe_flops,
            moe_bytes, "hbm", MOE_LAUNCHES)
        if c16.check() != tl.TL_OK:
            raise RuntimeError("moe_64e_16sm: device status not OK")
    out["moe_64e_16sm"]["combine_sms"] = 16
    oracle_time(out["moe_64e"], "moe_64e", inp, args)
    del xx, lg, wg, wu, wd, oo, ws

    # AllGather KV + self-attention (Attn-1 at 16k on 8 ranks)
    d = WORKLOADS["attn_16k"].dims
    inp = workload_inputs("attn_16k")
    W, Hh, L, hd = d["W"], d["heads"], d["l_r"], d["d"]
    q = dev_bf16(inp["q"], device)
    ks = [dev_bf16(x, device) for x in inp["k_shards"]]
    vs = [dev_bf16(x, device) for x in inp["v_shards"]]
    ao = torch.empty((Hh, L, hd), dtype=torch.bfloat16, device=device)
    ws = torch.zeros(tl.tl_ag_attention_workspace_bytes(W, Hh, L, hd), dtype=torch.uint8, device=device)
    rec("attn_16k", lambda: tl.tl_ag_attention(ctx, q, ks, vs, ao, ws, stream=stream), 4.0 * L * W * L * hd * Hh, 0,
        "tensor", 1)
    oracle_time(out["attn_16k"], "attn_16k", inp, args)
    return out


def e2e_ag(tl, ctx, inp, device, stream, W, mpr, n, k, args):
    """Same metric through the public API with host buffers: every step copies its inputs
    from pinned memory to the device, makes the call and reads the result back to pinned
    memory, all inside the timed region.  As a serving loop would, the device inputs and
    outputs are double-buffered and the three stages run on their own streams, ordered by
    events: step i+1's host-to-device copies overlap step i's call and device-to-host copy
    (the call itself waits for nothing but its own inputs)."""
    import torch
    ha = [pinned_bf16(x) for x in inp["a_shards"]]
    hb = pinned_bf16(inp["b"])
    hc = torch.empty((W * mpr, n), dtype=torch.bfloat16).pin_memory()
    a = [[torch.empty_like(x, device=device) for x in ha] for _ in range(2)]
    b = [torch.empty_like(hb, device=device) for _ in range(2)]
    c = [torch.empty((W * mpr, n), dtype=torch.bfloat16, device=device) for _ in range(2)]
    ws = torch.zeros(tl.tl_ag_gemm_workspace_bytes(W, mpr, n, k), dtype=torch.uint8, device=device)
    s_in, s_out = torch.cuda.Stream(device), torch.cuda.Stream(device)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_call = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    issued = [0]

    def step():
        i = issued[0]
        j = i % 2
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(ev_call[j])  # the call of step i-2 has read buffer set j
            for d_, h_ in zip(a[j], ha):
                d_.copy_(h_, non_blocking=True)
            b[j].copy_(hb, non_blocking=True)
            ev_in[j].record(s_in)
        stream.wait_event(ev_in[j])
        if i >= 2:
            stream.wait_event(ev_out[j])  # the copy-back of step i-2 has read c[j]
        tl.tl_ag_gemm(ctx, a[j], b[j], c[j], ws, stream=stream)
        ev_call[j].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_call[j])
            hc.copy_(c[j], non_blocking=True)
            ev_out[j].record(s_out)
        issued[0] += 1

    for _ in range(2):
        step()
    torch.cuda.synchronize()
    steps = args.e2e_steps
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    s_in.wait_event(e0)
    s_out.wait_event(e0)
    for _ in range(steps):
        step()
    stream.wait_event(ev_out[(issued[0] - 1) % 2])  # the last step's copy-back is inside
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    h2d = sum(x.numel() * 2 for x in ha) + hb.numel() * 2
    return {"value": round(ag_flops(W, mpr, n, k) / (ms * 1e-3) / 1e12, 2), "unit": UNIT,
            "ms_per_step": round(ms, 4), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": hc.numel() * 2,
            "steps": steps,
            "pipeline": "device inputs/outputs double-buffered; H2D, call and D2H on three streams ordered by events"}


# ----------------------------------------------------------------------------- CPU oracle
def oracle_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n and n[0]:
            return int(n[0])
    except Exception:
        pass
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def oracle_ag_sample(inp, rows_per_shard, cols):
    """The oracle on a sample of the workload: the first rows of every shard, the first cols of B."""
    import oracle
    shards = [x[:rows_per_shard] for x in inp["a_shards"]]
    bs = inp["b"][:, :cols]
    t0 = time.perf_counter()
    oracle.ag_gemm(shards, bs)
    dt = time.perf_counter() - t0
    W = len(shards)
    k = inp["b"].shape[0]
    return dt, 2.0 * W * rows_per_shard * cols * k


def cpu_baseline_ag(inp, seconds):
    """The fp64 oracle, as it stands, on a bounded sample of the AG+GEMM workload.

    The sample is the first `rows` rows of every shard times all columns of B; rows
    doubles from 32 until one run takes at least a third of `seconds` or covers the
    whole workload; the last run is reported.
    """
    n_full = inp["b"].shape[1]
    mpr = inp["a_shards"][0].shape[0]
    W = len(inp["a_shards"])
    k = inp["b"].shape[0]
    rows = 32
    while True:
        dt, fl = oracle_ag_sample(inp, rows, n_full)
        if dt >= seconds / 3 or rows >= mpr:
            break
        rows = min(mpr, rows * 2)
    return {"value": round(fl / dt / 1e12, 6), "unit": UNIT, "cores": oracle_threads(), "kind": "oracle",
            "sample": f"C rows 0..{rows - 1} of each of the {W} shards x all {n_full} columns "
                      f"({fl / 1e9:.1f} GFLOP of {2.0 * W * mpr * n_full * k / 1e9:.1f}), float64 numpy",
            "seconds": round(dt, 3)}


def oracle_time(r, name, inp, args):
    """The fp64 oracle, as it stands, on a bounded sample of one workload: the sample
    doubles until one run takes a third of the budget (or covers the workload); the
    rate is scaled to the full workload's FLOPs."""
    if args.no_cpu or dist_env()[0] != 0:
        return
    import oracle
    from seeded_inputs import WORKLOADS
    d = WORKLOADS[name].dims
    budget = args.cpu_seconds / 5

    def run(n):  # -> (seconds, sample FLOPs, description, full FLOPs, n at the full workload)
        if name == "rs_70b":
            W, m, nn, kr = d["W"], d["m"], d["n"], d["k_r"]
            t0 = time.perf_counter()
            oracle.gemm_rs([x[:n] for x in inp["a"]], inp["b"])
            return (time.perf_counter() - t0, 2.0 * W * n * nn * kr, f"rows 0..{n - 1} of S (all {W} producers)",
                    2.0 * W * m * nn * kr, m)
        if name == "mlp2_8b":
            W, T, hdim, f = d["W"], d["tokens"], d["hidden"], d["f_r"]
            r = n // W
            t0 = time.perf_counter()
            oracle.mlp2([x[:r] for x in inp["x_shards"]], inp["w1"], inp["w2"])
            return (time.perf_counter() - t0, 2.0 * W * (W * r) * hdim * f * 2, f"the first {r} tokens of each shard",
                    2.0 * W * T * hdim * f * 2, T)
        if name == "moe_64e":
            T, H, F, kk = d["T"], d["H"], d["F"], d["topk"]
            t0 = time.perf_counter()
            oracle.moe(inp["x"][:n], inp["logits"][:n], inp["w_gate"], inp["w_up"], inp["w_down"], kk)
            return (time.perf_counter() - t0, 2.0 * n * kk * H * F * 3, f"tokens 0..{n - 1}", 2.0 * T * kk * H * F * 3, T)
        W, Hh, L, hd = d["W"], d["heads"], d["l_r"], d["d"]
        heads, rows = ([0], range(n)) if n <= L else (range(n // L), range(L))  # n (head, row) pairs
        t0 = time.perf_counter()
        oracle.ag_attention_rows(inp["q"], inp["k_shards"], inp["v_shards"], heads, rows)
        desc = f"head 0, query rows 0..{n - 1}" if n <= L else f"heads 0..{n // L - 1}, all {L} query rows"
        return (time.perf_counter() - t0, 4.0 * len(heads) * len(rows) * W * L * hd, desc,
                4.0 * L * W * L * hd * Hh, L * Hh)

    # Sizes double until one run takes a third of the budget; the full-workload time is
    # extrapolated from the last two runs (the per-call widening of the weights is a fixed
    # cost, the rest grows with the sample).
    n, runs = 32, []
    while True:
        dt, fl, desc, full, n_full = run(n)
        runs.append((n, dt, fl, desc))
        if (dt >= budget / 3 and len(runs) >= 2) or n >= n_full:
            break
        n = min(n_full, n * 2)
    n1, t1, fl1, desc1 = runs[-1]
    if n1 >= n_full or len(runs) < 2:
        est = t1
    else:
        n0, t0 = runs[-2][0], runs[-2][1]
        est = t1 + max(0.0, (t1 - t0) / (n1 - n0)) * (n_full - n1)
    r["cpu_oracle"] = {"tflops": round(full / est / 1e12, 6), "est_full_s": round(est, 2), "seconds": round(t1, 3),
                       "sample": f"{desc1} ({fl1 / 1e9:.2f} GFLOP of {full / 1e9:.1f}) and the run at half that size, "
                                 f"extrapolated to the full workload; float64 numpy",
                       "cores": oracle_threads()}


def cpu_single_thread_ag(seconds):
    """The headline oracle sample again, in a child process limited to one BLAS thread."""
    import subprocess
    code = ("import json, bench; from seeded_inputs import workload_inputs; inp = workload_inputs(bench.WORKLOAD); "
            f"r = bench.cpu_baseline_ag(inp, {seconds!r}); print(json.dumps(r))")
    env = dict(os.environ)
    for v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS"):
        env[v] = "1"
    try:
        p = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True, text=True,
                           timeout=max(120, 10 * seconds))
        r = json.loads(p.stdout.strip().splitlines()[-1])
        return {"value": r["value"], "unit": r["unit"], "cores": 1, "sample": r["sample"], "seconds": r["seconds"]}
    except Exception as e:  # reported, not fatal: the all-core figure stands
        return {"error": str(e)[:200]}


# ----------------------------------------------------------------------------- reference arm
def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    from seeded_inputs import WORKLOADS, workload_inputs
    d = WORKLOADS[WORKLOAD].dims
    W, mpr, n, k = d["W"], d["m_per_rank"], d["n"], d["k"]
    inp = workload_inputs(WORKLOAD)
    # Each step is one output block: the first r rows of every shard x the first c columns
    # (W*r == c), the largest such block whose oracle time fits args.ref_budget / (W + K).
    per_step = args.ref_budget / (args.warmup + args.steps)
    c = 64
    while c < n:
        dt, _ = oracle_ag_sample(inp, max(1, (2 * c) // W), 2 * c)
        if dt > per_step:
            break
        c *= 2
    c = min(c, n)
    r = max(1, c // W)
    for _ in range(args.warmup):
        oracle_ag_sample(inp, r, c)
    ts, fls = [], []
    for _ in range(args.steps):
        dt, fl = oracle_ag_sample(inp, r, c)
        ts.append(dt)
        fls.append(fl)
    total_s = sum(ts)
    value = sum(fls) / total_s / 1e12
    sample = (f"per step: C rows 0..{r - 1} of each of the {W} shards x columns 0..{c - 1} "
              f"({fls[0] / 1e9:.3f} GFLOP), float64 numpy")
    line = {
        "metric": METRIC, "value": round(value, 6), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(total_s / args.steps * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "W": W, "m_per_rank": mpr, "n": n, "k": k},
        "impl": "reference",
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": oracle_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_profile(args):
    """Run one workload's call (3 warm-up + 1) and exit: the target of an ncu capture."""
    import torch

    import __graft_entry__ as ge
    ge.build()
    import communication_overlapped_gemm_gb300 as tl
    from seeded_inputs import WORKLOADS, workload_inputs
    torch.cuda.set_device(0)
    device = torch.device("cuda", 0)
    name = args.profile
    # the communication-alone legs and the low-latency gather run on their workloads' inputs
    base = {"allgather_70b": "ag_70b", "allgather_70b_tma": "ag_70b", "reduce_scatter_70b": "rs_70b",
            "ag_tiny_ll": "ag_tiny", "rs_70b_ring": "rs_70b"}.get(name, name)
    cfg = {"ag_tiny_ll": dict(ag_ll=1), "allgather_70b_tma": dict(mover_tma=1), "rs_70b_ring": dict(rs_ring=1)}.get(name, {})
    ctx = tl.Context(0, **cfg)
    d = WORKLOADS[base].dims
    inp = workload_inputs(base) if name != "reduce_scatter_70b" else None
    if name in ("allgather_70b", "allgather_70b_tma"):
        a = [dev_bf16(x, device) for x in inp["a_shards"]]
        ws = torch.zeros(tl.tl_ag_gemm_workspace_bytes(d["W"], d["m_per_rank"], d["n"], d["k"]), dtype=torch.uint8,
                         device=device)
        call = lambda: tl.tl_allgather(ctx, a, ws)
    elif name == "reduce_scatter_70b":
        # the W fp32 partials of the GEMM+RS workload (values do not matter for the copy's profile)
        g = torch.Generator(device=device).manual_seed(5)
        parts = [torch.randn((d["m"], d["n"]), dtype=torch.float32, device=device, generator=g) for _ in range(d["W"])]
        o = [torch.empty((d["m"] // d["W"], d["n"]), dtype=torch.bfloat16, device=device) for _ in range(d["W"])]
        call = lambda: tl.tl_reduce_scatter(ctx, parts, o)
    elif WORKLOADS[base].kind == "ag_gemm":
        a = [dev_bf16(x, device) for x in inp["a_shards"]]
        b = dev_bf16(inp["b"], device)
        c = torch.empty((d["W"] * d["m_per_rank"], d["n"]), dtype=torch.bfloat16, device=device)
        ws = torch.zeros(tl.tl_ag_gemm_workspace_bytes(d["W"], d["m_per_rank"], d["n"], d["k"]), dtype=torch.uint8,
                         device=device)
        call = lambda: tl.tl_ag_gemm(ctx, a, b, c, ws)
    elif WORKLOADS[base].kind == "gemm_rs":
        a = [dev_bf16(x, device) for x in inp["a"]]
        b = [dev_bf16(x, device) for x in inp["b"]]
        o = [torch.empty((d["m"] // d["W"], d["n"]), dtype=torch.bfloat16, device=device) for _ in range(d["W"])]
        wsb = tl.tl_gemm_rs_ring_workspace_bytes if name == "rs_70b_ring" else tl.tl_gemm_rs_workspace_bytes
        ws = torch.zeros(wsb(d["W"], d["m"], d["n"], d["k_r"]), dtype=torch.uint8, device=device)
        call = lambda: tl.tl_gemm_rs(ctx, a, b, o, ws)
    elif WORKLOADS[base].kind == "mlp2":
        x = [dev_bf16(v, device) for v in inp["x_shards"]]
        w1 = [dev_bf16(v, device) for v in inp["w1"]]
        w2 = [dev_bf16(v, device) for v in inp["w2"]]
        W, T = d["W"], d["tokens"]
        o = [torch.empty((T // W, d["hidden"]), dtype=torch.bfloat16, device=device) for _ in range(W)]
        ws = torch.zeros(tl.tl_mlp2_workspace_bytes(W, T, d["hidden"], d["f_r"]), dtype=torch.uint8, device=device)
        call = lambda: tl.tl_mlp2(ctx, x, w1, w2, o, ws)
    elif WORKLOADS[base].kind == "ag_attn":
        q = dev_bf16(inp["q"], device)
        ks = [dev_bf16(x, device) for x in inp["k_shards"]]
        vs = [dev_bf16(x, device) for x in inp["v_shards"]]
        ao = torch.empty((d["heads"], d["l_r"], d["d"]), dtype=torch.bfloat16, device=device)
        ws = torch.zeros(tl.tl_ag_attention_workspace_bytes(d["W"], d["heads"], d["l_r"], d["d"]), dtype=torch.uint8,
                         device=device)
        call = lambda: tl.tl_ag_attention(ctx, q, ks, vs, ao, ws)
    else:
        xx = dev_bf16(inp["x"], device)
        lg = torch.from_numpy(inp["logits"]).to(device)
        wg, wu, wd = (dev_bf16(inp[q], device) for q in ("w_gate", "w_up", "w_down"))
        oo = torch.empty((d["T"], d["H"]), dtype=torch.float32, device=device)
        ws = torch.zeros(tl.tl_moe_workspace_bytes(d["T"], d["H"], d["E"], d["F"], d["topk"]), dtype=torch.uint8,
                         device=device)
        call = lambda: tl.tl_moe_combine(ctx, xx, lg, d["topk"], wg, wu, wd, oo, ws)
    if not args.trace:
        for _ in range(4):
            call()
        torch.cuda.synchronize()
        rc = ctx.check()
        ctx.close()
        if rc != tl.TL_OK:
            raise RuntimeError(f"device status {rc}")
        print(json.dumps({"profiled": name, "calls": 4}))
        return
    # Traced run: 3 warm-up calls, an L2 flush, then one call with the trace buffer on.
    import numpy as np

    from communication_overlapped_gemm_gb300 import trace
    for _ in range(3):
        call()
    cap = args.trace_spans
    buf = torch.zeros(tl.tl_trace_bytes(ctx.num_ctas, cap), dtype=torch.uint8, device=device)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    flush.fill_(1)
    ctx.set_trace(buf, cap)
    call()
    torch.cuda.synchronize()
    ctx.set_trace(None, cap)
    rc = ctx.check()
    ctx.close()
    if rc != tl.TL_OK:
        raise RuntimeError(f"device status {rc}")
    tr = trace.parse(buf.cpu().numpy().tobytes())
    if args.trace.endswith(".npz"):
        np.savez_compressed(args.trace, spans=tr["spans"], counts=tr["counts"], grid=tr["grid"])
    else:
        trace.to_chrome(tr, args.trace)
    print(json.dumps({"traced": name, "grid": tr["grid"], "spans": int(tr["spans"].size), "dropped": tr["dropped"],
                      "chrome_json": args.trace, "summary": trace.summary(tr)}))


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--sub-steps", type=int, default=20, help="timed calls per extra workload")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="budget of the oracle CPU baseline sample")
    ap.add_argument("--ref-budget", type=float, default=120.0, help="seconds of oracle work in --impl reference")
    ap.add_argument("--quick", action="store_true", help="headline only (no extra workloads / e2e / overlap)")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--profile", choices=["ag_tiny", "ag_tiny_ll", "ag_70b", "allgather_70b", "allgather_70b_tma", "rs_70b",
                                          "rs_70b_ring", "reduce_scatter_70b", "mlp2_8b", "moe_64e", "attn_16k"],
                    help="only run this workload's call 4 times (target of an ncu capture), no timing")
    ap.add_argument("--trace", metavar="PATH", help="with --profile: trace one call (after 3 warm-up calls and an "
                    "L2 flush) and write its per-CTA timeline to PATH: Chrome trace JSON, or the decoded spans "
                    "(numpy .npz) when PATH ends in .npz")
    ap.add_argument("--trace-spans", type=int, default=2048, help="trace buffer spans per warp")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.trace and not args.profile:
        ap.error("--trace needs --profile WORKLOAD")
    if args.profile:
        run_profile(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
