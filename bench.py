#!/usr/bin/env python
"""Benchmark of the FarSkip-Collective MoE layer stack on GB300.

Default workload: the DeepSeek-V3-shaped MoE layer, T = 65,536 tokens
(32 x 2,048 prefill), d = 7168, 256 routed experts, top-8 normalised sigmoid,
expert width 2048, one shared expert of width 2048, bf16 storage with fp32
accumulation.  One step = one pass of the whole hot path (router + top-k,
dispatch, routed grouped SwiGLU GEMMs, shared expert, combine + FarSkip
update) over the T tokens, through the library's C ABI.

Prints ONE JSON line (rank 0).  Under torchrun each rank runs its own T tokens
(data-parallel, no collective on the data path): weak scaling.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME]
                  [--impl ours|reference] [--no-cpu-baseline]

--impl reference times the CPU oracle (test infrastructure, plain C fp64) on a
bounded token sample of the same workload on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from mixture_experts_layer_expert_gb300 import configs, synth  # noqa: E402

METRIC = "MoE layer tokens/s, DeepSeek-V3 shape, 64K tokens; % of roofline (BF16/HBM)"
METRIC_FP8 = "MoE layer tokens/s, FP8 E4M3 expert GEMMs; % of roofline (FP8/HBM)"
METRIC_TRAIN = "MoE layer training tokens/s (forward keeping state + backward); % of bf16 tensor peak"
FP8_PER_BF16 = 2.0     # nominal dense tensor rate ratio (4.5 / 2.25 PFLOP/s)
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "gemm_traffic.json")
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def peaks():
    try:
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        return p, "measured"
    except Exception:
        return dict(FALLBACK), "fallback"


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms in the background."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "--query-gpu=" + self.Q, "--format=csv,noheader,nounits",
                                          "-lms", "200", "-i", str(self.index)], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return self
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, power, reasons = [], None, [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
                power.append(float(parts[3]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        load = [s for s, p in zip(sm, power) if p > 0.25 * max(power)] if power else sm
        return {"sm_mhz": statistics.median(load) if load else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(power) if power else None}


def reduce_max(values, world, device="cpu"):
    """Max over ranks of per-rank timings (the only collective; not on the data path)."""
    if world <= 1:
        return list(values)
    t = torch.tensor(values, dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return t.tolist()


def cuda_events(n):
    return [torch.cuda.Event(enable_timing=True) for _ in range(n)]


def routed_alg_bytes(cfg, T):
    """Algorithmic bytes of one routed gate/up + down launch pair: every expert's
    weights read once (all E are touched when T k >= E), X_perm read, the hidden h
    written and read once (bf16), Y_perm written; in the stored precisions (FP8:
    E4M3 weights with one fp32 scale per output channel, E4M3 X_perm)."""
    a = 4 if cfg.dtype == "f32" else 2
    rows = T * cfg.k
    if cfg.dtype == "mxfp8":     # E4M3 codes plus one scale byte per 32 elements; the hidden is stored MX
        q = 1.0 + 1.0 / 32
        return float(cfg.E * 3 * cfg.d * cfg.c * q + rows * cfg.d * q + 2 * rows * cfg.c * q + rows * cfg.d * a)
    w = 1 if cfg.dtype == "fp8" else a
    weights = cfg.E * 3 * cfg.d * cfg.c * w + (cfg.E * (2 * cfg.c + cfg.d) * 4 if cfg.dtype == "fp8" else 0)
    x_perm = rows * cfg.d * (1 if cfg.dtype == "fp8" else a)
    return float(weights + x_perm + 2 * rows * cfg.c * a + rows * cfg.d * a)


def gemm_traffic(cfg_name):
    """DRAM bytes per launch of the gate/up GEMM from the committed ncu summary,
    valid only while the kernel source is unchanged (null otherwise)."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f)
        src = os.path.join(ROOT, "mixture_experts_layer_expert_gb300", "csrc", "gemm_tc.cu")
        h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        if rec.get("gemm_tc_sha") != h:
            return None
        return rec.get("per_launch", {}).get(cfg_name)
    except Exception:
        return None


# ----------------------------------------------------------------- our arm

def run_ours(args, cfg, rank, world, local):
    from mixture_experts_layer_expert_gb300 import build, fs

    build.build()
    fs.lib()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    prob = synth.make_problem(cfg, device=dev)
    stack = fs.FarSkipStack(cfg, prob["blocks"], device=dev)
    host_blocks = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        host_blocks = [{k: synth.to_numpy(v) for k, v in b.items()} for b in prob["blocks"]]
    x = prob["x"]
    del prob
    torch.cuda.empty_cache()
    T, L = cfg.T, cfg.L
    stream = torch.cuda.current_stream()

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    # ------------------------------------------------ timed region 1: the stack
    fwd = stack.forward_overlap if args.overlap else stack.forward
    for _ in range(args.warmup):
        fwd(x)
    torch.cuda.synchronize()
    st, code = fs.fs_get_error()
    if st != 0:
        raise RuntimeError("device error word after warm-up: %d" % code)
    graph_launches = None
    if args.graph:      # one CUDA graph of the whole stack, replayed per step
        l0 = fs.fs_launch_count()
        stack.capture(x, overlap=args.overlap)
        graph_launches = fs.fs_launch_count() - l0
        for _ in range(args.warmup):
            stack.replay()
        torch.cuda.synchronize()
        fwd = lambda _x: stack.replay()
    sampler = ClockSampler(local).start() if rank == 0 else None
    time.sleep(0.3 if sampler else 0)
    barrier()
    torch.cuda.synchronize()
    l0 = fs.fs_launch_count()
    e0, e1 = cuda_events(2)
    e0.record(stream)
    for _ in range(args.steps):
        fwd(x)
    e1.record(stream)
    torch.cuda.synchronize()
    launches = (fs.fs_launch_count() - l0) // args.steps if graph_launches is None else graph_launches
    barrier()
    ms = e0.elapsed_time(e1) / args.steps

    # ------------------------- timed region 2: per-stage events (same kernels)
    stage_ms = per_stage_timing(cfg, stack, x, args.steps, stream)

    # ------------------------------------------- timed region 3: end to end
    e2e_ms, h2d, d2h = e2e_timing(cfg, stack, x, max(2, args.steps), stream, graph=args.graph)
    clocks = sampler.stop() if sampler else None
    st, code = fs.fs_get_error()
    if st != 0:
        raise RuntimeError("device error word after timing: %d" % code)

    ms, e2e_ms = reduce_max([ms, e2e_ms], world, dev)

    if rank != 0:
        return None
    pk, pk_src = peaks()
    tokens = T * world
    value = tokens / (ms / 1e3)
    # layer roofline: max(FLOPs / bf16 peak, algorithmic bytes / HBM)
    flops = cfg.flops_per_block() * L
    bytes_ = cfg.alg_bytes_per_block() * L
    t_roof = max(flops / (pk["bf16_tflops"] * 1e12), bytes_ / (pk["hbm_gbs"] * 1e9))
    # dominant kernel: the routed grouped SwiGLU GEMMs (gate/up + down); tensor-bound
    # at prefill sizes, HBM-bound (expert weight streaming) at decode sizes
    routed_flops = 6.0 * T * cfg.k * cfg.d * cfg.c
    routed_ms = stage_ms["routed"] / L
    fp8 = cfg.dtype in ("fp8", "mxfp8")
    routed_bytes = routed_alg_bytes(cfg, T)
    peak = pk["bf16_tflops_sustained"] * (FP8_PER_BF16 if fp8 else 1.0)
    hbm_bound = routed_bytes / (pk["hbm_gbs"] * 1e9) > routed_flops / (peak * 1e12)
    if hbm_bound:
        roof = {"bound": "hbm", "kernel": "grouped_gemm_kernel (routed gate/up + down, tcgen05): expert weight streaming",
                "achieved": round(routed_bytes / (routed_ms / 1e3) / 1e9, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": round(routed_bytes / (routed_ms / 1e3) / 1e9 / pk["hbm_gbs"], 4),
                "peak_kind": "HBM copy, %s" % pk_src, "traffic": gemm_traffic(cfg.name),
                "bytes_per_launch_pair": routed_bytes, "ms_per_launch_pair": round(routed_ms, 4)}
    else:
        achieved = routed_flops / (routed_ms / 1e3) / 1e12
        roof = {"bound": "tensor", "kernel": "grouped_gemm_kernel (routed gate/up + down, tcgen05)",
                "achieved": round(achieved, 1), "peak": peak, "unit": "TFLOP/s",
                "frac": round(achieved / peak, 4),
                "peak_kind": ("fp8 = %.0f x bf16 sustained (nominal ratio), %s" % (FP8_PER_BF16, pk_src)) if fp8
                else "bf16 sustained, %s" % pk_src,
                "traffic": gemm_traffic(cfg.name),
                "flops_per_launch_pair": routed_flops, "ms_per_launch_pair": round(routed_ms, 4)}
    if fp8:   # expert GEMMs at the FP8 rate, the router at the bf16 rate
        expert_flops = cfg.gemm_flops_per_block() * L
        t_flops = (expert_flops / (FP8_PER_BF16 * pk["bf16_tflops"] * 1e12)
                   + (flops - expert_flops) / (pk["bf16_tflops"] * 1e12))
        t_roof = max(t_flops, bytes_ / (pk["hbm_gbs"] * 1e9))
    else:
        t_flops = flops / (pk["bf16_tflops"] * 1e12)
    line = {
        "metric": METRIC_FP8 if fp8 else METRIC,
        "value": round(value, 1),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": {"bf16": "bf16", "f32": "f32", "fp8": "e4m3", "mxfp8": "e4m3+ue8m0/32"}[cfg.dtype],
        "data": "synthetic: seeded x~N(0,1), weights~N(0,1/fan_in), uniform router",
        "config": {"workload": configs.describe(cfg),
                   "schedule": ("two-stream overlap" if args.overlap else "one stream") + (", CUDA graph" if args.graph
                                                                                          else ""),
                   "T_per_gpu": T, "d": cfg.d, "E": cfg.E, "k": cfg.k,
                   "c": cfg.c, "n_shared": cfg.n_shared, "c_shared": cfg.c_shared, "L": L, "gate": cfg.gate,
                   "wiring": cfg.wiring,
                   "l2": "inputs larger than L2 (x %.2f GB, weights %.1f GB per block)" % (
                       T * cfg.d * 2 / 1e9, cfg.alg_bytes_per_block() / 1e9)},
        "roofline": roof,
        "layer_roofline": {"bound": "tensor" if t_flops >= bytes_ / (pk["hbm_gbs"] * 1e9)
                           else "hbm", "tokens_per_s_at_roofline": round(T / t_roof, 1),
                           "frac": round((T / (ms / 1e3)) / (T / t_roof), 4),
                           "tflops": round(flops / (ms / 1e3) / 1e12, 1),
                           "peaks": {"bf16_tflops": pk["bf16_tflops"], "hbm_gbs": pk["hbm_gbs"], "source": pk_src}},
        "breakdown_ms": {k: round(v, 4) for k, v in stage_ms.items()},
        "e2e": {"value": round(tokens / (e2e_ms / 1e3), 1), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4),
                "schedule": "double-buffered: step i+1's H2D and step i's D2H on two copy streams beside step i's compute"
                if not args.graph else "one CUDA graph replayed per step, copies in between"},
        "gpu_launches": int(launches * args.steps),
        "gpu_launches_per_step": int(launches),
        "clocks": clocks,
    }
    if host_blocks is not None:
        line["cpu_baseline"] = cpu_baseline(cfg, host_blocks, x, args.cpu_sample)
    return line


def per_stage_timing(cfg, stack, x, steps, stream):
    """The same stack driven through the single-step C-ABI entry points with
    CUDA events between stages (launch sequence identical to fs_farskip_stack)."""
    from mixture_experts_layer_expert_gb300 import fs
    T, d, k, E = cfg.T, cfg.d, cfg.k, cfg.E
    desc = stack.desc
    ws = fs.alloc_workspace(desc, 0)
    dev = x.device
    i32 = dict(dtype=torch.int32, device=dev)
    idx, w = torch.empty((T, k), **i32), torch.empty((T, k), dtype=torch.float32, device=dev)
    counts, offsets = torch.empty(E, **i32), torch.empty(E + 1, **i32)
    prow = fs.fs_dispatch_rows(desc)      # T k, or the MX path's 128-row-padded capacity
    pos, perm = torch.empty(T * k, **i32), torch.empty(prow, **i32)
    if cfg.dtype == "fp8":
        x_perm = fs.fp8_rows_empty(T * k, d, dev)
    elif cfg.dtype == "mxfp8":
        x_perm = fs.mx_rows_empty(prow, d, dev)
    else:
        x_perm = torch.empty((T * k, d), dtype=x.dtype, device=dev)
    y_perm = torch.empty((prow, d), dtype=x.dtype, device=dev)
    s = torch.empty((T, d), dtype=torch.float32, device=dev) if cfg.n_shared else None
    L = len(stack.blocks)
    o_bufs = [torch.empty((T, d), dtype=torch.float32, device=dev) for _ in range(3)]
    os_bufs = [torch.empty((T, d), dtype=torch.float32, device=dev) for _ in range(2)]
    u_bufs = [torch.empty((T, d), dtype=x.dtype, device=dev) for _ in range(2)]
    names = ["router", "dispatch", "routed", "shared", "combine"]
    tot = {n: 0.0 for n in names}
    for it in range(steps + 1):     # the first pass warms the extra buffers
        u, o_prev = x, x
        for b, pw in enumerate(stack.blocks):
            last = b == L - 1
            ev = cuda_events(6)
            ev[0].record(stream)
            fs.fs_router_topk(desc, u, pw["w_r"], pw["bias"], idx, w, None, ws)
            ev[1].record(stream)
            fs.fs_dispatch(desc, idx, u, counts, offsets, pos, perm, x_perm, ws)
            ev[2].record(stream)
            fs.fs_grouped_swiglu(desc, x_perm, offsets, pw["w13"], pw["w3"], y_perm, ws)
            ev[3].record(stream)
            if s is not None:
                fs.fs_shared_expert(desc, u, pw["w13_shared"], pw["w3_shared"], s, ws)
            ev[4].record(stream)
            o_k = stack.o_full if last else o_bufs[b % 3]
            os_k = stack.o_partial if last else os_bufs[b % 2]
            u_next = None if last else u_bufs[b % 2]
            fs.fs_combine(desc, y_perm, pos, w, o_prev, s, os_k, o_k, u_next, stack.wiring)
            ev[5].record(stream)
            torch.cuda.synchronize()
            if it > 0:
                for i, n in enumerate(names):
                    tot[n] += ev[i].elapsed_time(ev[i + 1])
            u = u_next
            o_prev = o_k
    return {n: v / steps for n, v in tot.items()}


def e2e_timing(cfg, stack, x, steps, stream, graph=False):
    """Host buffers in, host buffer out: every step copies its x from pinned host
    memory, runs the stack through the C ABI and copies o_L back.  Double-buffered:
    step i+1's input upload and step i's result download run on a copy stream
    beside step i's compute (each step's copies stay inside the timed region).
    With graph, the single captured input buffer is refilled and replayed in turn."""
    if not graph:
        return e2e_timing_pipelined(stack, x, steps, stream)
    x_host = x.cpu().pin_memory()
    o_host = torch.empty(stack.o_full.shape, dtype=stack.o_full.dtype).pin_memory()
    x_dev = x if graph else torch.empty_like(x)
    run = (lambda: stack.replay()) if graph else (lambda: stack.forward(x_dev))
    for _ in range(2):
        x_dev.copy_(x_host, non_blocking=True)
        run()
        o_host.copy_(stack.o_full, non_blocking=True)
    torch.cuda.synchronize()
    e0, e1 = cuda_events(2)
    e0.record(stream)
    for _ in range(steps):
        x_dev.copy_(x_host, non_blocking=True)
        run()
        o_host.copy_(stack.o_full, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    nb = x.numel() * x.element_size()
    return e0.elapsed_time(e1) / steps, nb, stack.o_full.numel() * stack.o_full.element_size()


def e2e_timing_pipelined(stack, x, steps, stream):
    """Uploads on one copy stream and downloads on another (separate copy engines;
    with both directions on one stream the overlap with compute depended on the
    box), step i+1's upload issued before step i's download."""
    from mixture_experts_layer_expert_gb300 import fs

    x_host = x.cpu().pin_memory()
    o_host = torch.empty(stack.o_full.shape, dtype=stack.o_full.dtype).pin_memory()
    xs = [torch.empty_like(x) for _ in range(2)]
    outs = [(torch.empty_like(stack.o_full), torch.empty_like(stack.o_partial)) for _ in range(2)]
    cs = torch.cuda.Stream(device=x.device)      # uploads
    cd = torch.cuda.Stream(device=x.device)      # downloads
    ev = {k: [torch.cuda.Event() for _ in range(2)] for k in ("h2d", "comp", "d2h")}
    L = len(stack.blocks)

    def upload(i):                            # step i's input, once step i-2 has finished reading the buffer
        b = i % 2
        if i >= 2:
            cs.wait_event(ev["comp"][b])
        with torch.cuda.stream(cs):
            xs[b].copy_(x_host, non_blocking=True)
        ev["h2d"][b].record(cs)

    def run(n):
        # the next input arrives during this step's compute and this result
        # leaves during the next
        upload(0)
        for i in range(n):
            b = i % 2
            stream.wait_event(ev["h2d"][b])
            if i >= 2:
                stream.wait_event(ev["d2h"][b])     # step i-2's result has left outs[b]
            fs.fs_farskip_stack(stack.desc, L, stack.wiring, stack.blocks, xs[b], outs[b][0], outs[b][1], stack.ws,
                                stream)
            ev["comp"][b].record(stream)
            if i + 1 < n:
                upload(i + 1)
            cd.wait_event(ev["comp"][b])
            with torch.cuda.stream(cd):
                o_host.copy_(outs[b][0], non_blocking=True)
            ev["d2h"][b].record(cd)

    run(2)                                    # untimed: first writes into the new device buffers
    torch.cuda.synchronize()
    e0, e1 = cuda_events(2)
    e0.record(stream)
    cs.wait_event(e0)
    cd.wait_event(e0)
    run(steps)
    stream.wait_stream(cs)
    stream.wait_stream(cd)
    e1.record(stream)
    torch.cuda.synchronize()
    nb = x.numel() * x.element_size()
    return e0.elapsed_time(e1) / steps, nb, stack.o_full.numel() * stack.o_full.element_size()


# ------------------------------------------------------------ training step

def train_e2e_pipelined(tr, x, dO, steps, stream):
    """Training steps with their host copies: x, dO (pinned) up and dx down every
    step, beside the compute: uploads on one copy stream, downloads on another
    (separate copy engines), step i+1's uploads issued before step i's download."""
    x_h, d_h = x.cpu().pin_memory(), dO.cpu().pin_memory()
    dx_h = torch.empty(tr.dx.shape, dtype=tr.dx.dtype).pin_memory()
    xs = [torch.empty_like(x) for _ in range(2)]
    ds = [torch.empty_like(dO) for _ in range(2)]
    dxs = [torch.empty_like(tr.dx) for _ in range(2)]
    cs = torch.cuda.Stream(device=x.device)      # uploads
    cd = torch.cuda.Stream(device=x.device)      # downloads
    ev = {k: [torch.cuda.Event() for _ in range(2)] for k in ("h2d", "comp", "d2h")}

    def upload(i):                     # step i's inputs, once step i-2 has finished reading them
        b = i % 2
        if i >= 2:
            cs.wait_event(ev["comp"][b])
        with torch.cuda.stream(cs):
            xs[b].copy_(x_h, non_blocking=True)
            ds[b].copy_(d_h, non_blocking=True)
        ev["h2d"][b].record(cs)

    def run(n):
        upload(0)
        for i in range(n):
            b = i % 2
            stream.wait_event(ev["h2d"][b])
            if i >= 2:
                stream.wait_event(ev["d2h"][b])      # step i-2's dx has left dxs[b]
            tr.forward(xs[b], stream=stream)
            tr.backward(ds[b], stream=stream, dx=dxs[b])
            ev["comp"][b].record(stream)
            if i + 1 < n:
                upload(i + 1)
            cd.wait_event(ev["comp"][b])
            with torch.cuda.stream(cd):
                dx_h.copy_(dxs[b], non_blocking=True)
            ev["d2h"][b].record(cd)

    run(2)                             # untimed: first writes into the new device buffers
    torch.cuda.synchronize()
    e0, e1 = cuda_events(2)
    e0.record(stream)
    cs.wait_event(e0)
    cd.wait_event(e0)
    run(steps)
    stream.wait_stream(cs)
    stream.wait_stream(cd)
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


def run_train(args, cfg, rank, world, local):
    """One step = fs_farskip_stack_train + fs_farskip_stack_backward over T tokens
    (bf16), with a fixed output gradient dO resident on the device."""
    from mixture_experts_layer_expert_gb300 import build, fs

    build.build()
    fs.lib()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    prob = synth.make_problem(cfg, device=dev)
    tr = fs.FarSkipTrainer(cfg, prob["blocks"], device=dev)
    x = prob["x"]
    del prob
    torch.cuda.empty_cache()
    T, L = cfg.T, cfg.L
    g = torch.Generator(device=dev).manual_seed(3)
    dO = torch.randn((T, cfg.d), generator=g, device=dev)
    stream = torch.cuda.current_stream()

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    for _ in range(args.warmup):
        tr.forward(x)
        tr.backward(dO)
    torch.cuda.synchronize()
    st, code = fs.fs_get_error()
    if st != 0:
        raise RuntimeError("device error word after warm-up: %d" % code)
    sampler = ClockSampler(local).start() if rank == 0 else None
    time.sleep(0.3 if sampler else 0)
    barrier()
    torch.cuda.synchronize()
    l0 = fs.fs_launch_count()
    ev = [cuda_events(3) for _ in range(args.steps)]
    for i in range(args.steps):
        ev[i][0].record(stream)
        tr.forward(x)
        ev[i][1].record(stream)
        tr.backward(dO)
        ev[i][2].record(stream)
    torch.cuda.synchronize()
    launches = (fs.fs_launch_count() - l0) // args.steps
    barrier()
    fwd_ms = sum(e[0].elapsed_time(e[1]) for e in ev) / args.steps
    bwd_ms = sum(e[1].elapsed_time(e[2]) for e in ev) / args.steps
    ms = fwd_ms + bwd_ms
    # end to end: x and dO from pinned host memory, dx back to the host, every step;
    # double-buffered like the inference stack: step i+1's inputs go up and step
    # i's dx comes down on a copy stream while step i+1 computes
    e2e_ms = train_e2e_pipelined(tr, x, dO, max(2, args.steps), stream)
    clocks = sampler.stop() if sampler else None
    st, code = fs.fs_get_error()
    if st != 0:
        raise RuntimeError("device error word after timing: %d" % code)
    ms, e2e_ms = reduce_max([ms, e2e_ms], world, dev)
    if rank != 0:
        return None
    pk, pk_src = peaks()
    gemm = cfg.gemm_flops_per_block() * L
    router = 2.0 * T * cfg.d * cfg.E * L
    flops = 3.0 * gemm + 3.0 * router          # forward, input gradients, weight gradients
    tflops = flops / (ms / 1e3) / 1e12
    peak = pk["bf16_tflops_sustained"]
    return {
        "metric": METRIC_TRAIN,
        "value": round(T * world / (ms / 1e3), 1),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic: seeded x~N(0,1), weights~N(0,1/fan_in), output gradient dO~N(0,1)",
        "config": {"workload": configs.describe(cfg) + ", training step", "T_per_gpu": T, "L": L,
                   "wiring": cfg.wiring, "l2": "inputs larger than L2"},
        "roofline": {"bound": "tensor", "kernel": "all GEMMs of the step (forward, input and weight gradients)",
                     "achieved": round(tflops, 1), "peak": peak, "unit": "TFLOP/s", "frac": round(tflops / peak, 4),
                     "peak_kind": "bf16 sustained, %s" % pk_src, "traffic": None,
                     "flops_per_step": flops},
        "breakdown_ms": {"forward_train": round(fwd_ms, 4), "backward": round(bwd_ms, 4)},
        "e2e": {"value": round(T * world / (e2e_ms / 1e3), 1), "unit": "tokens/s",
                "h2d_bytes_per_step": x.numel() * x.element_size() + dO.numel() * dO.element_size(),
                "d2h_bytes_per_step": tr.dx.numel() * tr.dx.element_size(), "ms_per_step": round(e2e_ms, 4),
                "schedule": "double-buffered: step i+1's H2D and step i's D2H on two copy streams beside step i's compute"},
        "gpu_launches": int(launches * args.steps),
        "gpu_launches_per_step": int(launches),
        "clocks": clocks,
    }


# ------------------------------------------------------------ CPU oracle

def oracle_cfg_for(cfg):
    import oracle
    dt = oracle.F32 if cfg.dtype == "f32" else oracle.BF16
    st = oracle.STORE_F32 if cfg.dtype == "f32" else oracle.STORE_BF16
    return oracle.make_cfg(cfg.d, cfg.E, cfg.k, cfg.c, cfg.n_shared, cfg.c_shared, cfg.gate, dt, st,
                           fp8={"fp8": "row", "mxfp8": "mx"}.get(cfg.dtype, False))


def cpu_baseline(cfg, host_blocks, x, sample):
    import oracle
    oracle.build()
    rows = np.arange(sample)
    xs = synth.to_numpy(x[:sample])
    oc = oracle_cfg_for(cfg)
    ws = [oracle.Weights(**b) for b in host_blocks]
    t0 = time.perf_counter()
    oracle.stack(oc, ws, cfg.wiring, xs, want_logits=False)
    dt_s = time.perf_counter() - t0
    return {"value": round(len(rows) / dt_s, 3), "unit": "tokens/s", "cores": oracle.num_threads(),
            "kind": "oracle", "sample": "first %d of the %d tokens, all L=%d blocks (plain C fp64, OpenMP over tokens)"
            % (sample, cfg.T, cfg.L), "seconds": round(dt_s, 2)}


# -------------------------------------------------------- reference arm

def run_reference(args, cfg, rank, world):
    if rank != 0:
        return None
    import oracle
    oracle.build()
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    T = args.ref_sample
    x = synth.make_x(cfg, device=dev, T=cfg.T)[:T]
    blocks = [synth.make_block_weights(cfg, b, device=dev) for b in range(cfg.L)]
    hb = [oracle.Weights(**{k: synth.to_numpy(v) for k, v in b.items()}) for b in blocks]
    del blocks
    xs = synth.to_numpy(x)
    oc = oracle_cfg_for(cfg)
    for _ in range(args.warmup):
        oracle.stack(oc, hb, cfg.wiring, xs[: max(1, T // 8)], want_logits=False)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.stack(oc, hb, cfg.wiring, xs, want_logits=False)
    sec = (time.perf_counter() - t0) / args.steps
    value = T / sec
    sample = "%d of the %d tokens per step, all L=%d blocks" % (T, cfg.T, cfg.L)
    return {"impl": "reference", "metric": METRIC_FP8 if cfg.dtype in ("fp8", "mxfp8") else METRIC, "value": round(value, 3), "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(sec * 1e3, 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic: seeded x~N(0,1), weights~N(0,1/fan_in)",
            "config": {"workload": configs.describe(cfg), "tokens_per_step": T},
            "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "cores": oracle.num_threads(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--config", default="v3", choices=sorted(configs.CONFIGS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-sample", type=int, default=1024)
    ap.add_argument("--ref-sample", type=int, default=64)
    ap.add_argument("--graph", action="store_true",
                    help="capture the stack once as a CUDA graph and replay it per step")
    ap.add_argument("--train", action="store_true",
                    help="time a training step (forward keeping state + backward) instead of the forward")
    ap.add_argument("--overlap", action="store_true",
                    help="two-stream FarSkip schedule (router/dispatch/shared of block k+1 beside block k's routed GEMMs)")
    args = ap.parse_args()
    rank, world, local = dist_env()
    cfg = configs.CONFIGS[args.config]
    if world > 1 and not torch.distributed.is_initialized():
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        torch.distributed.init_process_group(backend=backend)
    if args.impl == "reference":
        line = run_reference(args, cfg, rank, world)
    elif args.train:
        line = run_train(args, cfg, rank, world, local)
    else:
        line = run_ours(args, cfg, rank, world, local)
    if line is not None:
        print(json.dumps(line), flush=True)
    if world > 1 and torch.distributed.is_initialized():
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
