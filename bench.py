#!/usr/bin/env python3
"""Benchmark of the NVFP4 routed-MoE expert path on one GB300 (or N independent replicas).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

One step = one pass of the whole hot path over one batch: moe_quantize_input,
moe_plan and moe_grouped_fp4_forward (permute, GEMM1 + SwiGLU/ReLU^2 + NVFP4
requant, GEMM2, finalize). Inputs (BF16 hidden states, routing) and the prepared
NVFP4 weights are resident in HBM; L2 is flushed between steps outside the timed events
(a 256 MB write, then a 256 MB read of a second buffer so the lines left in L2 are clean;
`--l2-flush write` skips the read). Rank 0 prints one JSON line.

--impl reference times the CPU oracle (oracle/) on the machine's host cores on a
bounded sample of the same workload (this repository's reference arm).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import moe_inputs as mi  # noqa: E402

METRIC = "MoE layer tokens/s; % of NVFP4-TC/HBM roofline (decode T=8, prefill 4k)"
NV = 0.5 + 1.0 / 16.0      # NVFP4 bytes per element: packed E2M1 + one E4M3 scale per 16
FP4_OVER_BF16 = 13.5 / 2.25  # nominal dense ratio (GB300): FP4 tensor rate / BF16 tensor rate


OUTPUT_MODES = {"finalized": 1, "accumulate": 2}


def workload_name(cfg) -> str:
    s = f"{cfg.name}: T={cfg.M} H={cfg.H} I={cfg.I} E={cfg.E} top_k={cfg.top_k} {cfg.act}"
    if cfg.num_local is not None:
        s += f" local={cfg.local_offset}..{cfg.local_offset + cfg.El - 1}"
    if cfg.skew:
        s += f" zipf={cfg.skew}"
    return s


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# --------------------------------------------------------------------------- replicas
def max_over_ranks(x: float, world: int, device=None) -> float:
    """The largest of every rank's x, returned on every rank (x itself for one process). The
    whole job is timed by its slowest replica; `device` is where the reduction tensor lives
    (the GPU for NCCL, None for gloo)."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(tokens_per_rank: int, ms_slowest: float, world: int) -> float:
    """Whole-job tokens/s: `world` independent replicas, each taking tokens_per_rank tokens
    per step, timed by the slowest one."""
    return world * tokens_per_rank / (ms_slowest * 1e-3)


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# --------------------------------------------------------------------------- algorithmic work
def kernel_work(cfg, ids):
    """Per-launch work of each kernel of one step (no padding rows, no unused experts).

    `bytes` is the scope table's algorithmic count: the weights of the active local experts
    and their alphas, and the layer's own inputs and outputs (BF16 hidden states in, BF16
    output out, routing ids and weights), each charged to the kernel that reads or writes
    it; intermediates and permuted copies are excluded, since an implementation may avoid
    them, so the kernels' `bytes` sum to the whole step's. `bytes_incl_intermediates` adds
    what this implementation writes and reads back between its kernels (the NVFP4 activation
    pack and its permuted rows, the NVFP4 intermediate, the BF16 expert rows)."""
    l = ids.astype(np.int64) - cfg.local_offset
    valid = (l >= 0) & (l < cfg.El)
    R = int(valid.sum())
    active = int(np.unique(l[valid]).size)
    M, H, I, N1, k = cfg.M, cfg.H, cfg.I, cfg.N1, cfg.top_k
    w = {
        "quantize": {"bytes": M * H * 2, "bytes_incl_intermediates": M * H * 2 + M * H * NV + M * 4,
                     "flops": 0.0},
        "plan": {"bytes": M * k * 4, "bytes_incl_intermediates": M * k * 4 * 2 + cfg.El * 8, "flops": 0.0},
        "permute": {"bytes": 0, "bytes_incl_intermediates": 2 * R * H * NV, "flops": 0.0},
        "gemm1": {"bytes": active * N1 * H * NV + cfg.El * 4,
                  "bytes_incl_intermediates": active * N1 * H * NV + R * H * NV + R * I * NV + cfg.El * 4,
                  "flops": 2.0 * R * H * N1},
        "gemm2": {"bytes": active * H * I * NV + cfg.El * 4,
                  "bytes_incl_intermediates": active * H * I * NV + R * I * NV + R * H * 2 + cfg.El * 4,
                  "flops": 2.0 * R * I * H},
        "finalize": {"bytes": M * H * 2 + M * k * 4,
                     "bytes_incl_intermediates": R * H * 2 + M * k * 8 + M * H * 2, "flops": 0.0},
    }
    step = mi.algorithmic_work(cfg, ids, finalize=True)
    return w, step, R, active


def roofline(bytes_, flops, t_s, peaks):
    """Roofline of one launch: the bound is the larger of bytes at the HBM peak and FLOPs at
    the FP4 tensor peak; frac = that time / the measured time t_s."""
    fp4_peak = peaks["bf16_tflops"] * FP4_OVER_BF16
    hbm_time = bytes_ / (peaks["hbm_gbs"] * 1e9)
    tc_time = flops / (fp4_peak * 1e12)
    if hbm_time >= tc_time:
        r = {"bound": "hbm", "achieved": bytes_ / t_s / 1e9, "peak": peaks["hbm_gbs"], "unit": "GB/s"}
    else:
        r = {"bound": "tensor", "achieved": flops / t_s / 1e12, "peak": fp4_peak, "unit": "TFLOP/s"}
    r["frac"] = r["achieved"] / r["peak"]
    r["peak_source"] = (f"{peaks['source']} HBM copy" if r["bound"] == "hbm"
                        else f"{peaks['source']} bf16 burst x {FP4_OVER_BF16:g} (nominal FP4/BF16)")
    return r


# --------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append(ln.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.12)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------- GPU arm
def weight_key(cfg) -> tuple:
    """What the prepared layer of a workload depends on: workloads with equal keys share it."""
    return (cfg.H, cfg.I, cfg.E, cfg.act, cfg.weight_seed, cfg.local_offset, cfg.El, cfg.fc2_input_scale,
            cfg.scale_mode)


def setup_layer(cfg, dev):
    import torch

    import nvfp4_routed_moe_sort_gb300 as pkg
    # draw and quantise one expert at a time (the BF16 stacks of the large configs are 22 GB)
    El = cfg.El
    d1 = torch.empty(El, cfg.N1, cfg.H // 2, dtype=torch.uint8, device=dev)
    s1 = torch.empty(El, cfg.N1, cfg.H // 16, dtype=torch.uint8, device=dev)
    a1 = torch.empty(El, dtype=torch.float32, device=dev)
    d2 = torch.empty(El, cfg.H, cfg.I // 2, dtype=torch.uint8, device=dev)
    s2 = torch.empty(El, cfg.H, cfg.I // 16, dtype=torch.uint8, device=dev)
    a2 = torch.empty(El, dtype=torch.float32, device=dev)
    scratch = torch.empty(4, dtype=torch.float32, device=dev)
    alpha = torch.empty(4, dtype=torch.float32, device=dev)   # 16-byte aligned per-call output
    for l in range(El):
        w1 = mi.expert_w1_bf16(cfg, l, dev)
        pkg.moe_quantize_weights(w1.view(torch.int16)[None], d1[l:l + 1], s1[l:l + 1], alpha, scratch)
        a1[l] = alpha[0]
        del w1
        w2 = mi.expert_w2_bf16(cfg, l, dev)
        pkg.moe_quantize_weights(w2.view(torch.int16)[None], d2[l:l + 1], s2[l:l + 1], alpha, scratch)
        a2[l] = alpha[0]
        del w2
    layer = pkg.NVFP4RoutedMoE(d1, s1, a1, d2, s2, a2, activation=cfg.act, num_experts=cfg.E,
                               local_expert_offset=cfg.local_offset, fc2_input_scale=cfg.fc2_input_scale,
                               scale_mode=cfg.scale_mode)
    torch.cuda.synchronize()
    return layer


def setup_inputs(cfg, dev):
    x = mi.hidden_bf16(cfg, dev)
    ids, tw = mi.routing(cfg)
    return x, ids, tw


def kernel_source_hash() -> str:
    """sha256 prefix of the GEMM kernel sources (gemm_kernel.cuh, gemm_decode.cuh, common.cuh)."""
    csrc = os.path.join(ROOT, "nvfp4_routed_moe_sort_gb300", "csrc")
    h = hashlib.sha256()
    for name in ("gemm_kernel.cuh", "gemm_decode.cuh", "common.cuh"):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def traffic_from_profiles(kernel: str, workload: str):
    """DRAM bytes per launch of `kernel` from the committed ncu summary
    (profiles/dram_traffic.txt), or None when the kernel's source has changed since the
    counters were taken (kernel_source_hash)."""
    kernel = {"gemm1+gemm2 (chained)": "gemm_chained", "gemm1+gemm2 (decode)": "gemm_decode"}.get(kernel, kernel)
    p = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(p):
        return None
    h = kernel_source_hash()
    with open(p) as f:
        for ln in f:
            parts = ln.split()
            if len(parts) == 5 and not ln.startswith("#") and parts[0] == workload and parts[1] == kernel:
                return int(parts[2]) if parts[4] == h else None
    return None


class L2Flush:
    """Evicts the step's data from the 129 MB L2 between steps: a 256 MB write and, unless
    write-only, a 256 MB read of a second buffer, so that the lines left in L2 are clean
    and the timed step does not pay for writing the flush buffer back."""

    def __init__(self, dev, clean: bool):
        import torch
        self.w = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        self.r = torch.zeros(256 << 20, dtype=torch.uint8, device=dev).view(torch.int64) if clean else None
        self.sink = None

    def __call__(self):
        self.w.zero_()
        if self.r is not None:
            self.sink = self.r.sum()


def measure(args, cfg, layer, x, ids, tw, dev, world, with_e2e: bool):
    """One workload: K timed CUDA-graph replays of the whole step (L2 flushed between them),
    the per-kernel split from eager calls, the rooflines, and optionally the end-to-end run."""
    import torch

    ids_t = torch.from_numpy(ids).to(dev)
    tw_t = torch.from_numpy(tw).to(dev)
    M, k = ids.shape
    mode = OUTPUT_MODES[args.output]
    b = layer.routed_buffers(M, k, mode)
    # accumulated output: every step adds into this caller-owned tensor
    acc_out = torch.zeros(M, cfg.H, dtype=torch.bfloat16, device=dev) if mode == 2 else None
    flush = L2Flush(dev, clean=args.l2_flush == "write+read")
    n_ev = 5
    K, W = args.steps, args.warmup

    # the timed step: one CUDA-graph replay of the whole path
    graph = layer.capture(x, ids_t, tw_t, mode, out=acc_out)
    for i in range(W):
        flush()
        graph.replay()
    torch.cuda.synchronize()
    barrier(world)
    s_ev, e_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(dev.index)
    clocks.start()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    step_times = []
    for i in range(K):
        flush()
        s_ev.record()
        graph.replay()
        e_ev.record()
        e_ev.synchronize()
        step_times.append(s_ev.elapsed_time(e_ev))
    torch.cuda.synchronize()
    barrier(world)
    wall = time.perf_counter() - t0
    clk = clocks.stop()
    # kernel boundaries: the same calls launched eagerly with an event between kernels. A
    # device-side sleep enqueued first lets the host queue every step before the GPU starts,
    # so the events bracket device time only (no host gaps).
    KE = min(K, 50)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(n_ev)] for _ in range(KE)]
    for row in evs:          # torch creates the CUDA event on its first record
        for e in row:
            e.record()
    for _ in range(W):
        flush()
        layer.forward(x, ids_t, tw_t, mode, out=acc_out)
    torch.cuda.synchronize()
    torch.cuda._sleep(int(60e6))   # ~30 ms at 2 GHz
    for e in evs:
        flush()
        layer.routed(x, ids_t, tw_t, b, mode, step_events=e, out=acc_out)
    torch.cuda.synchronize()
    kern_times = [[e[j].elapsed_time(e[j + 1]) for j in range(n_ev - 1)] for e in evs]
    eager_ms = float(np.mean([e[0].elapsed_time(e[4]) for e in evs]))
    assert layer.device_status(M, k, mode) == 0, "device status word set"
    # prologue = quantise + plan + permute (one kernel for small batches)
    names = ["prologue", "gemm1", "gemm2", "combine"]
    per = {n: [t[c] for t in kern_times] for c, n in enumerate(names)}
    ms = max_over_ranks(float(np.mean(step_times)), world, dev)
    work, stepw, R, active = kernel_work(cfg, ids)
    kern_ms = {n: float(np.mean(v)) for n, v in per.items()}
    # GEMM1 and GEMM2 run as one launch (its time is the gemm1 interval): the decode kernel
    # (weights as the 128-row MMA operand) up to 16 tokens, else the chained one
    dom = "gemm1+gemm2 (decode)" if M <= 16 else "gemm1+gemm2 (chained)"
    kern_ms[dom] = kern_ms.pop("gemm1") + kern_ms.pop("gemm2")
    work[dom] = {key: work["gemm1"][key] + work["gemm2"][key]
                 for key in ("bytes", "bytes_incl_intermediates", "flops")}
    peaks = load_peaks()
    t_dom = kern_ms[dom] * 1e-3
    roof = roofline(work[dom]["bytes"], work[dom]["flops"], t_dom, peaks)
    roof["kernel"] = dom
    roof["bytes"] = work[dom]["bytes"]
    roof["flops"] = work[dom]["flops"]
    roof["traffic"] = traffic_from_profiles(dom, cfg.name)
    incl = roofline(work[dom]["bytes_incl_intermediates"], work[dom]["flops"], t_dom, peaks)
    roof["frac_incl_intermediates"] = incl["frac"]
    roof["bytes_incl_intermediates"] = work[dom]["bytes_incl_intermediates"]
    fp4_peak = peaks["bf16_tflops"] * FP4_OVER_BF16
    step_roof_s = max(stepw["bytes"] / (peaks["hbm_gbs"] * 1e9), stepw["flops"] / (fp4_peak * 1e12))
    # end to end through the public API with host buffers
    e2e = run_e2e(layer, x, ids, tw, dev, max(3, min(K, 50)), flush) if with_e2e else None
    if e2e is not None:  # the whole job end to end: every replica's copies and step, the slowest
        e2e["ms_per_step"] = max_over_ranks(e2e["ms_per_step"], world, dev)
        e2e["value"] = replica_throughput(M, e2e["ms_per_step"], world)
    # the same graph with a write-only flush (its dirty lines are written back during the step)
    wo = L2Flush(dev, clean=False)
    wo_times = []
    for i in range(min(K, 50)):
        wo()
        s_ev.record()
        graph.replay()
        e_ev.record()
        e_ev.synchronize()
        wo_times.append(s_ev.elapsed_time(e_ev))
    del wo, flush, graph
    small = M * k <= 2048 and M * cfg.H <= (1 << 17)
    # small: prologue, GEMMs (one launch), combine; otherwise the plan (one kernel up to 2048
    # slots, else three), the quantiser storing into the plan rows, GEMMs, combine
    if small:
        launches_per_step = 3
    else:
        launches_per_step = (1 if M * k <= 2048 else 3) + 3
    return {
        "metric": METRIC, "value": replica_throughput(M, ms, world), "unit": "tokens/s", "n_gpus": world, "steps": K,
        "warmup": W, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "nvfp4 (e2m1 x e2m1, e4m3 block scales, fp32 accumulate)", "data": "synthetic",
        "config": {"workload": workload_name(cfg), "tokens": M, "hidden": cfg.H, "inter": cfg.I,
                   "experts": cfg.E, "top_k": k, "routed_rows": R, "active_experts": active,
                   "l2": ("flushed between steps outside the timed events: 256 MB write"
                          + (", then 256 MB read of a second buffer (clean lines)"
                             if args.l2_flush == "write+read" else "")),
                   "output": args.output,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": roof,
        "step_roofline": {"frac": step_roof_s / (ms * 1e-3), "bytes": stepw["bytes"], "flops": stepw["flops"],
                          "note": "whole step: max(bytes/HBM peak, flops/FP4 peak) over measured step time"},
        "kernels_ms": kern_ms,
        "timing": "each step is one CUDA-graph replay of the whole path, timed by events on its stream; "
                  "kernel times from the same calls launched eagerly with events between the kernels, "
                  "queued behind a device sleep so no host gap is timed; "
                  f"an eager step takes {eager_ms:.4f} ms",
        "eager_ms_per_step": eager_ms,
        "write_only_flush_ms_per_step": float(np.mean(wo_times)),
        "e2e": e2e,
        "gpu_launches": launches_per_step * K,
        "clocks": clk,
        "wall_s_timed_region": wall,
    }


# the metric's other configurations, measured in the same run after the headline one
EXTRA_WORKLOADS = ["decode_t4", "wide_decode", "prefill_uniform", "prefill_skewed", "relu2_ep"]


def workload_summary(r: dict) -> dict:
    """The fields of one extra workload's measurement kept in the `workloads` object."""
    c = r["config"]
    return {"workload": c["workload"], "tokens": c["tokens"], "routed_rows": c["routed_rows"],
            "active_experts": c["active_experts"], "ms_per_step": r["ms_per_step"], "tokens_per_s": r["value"],
            "step_roofline": r["step_roofline"], "roofline": r["roofline"], "kernels_ms": r["kernels_ms"],
            "eager_ms_per_step": r["eager_ms_per_step"], "gpu_launches": r["gpu_launches"], "clocks": r["clocks"]}


def run_gpu(args, cfg, rank, world):
    import torch

    dev = torch.device(f"cuda:{int(os.environ.get('LOCAL_RANK', 0))}")
    torch.cuda.set_device(dev)
    from nvfp4_routed_moe_sort_gb300.build import build
    build()
    layers = {}

    def layer_for(c):
        key = weight_key(c)
        if key not in layers:
            layers.clear()            # one weight set resident at a time
            torch.cuda.empty_cache()
            layers[key] = setup_layer(c, dev)
        return layers[key]

    x, ids, tw = setup_inputs(cfg, dev)
    res = measure(args, cfg, layer_for(cfg), x, ids, tw, dev, world, with_e2e=not args.no_e2e)
    extra = [] if args.workloads == "none" else (
        EXTRA_WORKLOADS if args.workloads == "all" else [w for w in args.workloads.split(",") if w])
    extra = [w for w in extra if w != args.workload and not args.set]
    if extra:
        # group workloads that share a weight set, so each set is prepared once
        order = sorted(extra, key=lambda w: (weight_key(mi.CONFIGS[w]) != weight_key(cfg),
                                             str(weight_key(mi.CONFIGS[w]))))
        res["workloads"] = {}
        for w in order:
            c = mi.CONFIGS[w]
            xw, idw, tww = setup_inputs(c, dev)
            r = measure(args, c, layer_for(c), xw, idw, tww, dev, world, with_e2e=False)
            res["workloads"][w] = workload_summary(r)
            del xw
        res["workloads"] = {w: res["workloads"][w] for w in extra}
    return res


def run_e2e(layer, x, ids, tw, dev, steps, flush):
    """Host buffers in, host buffer out, through NVFP4RoutedMoE.capture_host: one CUDA graph per
    step from the step's inputs in one pinned host buffer (hidden states, routing ids and
    weights) to the output in a pinned host tensor. The reported figure is the API's own
    choice of transfer (`transfer`); the other variant is timed too and reported beside it."""
    import torch
    from nvfp4_routed_moe_sort_gb300 import HostStaging
    M, k = ids.shape
    H = x.shape[1]
    staging = HostStaging(M, H, k, dev)
    staging.x.copy_(x.cpu())
    staging.ids.copy_(torch.from_numpy(np.ascontiguousarray(ids, dtype=np.int32)))
    staging.weights.copy_(torch.from_numpy(np.ascontiguousarray(tw, dtype=np.float32)))
    hout = torch.empty(M, H, dtype=torch.bfloat16).pin_memory()

    def time_graph(graph):
        times = []
        for i in range(steps + 3):
            flush()
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record()
            graph.replay()
            e.record()
            e.synchronize()
            if i >= 3:
                times.append(s.elapsed_time(e))
        return float(np.mean(times))

    graph = layer.capture_host(staging, hout)
    direct = staging.direct
    ms = time_graph(graph)
    other = time_graph(layer.capture_host(staging, hout, direct=not direct))
    kinds = {True: "in place: the kernels read the pinned inputs and write the pinned output over NVLink-C2C",
             False: "copies: one H2D copy of the staging buffer and one D2H copy of the output, in the graph"}
    in_bytes = staging.x.numel() * 2 + staging.ids.numel() * 4 + staging.weights.numel() * 4
    return {"value": M / (ms * 1e-3), "unit": "tokens/s", "ms_per_step": ms,
            "h2d_bytes_per_step": int(in_bytes if direct else staging.nbytes),
            "d2h_bytes_per_step": int(hout.numel() * 2),
            "h2d_copies_per_step": 0 if direct else 1, "transfer": kinds[direct],
            "other_transfer": {"transfer": kinds[not direct], "ms_per_step": other},
            "output": "finalized"}


# --------------------------------------------------------------------------- oracle arm
def blas_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count() or 1


class OracleArm:
    """The CPU oracle on a fixed sample of the workload's tokens (weights prepared once)."""

    def __init__(self, cfg, n_tokens: int):
        from oracle import moe as O
        from oracle import quantize as Q
        self.cfg = cfg
        self.O = O
        self.Q = Q
        dev = "cuda" if _cuda_available() else "cpu"
        x = mi.hidden_bf16(cfg, dev).float().cpu().numpy()
        self.ids, self.tw = mi.routing(cfg)
        self.tokens = list(range(min(n_tokens, cfg.M)))
        self.x = x[self.tokens]
        cache = {}

        def load(l):
            if l not in cache:
                w1 = mi.expert_w1_bf16(cfg, l, dev).float().cpu().numpy()
                w2 = mi.expert_w2_bf16(cfg, l, dev).float().cpu().numpy()
                cache[l] = (Q.quantize_weight(w1), Q.quantize_weight(w2))
            return cache[l]
        self.W = O.ExpertWeights(cfg.El, cfg.H, cfg.I, cfg.gated, load)
        for t in self.tokens:                        # weight preparation is not timed
            for j in range(cfg.top_k):
                l = int(self.ids[t, j]) - cfg.local_offset
                if 0 <= l < cfg.El:
                    self.W.get(l)

    def step(self):
        cfg = self.cfg
        xq, xsf, xs = self.Q.quantize_activations(self.x, cfg.scale_mode)
        n = len(self.tokens)
        ids = self.ids[self.tokens]
        tw = self.tw[self.tokens]
        return self.O.forward_tokens(list(range(n)), xq, xsf, xs, ids, tw, self.W, cfg.act,
                                     local_expert_offset=cfg.local_offset,
                                     fc2_input_scale=cfg.fc2_input_scale)["out"]


def _cuda_available() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


def oracle_sample_tokens(cfg) -> int:
    # about 1-3 s of oracle work per step on a many-core host
    big = cfg.H * cfg.N1 > 8_000_000
    return 1 if big else min(cfg.M, 2)


def run_reference(args, cfg):
    arm = OracleArm(cfg, oracle_sample_tokens(cfg))
    for _ in range(args.warmup):
        arm.step()
    times = []
    for _ in range(args.steps):
        t = time.perf_counter()
        arm.step()
        times.append(time.perf_counter() - t)
    s = float(np.mean(times))
    n = len(arm.tokens)
    v = n / s
    sample = f"tokens {arm.tokens} of the batch per step (all their routed experts), weights prepared untimed"
    return {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": s * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64 sums / f32 codecs (CPU oracle)", "data": "synthetic",
        "config": {"workload": workload_name(cfg), "tokens": cfg.M},
        "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": blas_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def cpu_baseline(cfg, budget_s: float = 12.0):
    """The oracle as it stands, on a bounded sample of the workload, on this host's cores."""
    arm = OracleArm(cfg, oracle_sample_tokens(cfg))
    t0 = time.perf_counter()
    n = 0
    while True:
        arm.step()
        n += 1
        if time.perf_counter() - t0 > budget_s or n >= 20:
            break
    s = (time.perf_counter() - t0) / n
    return {"value": len(arm.tokens) / s, "unit": "tokens/s", "cores": blas_threads(), "kind": "oracle",
            "sample": f"{n} passes over tokens {arm.tokens} (all their routed experts); weights prepared untimed"}


# --------------------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="decode_t8", choices=sorted(mi.CONFIGS))
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--l2-flush", default="write+read", choices=["write+read", "write"],
                    help="between steps: a 256 MB write, then (default) a 256 MB read leaving clean lines")
    ap.add_argument("--output", default="finalized", choices=sorted(OUTPUT_MODES),
                    help="finalized: ordered combine into a fresh out; accumulate: FP32 reduction into out")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer run (profiling)")
    ap.add_argument("--set", action="append", default=[], metavar="FIELD=VALUE",
                    help="override a workload field (e.g. E=64 M=1024) for smaller profiling cases")
    ap.add_argument("--workloads", default="all",
                    help="the other configurations measured in the same run and reported in the `workloads` "
                         "object: all (default), none, or a comma-separated list")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3 (untimed warm-up steps before the timed region)")
    cfg = mi.CONFIGS[args.workload]
    for kv in args.set:
        k_, v_ = kv.split("=", 1)
        cur = getattr(cfg, k_)
        cfg = cfg.with_(**{k_: type(cur)(v_) if cur is not None else int(v_)})
    if args.set:
        cfg = cfg.with_(name=cfg.name + "[" + ",".join(args.set) + "]")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank != 0:
            return 0
        print(json.dumps(run_reference(args, cfg)), flush=True)
        return 0
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        dist.init_process_group("nccl")
    res = run_gpu(args, cfg, rank, world)
    if rank == 0:
        if not args.no_cpu_baseline:
            res["cpu_baseline"] = cpu_baseline(cfg)
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
