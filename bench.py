#!/usr/bin/env python
"""Benchmark of the int4 routed-MoE FFN step on GB300.

One step = one moe_forward call (router, top-k, gate/up + SwiGLU, down +
combine + shared expert) on one batch of synthetic tokens, default the
GLM-5.2 MoE layer at decode (T=1, H=6144, E=256, top-8, inter 2048, one
shared expert, int4 per-row weights, all 256 experts resident in HBM).

Timing: W warm-up steps, then exactly K steps back to back between two CUDA
events on the launching stream.  The layer is resident in L copies (default
8) at distinct device addresses, and step i uses copy i mod L: inputs larger
than L2 (L x 4.84 GB for the GLM-5.2 layer), so every step reads its weights
from HBM, as a decode loop that walks a model's MoE layers does; no flush is
needed.  Inputs rotate over 16 token vectors, so the routed experts change from
step to step.  value = tokens / timed span (whole job; max over ranks under
torchrun).  Beside it: the same steps each bracketed by events after an L2
flush (one copy, 256 MiB write + 256 MiB read outside the events).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time
from pathlib import Path

import numpy as np

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

import synth  # noqa: E402

METRIC = "MoE-layer decode tokens/s and achieved HBM GB/s vs ~8 TB/s (GLM-5.2 shape)"
N_X = 16                      # distinct token batches rotated through the steps
FLUSH_BYTES = 256 << 20       # > 129 MB L2
# committed ncu traffic summaries: dominant kernel -> (summary file, the source it was taken from)
# committed ncu DRAM summaries per (dominant kernel, workload, tokens per step)
TRAFFIC_FILES = {
    ("fused", "glm_decode", 1): ("traffic_decode_fused_glm_decode.txt", "moe_decode.cu"),
    ("gate_up", "glm_batched", 512): ("traffic_gateup_batched_glm.txt", "moe_kernels.cu"),
}


# --------------------------------------------------------------------------- helpers

def expert_bytes(H: int, I: int, fmt: int = 0) -> int:
    """Gate/up/down weight bytes (int4 packed or int8) + float32 per-row scales of one expert."""
    return synth.slab_bytes(H, I, fmt) + 4 * synth.scale_count(H, I, fmt)


def gateup_bytes(H: int, I: int, fmt: int = 0) -> int:
    """Bytes the gate/up kernel must read for one expert: two [I, H] weight
    matrices (H/2 bytes per int4 row, H per int8 row) and their 2I float32 scales."""
    return 2 * I * (H if fmt == 1 else (H + 1) // 2) + (2 * I * H // 64 * 4 if fmt == 2 else 8 * I)


def step_bytes(wl, T: int, touched: int) -> int:
    """Algorithmic HBM bytes of one step: router weight and bias, every routed
    expert the batch touches (each read once), the shared expert, x and y."""
    b = wl.E * wl.H * 4 + wl.E * 4 + touched * expert_bytes(wl.H, wl.I, wl.expert_format)
    if wl.n_shared:
        b += expert_bytes(wl.H, wl.I_shared, wl.shared_format)
    return b + 2 * T * wl.H * 4


FORMAT_NAMES = {0: "int4 per-row", 1: "int8 per-row", 2: "int4 affine group-64"}


def workload_desc(wl) -> str:
    route = ("softmax top-k" if wl.score_func == 1 else
             f"sigmoid+bias noaux_tc n_group={wl.n_group}" + (f" topk_group={wl.topk_group}" if wl.n_group > 1 else ""))
    s = (f"{wl.name}: T={wl.T}, H={wl.H}, E={wl.E} routed, top-{wl.K}, moe_inter={wl.I}, "
         f"{wl.n_shared} shared (inter {wl.I_shared}), {route}, "
         f"{'norm_topk' if wl.norm_topk else 'no renorm'}, routed_scale={wl.routed_scale}, "
         f"{FORMAT_NAMES[wl.expert_format]} routed weights"
         + (f", {FORMAT_NAMES[wl.shared_format]} shared" if wl.n_shared else "")
         + f", seed {wl.seed}")
    if wl.n_layers > 1:
        s += f", {wl.n_layers} chained layers x <- x + moe(rmsnorm(x))"
    return s


def rank_streams(rank: int, world: int, n: int) -> list[int]:
    """Token-stream ids of one rank: disjoint across ranks (weak scaling, no
    data exchange: each rank runs its own copy of the layer on its own tokens)."""
    return [rank * 100_000 + i for i in range(n)]


def reduce_max(value: float, dist_on: bool) -> float:
    if not dist_on:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist_on: bool):
    if dist_on:
        import torch.distributed as dist
        dist.barrier()


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,utilization.gpu,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.15)
        return self

    def __exit__(self, *exc):
        time.sleep(0.1)
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        rows = []
        for l in self.lines:
            f = [v.strip() for v in l.split(",")]
            if len(f) < 10:
                continue
            try:
                rows.append(dict(sm=float(f[1]), smax=float(f[2]), util=float(f[4]),
                                 hw=f[6], hwt=f[7], swt=f[8], pcap=f[9]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        load = [r for r in rows if r["util"] > 0] or rows
        reasons = set()
        for r in load:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("pcap", "sw_power_cap")):
                if r[key].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in load),
                "sm_max_mhz": max(r["smax"] for r in rows), "reasons": sorted(reasons),
                "samples": len(load)}


def measured_peaks():
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        d = json.loads(p.read_text())
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def measured_tensor_peak():
    """Dense f16/bf16 tensor rate: the measured cuBLAS bf16 burst figure (the
    f16 and bf16 tensor rates are the same), else the recipe's fallback."""
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        d = json.loads(p.read_text())
        if "bf16_tflops" in d:
            return float(d["bf16_tflops"]), "measured (MEASURED_PEAKS.json bf16_tflops, burst; f16 = bf16 rate)"
    return 1900.0, "fallback (1.9 PFLOP/s bf16 burst)"


def binding_roofline(hbm_frac: float, tensor_frac: float) -> str:
    """The roof a tensor-core kernel is nearer to: 'tensor' when its fraction of the tensor
    peak is at least its fraction of the copy bandwidth, else 'hbm' (small batches stream
    weights far below the tensor peak)."""
    return "tensor" if tensor_frac >= hbm_frac else "hbm"


def recorded_traffic(kind: str, workload: str, T: int):
    """DRAM bytes per launch of the dominant kernel from the committed ncu
    summary of this workload, or None when there is none or the kernel source
    changed since the capture."""
    if (kind, workload, T) not in TRAFFIC_FILES:
        return None
    name, src_name = TRAFFIC_FILES[(kind, workload, T)]
    f = ROOT / "profiles" / name
    if not f.exists():
        return None
    kv = {}
    for line in f.read_text().splitlines():
        if ":" in line and not line.startswith("#"):
            k, v = line.split(":", 1)
            kv[k.strip()] = v.strip()
    src = ROOT / "int4_moe_expert_gb300" / "csrc" / src_name
    sha = hashlib.sha256(src.read_bytes()).hexdigest()[:16]
    if kv.get("kernel_source_sha256_16") != sha or "traffic_bytes_per_launch" not in kv:
        return None
    return float(kv["traffic_bytes_per_launch"])



def kernel_span_stats(moe, cfg, copies, xs, y, T, stream, wl):
    """Kernel-only time of the decode step: the kernel's own global-timer trace (a handle
    with MOE_FLAG_TRACE over the same weights, one per layer copy), from the first block's
    start (past the wait for the previous kernel) to the last block's end, calls back to back
    in the bench's rotation; the event-timed step adds the launch and the gap between calls."""
    import ctypes as C
    import numpy as np
    import torch
    tcfg = moe.MoeConfig.from_buffer_copy(cfg)
    tcfg.flags |= moe.MOE_FLAG_TRACE
    traced = [moe.MoeLayer(tcfg, c.router_w, c.router_b, c.slabs, c.scales, c.sh_slab, c.sh_scale,
                           max_tokens=T) for c in copies]
    spans, gaps = [], []
    try:
        for rep in range(8):
            for i in range(3 * len(traced)):
                moe.moe_forward(traced[i % len(traced)].handle, xs[i % len(xs)], T, y, stream)
            torch.cuda.synchronize()
            recs = []
            for t in traced:
                tr = moe.moe_trace_read(t.handle).astype(np.int64)
                st, en = tr[:, 0], tr[:, 6]
                if (st > 0).all() and (en > 0).all():
                    recs.append((int(st.min()), int(en.max())))
            recs.sort()
            for (a0, a1), (b0, _) in zip(recs, recs[1:]):
                spans.append((a1 - a0) / 1e3)
                gaps.append((b0 - a1) / 1e3)
        for t in traced:
            assert moe.moe_device_error(t.handle) == 0
    finally:
        for t in traced:
            t.close()
    if not spans:
        return None
    span = statistics.median(spans)
    b = step_bytes(wl, T, wl.K)
    return {"median_us": round(span, 2), "gap_median_us": round(statistics.median(gaps), 2),
            "hbm_frac_of_span": round(b / (span * 1e-6) / 1e9 / measured_peaks()[0], 4),
            "note": ("first block start (past the wait for the previous kernel) to last block end, "
                     "from the kernel's global-timer trace (a traced handle per layer copy, same "
                     "weights), calls back to back; gap = last block end to the next call's first "
                     "block start (launch + wait)")}

# --------------------------------------------------------------------------- our arm

def run_ours(args, rank, world, local_rank, dist_on):
    import torch
    import int4_moe_expert_gb300 as moe

    wl = synth.WORKLOADS[args.workload]
    if wl.n_layers > 1:
        return run_stack(args, rank, world, local_rank, dist_on)
    if args.resident_experts:
        # profiling captures: same per-launch expert work, fewer experts resident
        import dataclasses
        wl = dataclasses.replace(wl, E=args.resident_experts, name=wl.name + f"_e{args.resident_experts}")
    if args.tokens:
        # a small decode batch (e.g. a speculative-verify batch) of the same layer
        import dataclasses
        wl = dataclasses.replace(wl, T=args.tokens, name=wl.name + f"_t{args.tokens}")
    T = wl.T
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    li = synth.layer_inputs(wl, experts=[0] if args.alias_experts else None)
    cfg = moe.make_config(wl.H, wl.E, wl.K, wl.I, wl.n_shared, wl.I_shared, wl.routed_scale,
                          wl.norm_topk, False, wl.rms_eps, n_group=wl.n_group, topk_group=wl.topk_group,
                          score_func=wl.score_func, cuda_cores=args.cuda_cores,
                          expert_format=wl.expert_format, shared_format=wl.shared_format)
    slabs, scales = li.slabs, li.scales
    if args.alias_experts:
        # profiling only: every expert pointer aliases expert 0's slab
        slabs, scales = li.slabs[:1], li.scales[:1]
    layer = moe.MoeLayer(cfg, li.router_w, li.router_b, slabs, scales, li.sh_slab,
                         li.sh_scale, max_tokens=T, expert_rows=[0] * wl.E if args.alias_experts else None)
    # further resident copies of the layer at distinct addresses (device-side copies of the
    # same weights): the timed steps walk them in rotation, so no step finds its weights in L2
    L = max(1, args.layer_copies)
    copies = [layer]
    for _ in range(L - 1):
        copies.append(moe.MoeLayer(cfg, *[None if t is None else t.clone() for t in
                                          (layer.router_w, layer.router_b, layer.slabs, layer.scales,
                                           layer.sh_slab, layer.sh_scale)],
                                   max_tokens=T, expert_rows=[0] * wl.E if args.alias_experts else None))
    streams = rank_streams(rank, world, N_X)
    xs_host = [synth.tokens(wl, T=T, stream=s) for s in streams]
    xs = [torch.from_numpy(x).to(dev) for x in xs_host]
    y = torch.empty((T, wl.H), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    flush_w = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    flush_r = torch.ones(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    sink = torch.empty(1, dtype=torch.float32, device=dev)

    def flush():
        flush_w.zero_()
        torch.sum(flush_r, dim=0, keepdim=True, out=sink)

    # routing of each rotated batch (for the algorithmic byte count)
    touched = []
    for x in xs:
        _, idx, _ = layer.forward_debug(x)
        touched.append(len(set(idx.cpu().numpy().ravel().tolist())))
    torch.cuda.synchronize()

    for i in range(args.warmup):
        moe.moe_forward(copies[i % L].handle, xs[i % N_X], T, y, stream)
    torch.cuda.synchronize()

    # the timed region: K steps back to back, copy i mod L and token batch i mod 16
    K = args.steps
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    barrier(dist_on)
    torch.cuda.synchronize()
    with ClockSampler(local_rank) as clk:
        t_start.record(stream)
        for i in range(K):
            moe.moe_forward(copies[i % L].handle, xs[i % N_X], T, y, stream)
        t_end.record(stream)
        torch.cuda.synchronize()
    barrier(dist_on)
    total_ms = reduce_max(t_start.elapsed_time(t_end), dist_on)
    for ly in copies:
        assert moe.moe_device_error(ly.handle) == 0

    # beside it (not the value): each step alone between two events, (a) in the same rotation
    # with no flush, (b) on one copy with L2 flushed before the step (outside the events)
    def per_step(n, flushed):
        e0 = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        e1 = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        for i in range(n):
            if flushed:
                flush()
            e0[i].record(stream)
            moe.moe_forward((copies[0] if flushed else copies[i % L]).handle, xs[i % N_X], T, y, stream)
            e1[i].record(stream)
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in zip(e0, e1)]
    n_side = min(K, 500)
    step_ms = per_step(n_side, False)
    step_ms_flushed = per_step(n_side, True)
    step_sorted = sorted(step_ms)
    step_stats = {"median_us": round(1e3 * statistics.median(step_ms), 2),
                  "p10_us": round(1e3 * step_sorted[len(step_sorted) // 10], 2),
                  "p90_us": round(1e3 * step_sorted[(9 * len(step_sorted)) // 10], 2),
                  "max_us": round(1e3 * step_sorted[-1], 2),
                  "note": f"{n_side} steps, each alone between two events (launch included), same rotation"}
    flushed_stats = {"median_us": round(1e3 * statistics.median(step_ms_flushed), 2),
                     "mean_us": round(1e3 * statistics.mean(step_ms_flushed), 2),
                     "note": (f"{n_side} steps on one copy, each between two events after an L2 flush "
                              "(256 MiB write + 256 MiB read, outside the events): the protocol of "
                              "earlier measurements")}
    assert moe.moe_device_error(layer.handle) == 0

    # One launch per step on the decode path (the step events bracket exactly that kernel);
    # otherwise router, gate/up, down (+ combine).
    # (up to moe_streaming_decode_max_tokens tokens: one single-token decode step per token)
    fused = T <= moe.moe_streaming_decode_max_tokens(layer.handle)
    kernel_span = kernel_span_stats(moe, cfg, copies, xs, y, T, stream, wl) if fused and T == 1 else None
    # launches per step: the fused kernel; or router, gate/up, down; or router (+ activation
    # conversion when T > 8), gate/up, down, combine; the tcgen05 path (T >= 256, int4) adds the
    # copy of the activations into its item-blocked layout
    # (T == 1 with an int8 expert runs the tensor-core flow: router, gate/up, down, combine)
    t1_tensor = T == 1 and (wl.expert_format != 0 or (wl.n_shared and wl.shared_format != 0))
    tc5 = (T >= 256 and not fused and wl.expert_format == 0 and (not wl.n_shared or wl.shared_format == 0)
           and bool(moe.moe_uses_tensor_cores(layer.handle)))
    kernels_per_step = T if fused else ((4 if t1_tensor else 3) if T == 1 else (4 if T <= 8 else 5) + (1 if tc5 else 0))
    stage_ms, n_calls, event_ms = None, 0, 0.0
    if not fused:
        # Per-kernel times: the same steps again with the library recording an
        # event at every kernel boundary (those events add GPU time and stop the
        # kernels overlapping, so this pass is kept out of the timed one above).
        n_prof = min(K, 4096)
        moe.moe_profile_start(layer.handle, n_prof)
        for i in range(n_prof):
            flush()
            moe.moe_forward(layer.handle, xs[i % N_X], T, y, stream)
        torch.cuda.synchronize()
        n_calls, stage_ms = moe.moe_profile_read(layer.handle)
        moe.moe_profile_start(layer.handle, 0)
        # GPU time one event boundary adds (two events back to back, cold L2)
        ea = [torch.cuda.Event(enable_timing=True) for _ in range(200)]
        eb = [torch.cuda.Event(enable_timing=True) for _ in range(200)]
        for i in range(200):
            flush()
            ea[i].record(stream)
            eb[i].record(stream)
        torch.cuda.synchronize()
        event_ms = statistics.median(a.elapsed_time(b) for a, b in zip(ea, eb))

    # end to end through the host entry point (pinned host buffers)
    xh = [torch.from_numpy(x).pin_memory() for x in xs_host]
    yh = torch.empty((T, wl.H), dtype=torch.float32).pin_memory()
    for i in range(min(args.warmup, 10)):
        moe.moe_forward_host(copies[i % L].handle, xh[i % N_X], T, yh, stream)
    barrier(dist_on)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(K):
        moe.moe_forward_host(copies[i % L].handle, xh[i % N_X], T, yh, stream)
    e2e_s = time.perf_counter() - t0
    e2e_s = reduce_max(e2e_s, dist_on)
    barrier(dist_on)

    tokens = world * K * T
    value = tokens / (total_ms / 1e3)
    ms_per_step = total_ms / K
    mean_touched = float(np.mean(touched))
    bytes_step = float(np.mean([step_bytes(wl, T, t) for t in touched]))
    peak, peak_kind = measured_peaks()
    if fused:
        # dominant (only) kernel: the whole step; its bytes are the step's bytes
        dom_kind = "fused"
        dom_name = ("decode_fused_kernel: router + top-k + gate/up + SwiGLU + down + combine, "
                    "one launch (programmatic dependent launch) per token, T=%d" % T)
        dom_bytes = bytes_step
        dom_ms = total_ms / K
        units = wl.K + wl.n_shared
    else:
        # dominant kernel: gate/up + SwiGLU over the touched experts + the shared one
        dom_kind = "gate_up"
        dom_name = "gate/up + SwiGLU (int4 GEMV/GEMM), T=%d" % T
        n_r = mean_touched if T > 1 else wl.K
        units = n_r + wl.n_shared
        dom_bytes = (n_r * gateup_bytes(wl.H, wl.I, wl.expert_format) +
                     (gateup_bytes(wl.H, wl.I_shared, wl.shared_format) if wl.n_shared else 0))
        dom_ms = stage_ms["gate_up"] - event_ms
    achieved = dom_bytes / (dom_ms / 1e3) / 1e9
    tensor = T > 1 and not fused and moe.moe_uses_tensor_cores(layer.handle)
    if tensor:
        # gate/up on the tensor cores: 2 FLOP per weight per (token, expert) pair
        dom_name = (("tc_expert_kernel<GU>: gate/up + SwiGLU on tcgen05 (warp-specialised: dequantised weights "
                     "in tensor memory as A, activations by bulk copy in shared memory, f32 accumulators in "
                     "tensor memory), T=%d") if tc5 else
                    "mma_expert_kernel<GU>: gate/up + SwiGLU on the tensor cores (mma.sync f16), T=%d") % T
        dom_flops = T * (wl.K * 4 * wl.I * wl.H + wl.n_shared * 4 * wl.I_shared * wl.H)
        tpeak, tpeak_kind = measured_tensor_peak()
        achieved_t = dom_flops / (dom_ms / 1e3) / 1e12
    out = None
    if rank == 0:
        out = {
            "metric": METRIC,
            "value": round(value, 2),
            "unit": "tokens/s",
            "n_gpus": world,
            "steps": K,
            "warmup": args.warmup,
            "ms_per_step": round(ms_per_step, 6),
            "step_time_distribution": step_stats,
            "step_time_flushed": flushed_stats,
            "kernel_span": kernel_span,
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": ("int4 x f16 -> f32 (tensor cores: tcgen05 for T >= 256, mma.sync below), "
                      "f32 router/scales/SwiGLU/combine" if tensor else
                      "int4 x fx16 -> s32 (exact dp4a sums), f32 router/scales/SwiGLU/combine" if fused else
                      "int4 x f32 -> f32 (CUDA cores), f32 router/scales/SwiGLU/combine"),
            "data": "synthetic (seeded SplitMix64; shapes and distributions of the workload)",
            "config": {
                "workload": workload_desc(wl),
                "tokens_per_step": T,
                "experts_resident_GB": round(wl.E * expert_bytes(wl.H, wl.I, wl.expert_format) / 1e9, 3),
                "l2": (f"not flushed: inputs larger than L2 -- {L} resident copies of the layer at distinct "
                       f"addresses ({round(L * wl.E * expert_bytes(wl.H, wl.I, wl.expert_format) / 1e9, 1)} GB "
                       "of experts), step i uses copy i mod L, so no step finds its weights in L2"),
                "layer_copies": L,
                "x_rotation": N_X,
                "parallelism": f"{world} independent replicas (no collective on the data path)",
            },
            "hbm": {
                "algorithmic_bytes_per_step": int(bytes_step),
                "achieved_gbs_per_step": round(bytes_step / (ms_per_step / 1e3) / 1e9, 1),
                "vs_8tbs": round(bytes_step / (ms_per_step / 1e3) / 8e12, 4),
                "vs_measured_peak": round(bytes_step / (ms_per_step / 1e3) / 1e9 / peak, 4),
                "mean_routed_experts_touched": mean_touched,
            },
            "roofline": {
                "kernel": dom_name,
                "bound": "hbm",
                "achieved": round(achieved, 1),
                "peak": peak,
                "peak_kind": peak_kind + " (MEASURED_PEAKS.json hbm_gbs, copy)" if peak_kind == "measured" else peak_kind,
                "unit": "GB/s",
                "frac": round(achieved / peak, 4),
                "traffic": recorded_traffic(dom_kind, wl.name, T),
                "algorithmic_bytes_per_launch": int(dom_bytes),
                "experts_per_launch": units,
                "launch_ms": round(dom_ms, 6),
                "launch_ms_source": ("timed span / K (K back-to-back launches between two events)" if fused else
                                     "profiled pass, event boundary time subtracted"),
            },
            "e2e": {
                "value": round(tokens / e2e_s, 2),
                "unit": "tokens/s",
                "h2d_bytes_per_step": T * wl.H * 4,
                "d2h_bytes_per_step": T * wl.H * 4,
                "api": "moe_forward_host (pinned host x/y, copies + step + stream sync), same rotation",
            },
            "gpu_launches": world * K * kernels_per_step,
            "clocks": clk.summary(),
        }
        if tensor and binding_roofline(achieved / peak, achieved_t / tpeak) == "hbm":
            out["roofline"]["tensor_view"] = {"achieved_tflops": round(achieved_t, 1), "peak_tflops": tpeak,
                                              "frac": round(achieved_t / tpeak, 4),
                                              "flops_per_launch": int(dom_flops)}
        elif tensor:
            out["roofline"] = {
                "kernel": dom_name,
                "bound": "tensor",
                "achieved": round(achieved_t, 1),
                "peak": tpeak,
                "peak_kind": tpeak_kind,
                "unit": "TFLOP/s",
                "frac": round(achieved_t / tpeak, 4),
                "traffic": None,
                "flops_per_launch": int(dom_flops),
                "launch_ms": round(dom_ms, 6),
                "launch_ms_source": "profiled pass, event boundary time subtracted",
                "hbm_view": {"achieved_gbs": round(achieved, 1), "peak_gbs": peak,
                             "frac": round(achieved / peak, 4), "algorithmic_bytes_per_launch": int(dom_bytes)},
                "note": ("peak: the measured cuBLAS bf16 rate (f16 runs at the same rate); on this GPU "
                         "mma.sync reaches ~600 TFLOP/s in a register-only loop, and one tcgen05.mma of "
                         "M 128 x K 16 costs ~33-36 ns per SM for any N <= 128 when issued back to back "
                         "(2.2 PFLOP/s at N 128)"),
            }
        if stage_ms is not None:
            out["stages_ms"] = {k: round(v, 6) for k, v in stage_ms.items()}
            out["stages_note"] = ("separate pass with an event at each kernel boundary; "
                                  "event_boundary_ms (two events back to back) is subtracted from "
                                  "roofline.launch_ms")
            out["event_boundary_ms"] = round(event_ms, 6)
            out["stages_calls"] = n_calls
        if world == 1 and not args.no_cpu_baseline:
            out["cpu_baseline"] = cpu_baseline(wl, li, xs_host, args.cpu_seconds)
    for ly in copies:
        ly.close()
    return out


def run_stack(args, rank, world, local_rank, dist_on):
    """The chained decode stack (x <- x + moe(rmsnorm(x)) over n_layers layers, T=1,
    every layer's experts resident): one step = one token through every layer.  The
    chain of moe_forward calls is captured once in a CUDA graph (layer 0 reads a
    static input buffer, the layers alternate between two activation buffers) and
    replayed per step; the same chain launched call by call is timed beside it."""
    import torch
    import int4_moe_expert_gb300 as moe

    wl = synth.WORKLOADS[args.workload]
    L = wl.n_layers
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    cfg = moe.make_config(wl.H, wl.E, wl.K, wl.I, wl.n_shared, wl.I_shared, wl.routed_scale,
                          wl.norm_topk, True, wl.rms_eps)
    streams = rank_streams(rank, world, N_X)
    xs_host = [synth.tokens(wl, T=1, stream=s) for s in streams]
    # the oracle baseline runs while the layers are generated (one layer's weights on the
    # host at a time): the first N_CPU rotated tokens through the whole chain
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        cpu = {"x": [x[0].astype(np.float64) for x in xs_host[:8]], "s": 0.0}
    layers = []
    for l in range(L):
        li = synth.layer_inputs(wl, layer=l)
        layers.append(moe.MoeLayer(cfg, li.router_w, li.router_b, li.slabs, li.scales, li.sh_slab,
                                   li.sh_scale, max_tokens=1))
        if cpu is not None:
            ref = oracle.LayerRef.from_inputs(oracle.cfg_from_workload(wl), li)
            t0 = time.perf_counter()
            cpu["x"] = [ref.token(x)[0] for x in cpu["x"]]
            cpu["s"] += time.perf_counter() - t0
            del ref
        del li
    fused = all(moe.moe_uses_streaming_decode(ly.handle) for ly in layers)
    xs = [torch.from_numpy(x).to(dev) for x in xs_host]
    x_in = torch.empty((1, wl.H), dtype=torch.float32, device=dev)
    act = [torch.empty((1, wl.H), dtype=torch.float32, device=dev) for _ in range(2)]
    y_out = act[(L - 1) % 2]
    flush_w = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    flush_r = torch.ones(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    sink = torch.empty(1, dtype=torch.float32, device=dev)

    def flush():
        flush_w.zero_()
        torch.sum(flush_r, dim=0, keepdim=True, out=sink)

    def chain(stream=None):
        for l, ly in enumerate(layers):
            moe.moe_forward(ly.handle, x_in if l == 0 else act[(l - 1) % 2], 1, act[l % 2], stream)

    x_in.copy_(xs[0])
    chain()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        chain()
    stream = torch.cuda.current_stream()
    for i in range(args.warmup):
        x_in.copy_(xs[i % N_X])
        graph.replay()
    torch.cuda.synchronize()

    # the timed region: K tokens back to back (each: its input copied in, the 40 layers replayed);
    # a token reads 40 distinct layers (16 GB resident), so no step finds its weights in L2
    K = args.steps
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    barrier(dist_on)
    torch.cuda.synchronize()
    with ClockSampler(local_rank) as clk:
        t_start.record(stream)
        for i in range(K):
            x_in.copy_(xs[i % N_X])
            graph.replay()
        t_end.record(stream)
        torch.cuda.synchronize()
    barrier(dist_on)
    total_ms = reduce_max(t_start.elapsed_time(t_end), dist_on)
    # beside it: each token alone between two events after an L2 flush (outside the events)
    n_side = min(K, 200)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_side)]
    for i in range(n_side):
        flush()
        x_in.copy_(xs[i % N_X])
        ev[i][0].record(stream)
        graph.replay()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    step_sorted = sorted(step_ms)
    for ly in layers:
        assert moe.moe_device_error(ly.handle) == 0

    # the same chain, one launch call per layer (no graph)
    n_eager = min(K, 200)
    ev_e = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_eager)]
    for i in range(n_eager):
        flush()
        x_in.copy_(xs[i % N_X])
        ev_e[i][0].record(stream)
        chain(stream)
        ev_e[i][1].record(stream)
    torch.cuda.synchronize()
    eager_ms = statistics.median(a.elapsed_time(b) for a, b in ev_e)

    # end to end: pinned host token in, graph replay, pinned host result out
    xh = [torch.from_numpy(x).pin_memory() for x in xs_host]
    yh = torch.empty((1, wl.H), dtype=torch.float32).pin_memory()
    barrier(dist_on)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(K):
        x_in.copy_(xh[i % N_X], non_blocking=True)
        graph.replay()
        yh.copy_(y_out, non_blocking=True)
        stream.synchronize()
    e2e_s = time.perf_counter() - t0
    e2e_s = reduce_max(e2e_s, dist_on)
    barrier(dist_on)

    tokens = world * K
    value = tokens / (total_ms / 1e3)
    ms_per_step = total_ms / K
    layer_bytes = step_bytes(wl, 1, wl.K)
    bytes_step = L * layer_bytes
    peak, peak_kind = measured_peaks()
    layer_ms = ms_per_step / L
    achieved = layer_bytes / (layer_ms / 1e3) / 1e9
    out = None
    if rank == 0:
        out = {
            "metric": METRIC,
            "value": round(value, 2),
            "unit": "tokens/s",
            "n_gpus": world,
            "steps": K,
            "warmup": args.warmup,
            "ms_per_step": round(ms_per_step, 6),
            "step_time_flushed": {"median_us": round(1e3 * statistics.median(step_ms), 2),
                                  "p10_us": round(1e3 * step_sorted[len(step_sorted) // 10], 2),
                                  "p90_us": round(1e3 * step_sorted[(9 * len(step_sorted)) // 10], 2),
                                  "max_us": round(1e3 * step_sorted[-1], 2),
                                  "note": (f"{n_side} tokens, each alone between two events after an L2 "
                                           "flush (256 MiB write + 256 MiB read, outside the events)")},
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "int4 x fx16 -> s32 (exact dp4a sums), f32 router/scales/SwiGLU/combine/rmsnorm",
            "data": "synthetic (seeded SplitMix64; shapes and distributions of the workload)",
            "config": {
                "workload": workload_desc(wl),
                "tokens_per_step": 1,
                "experts_resident_GB": round(L * wl.E * expert_bytes(wl.H, wl.I) / 1e9, 3),
                "l2": (f"not flushed: inputs larger than L2 -- each token reads all {L} layers "
                       f"({round(L * wl.E * expert_bytes(wl.H, wl.I) / 1e9, 1)} GB resident), tokens back to back"),
                "x_rotation": N_X,
                "launch": (f"the {L} moe_forward calls captured once in a CUDA graph, replayed per step "
                           "(after a device copy of the step's token into the graph's input buffer)"),
                "parallelism": f"{world} independent replicas (no collective on the data path)",
            },
            "hbm": {
                "algorithmic_bytes_per_step": int(bytes_step),
                "achieved_gbs_per_step": round(bytes_step / (ms_per_step / 1e3) / 1e9, 1),
                "vs_8tbs": round(bytes_step / (ms_per_step / 1e3) / 8e12, 4),
                "vs_measured_peak": round(bytes_step / (ms_per_step / 1e3) / 1e9 / peak, 4),
                "routed_experts_per_layer": wl.K,
            },
            "roofline": {
                "kernel": ("decode_fused_kernel: one launch per layer (programmatic dependent launch), T=1" if fused else
                           "per-layer kernels, T=1"),
                "bound": "hbm",
                "achieved": round(achieved, 1),
                "peak": peak,
                "peak_kind": peak_kind + " (MEASURED_PEAKS.json hbm_gbs, copy)" if peak_kind == "measured" else peak_kind,
                "unit": "GB/s",
                "frac": round(achieved / peak, 4),
                "traffic": None,
                "algorithmic_bytes_per_launch": int(layer_bytes),
                "experts_per_launch": wl.K + wl.n_shared,
                "launch_ms": round(layer_ms, 6),
                "launch_ms_source": f"timed span / (K x {L}) (includes the gaps between the kernels and the input copy)",
            },
            "eager_chain": {"ms_per_step": round(eager_ms, 6),
                            "note": f"the same {L} calls launched one by one (median of {n_eager} steps)"},
            "e2e": {
                "value": round(tokens / e2e_s, 2),
                "unit": "tokens/s",
                "h2d_bytes_per_step": wl.H * 4,
                "d2h_bytes_per_step": wl.H * 4,
                "api": f"moe_forward x {L} captured in a CUDA graph; pinned host token in, result out, stream sync per token",
            },
            "gpu_launches": world * K * L * (1 if fused else 4),
            "clocks": clk.summary(),
        }
        if cpu is not None:
            n = len(cpu["x"])
            out["cpu_baseline"] = {
                "value": round(n / cpu["s"], 4), "unit": "tokens/s", "cores": oracle.threads(),
                "kind": "oracle",
                "sample": f"{n} tokens through all {L} layers of the same chain in the double-precision "
                          f"C oracle, OpenMP over output rows ({cpu['s']:.1f} s; weights generated "
                          f"outside the timed part)"}
    for ly in layers:
        ly.close()
    return out


def cpu_baseline(wl, li, xs_host, seconds):
    """The oracle, as it stands, on this host's cores over a bounded sample of
    the same workload (whole tokens through the layer in double precision), and
    the same on one core for a quarter of the time."""
    import oracle
    ref = oracle.LayerRef.from_inputs(oracle.cfg_from_workload(wl), li)

    def timed(budget):
        n_tok, i, t0 = 0, 0, time.perf_counter()
        while True:
            ref.forward(xs_host[i % len(xs_host)])
            n_tok += xs_host[0].shape[0]
            i += 1
            el = time.perf_counter() - t0
            if el >= budget or i >= 4096:
                return n_tok, i, el

    cores = oracle.threads()
    n_tok, i, el = timed(seconds)
    oracle.set_threads(1)
    try:
        n1, i1, el1 = timed(seconds / 4)
    finally:
        oracle.set_threads(cores)
    return {"value": round(n_tok / el, 4), "unit": "tokens/s", "cores": cores,
            "kind": "oracle",
            "sample": f"{n_tok} tokens ({i} calls of T={xs_host[0].shape[0]}) of the same layer "
                      f"through the double-precision C oracle, OpenMP over output rows, {el:.1f} s",
            "single_core": {"value": round(n1 / el1, 4), "unit": "tokens/s", "cores": 1,
                            "sample": f"{n1} tokens ({i1} calls), one thread, {el1:.1f} s"}}


# --------------------------------------------------------------------------- reference arm

def run_reference(args, world):
    """The oracle on the host cores, same workload and metric.  One step is one
    expert of one token (router included in a token's first step), so K steps
    stay within minutes; tokens = steps / (K + n_shared)."""
    import oracle
    wl = synth.WORKLOADS[args.workload]
    if wl.n_layers > 1:
        raise SystemExit("--impl reference times single-layer workloads")
    T = 1
    J = wl.K + wl.n_shared
    cfg = oracle.cfg_from_workload(wl)
    li = synth.layer_inputs(wl)
    ref = oracle.LayerRef.from_inputs(cfg, li)
    xs = [synth.tokens(wl, T=1, stream=s)[0].astype(np.float64) for s in range(N_X)]

    state = {"idx": None}

    def step(s):
        u, j = divmod(s, J)
        x = xs[u % N_X]
        if j == 0:
            state["idx"], _, _, _ = oracle.route(cfg, ref.router_w, ref.router_b, x)
        if j < wl.K:
            e = int(state["idx"][j])
            oracle.expert(wl.H, wl.I, li.slabs[e], li.scales[e], x)
        else:
            oracle.expert(wl.H, wl.I_shared, li.sh_slab, li.sh_scale, x)

    for s in range(args.warmup):
        step(s)
    t0 = time.perf_counter()
    for s in range(args.steps):
        step(s)
    el = time.perf_counter() - t0
    tokens = args.steps / J * T
    value = tokens / el
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 4),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(el / args.steps * 1e3, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded SplitMix64; shapes and distributions of the workload)",
        "config": {"workload": workload_desc(wl), "tokens_per_step": 1.0 / J,
                   "step": f"one of the {J} experts of one token (router on the token's first step)"},
        "cpu_baseline": {"kind": "oracle", "cores": oracle.threads(), "value": round(value, 4),
                         "unit": "tokens/s",
                         "sample": f"{args.steps} steps = {tokens:.1f} tokens of the layer in the "
                                   f"double-precision C oracle"},
        "e2e": {"value": round(value, 4), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


# --------------------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="glm_decode", choices=list(synth.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--alias-experts", action="store_true",
                    help="profiling only: all routed experts share one slab (router captures)")
    ap.add_argument("--tokens", type=int, default=0,
                    help="tokens per step instead of the workload's T (small decode batches)")
    ap.add_argument("--cuda-cores", action="store_true",
                    help="T > 1 on the CUDA-core kernels instead of the tensor cores (comparison)")
    ap.add_argument("--resident-experts", type=int, default=0,
                    help="profiling only: keep this many routed experts resident instead of E")
    ap.add_argument("--layer-copies", type=int, default=8,
                    help="resident copies of a single-layer workload, used in rotation (1: one copy)")
    args = ap.parse_args()
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world != args.gpus:
        raise SystemExit(f"--gpus {args.gpus} but WORLD_SIZE={world}")

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, world)), flush=True)
        return

    dist_on = world > 1
    if dist_on:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    out = run_ours(args, rank, world, local_rank, dist_on)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if dist_on:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
