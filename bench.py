#!/usr/bin/env python3
"""Benchmark of the MoE stage1 + combine hot path on GB300.

One step = the whole hot path over one batch of T tokens: routing layout
(moe_route_layout) -> quant + dispatch -> GEMM1 -> weighted combine, all in the
library's kernels on one stream, inputs resident in HBM.  Three variants of
the step are timed (--variant picks the one behind `value`): unfused
(moe_dispatch_quant, moe_grouped_gemm1, moe_combine), fused (moe_stage1 +
moe_combine) and overlap (moe_dispatch_quant + moe_grouped_gemm1_combine).  Default workload: T=8192 tokens, H=7168, 256 experts in 8
groups, top-8, GEMM1 N=4096, Zipf(1.2) expert popularity (synthetic, seeded).

Prints ONE JSON line (rank 0).  `value` is tokens/s of the step; per-kernel
microseconds, GEMM1 TFLOP/s and dispatch/combine GB/s ride along.  `--impl
reference` times the CPU oracle on a bounded sample of the same workload.

Multi-GPU: replicas only (every rank runs the same single-GPU workload; the
path has no data exchange), launched by torchrun; the max over ranks of the
timed region gives the whole-job throughput.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "stage1 µs & tokens/s at T=8192 (GEMM1 TFLOP/s); dispatch/combine HBM GB/s"

# DRAM bytes per launch of the roofline kernel (dram__bytes_read.sum + dram__bytes_write.sum) from one
# single-pass ncu capture of the full workload (the only metrics captured at full size: ncu reports
# "1 pass" for this metric set on the small profile_t8192_e32 workload, so nothing is saved or restored
# around the launch), keyed by workload, step variant and a hash of the code of every kernel source
# (comments aside).  A kernel changed since then reports null until captured again:
#   ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum,gpu__time_duration.sum --clock-control none \
#       -k regex:grouped_gemm1_kernel -s 3 -c 1 --csv --log-file traffic.csv \
#       python bench.py --steps 2 --warmup 3 --no-cpu-baseline --no-clocks
TRAFFIC = {("t8192_zipf1.2", "unfused", "8b4fdafdca1d9a95"): 6.507e9}


# Sources the dominant kernel (grouped_gemm1_kernel) is built from.
GEMM1_SOURCES = ["gemm1.cu", "gemm1.cuh", "common.cuh", "tmem_fold.cuh", "host_util.h"]


def kernel_source_hash() -> str:
    """Hash of the dominant kernel's sources' code: comments and blank space
    removed, so a comment edit keeps a capture valid and any code edit
    invalidates it."""
    import hashlib
    import re
    h = hashlib.sha1()
    csrc = os.path.join(ROOT, "combine_counting_sort_gb300", "csrc")
    for path in [os.path.join(csrc, f) for f in GEMM1_SOURCES]:
        with open(path) as fh:
            code = fh.read()
        code = re.sub(r"/\*.*?\*/", "", code, flags=re.S)
        code = re.sub(r"//[^\n]*", "", code)
        h.update(" ".join(code.split()).encode())
    return h.hexdigest()[:16]
UNIT = "tokens/s"
L2_FLUSH_BYTES = 512 << 20          # > 129 MB L2
FP8_OVER_BF16 = 2.0                 # nominal dense fp8 / bf16 tensor ratio (4.5 / 2.25 PFLOP/s)


# ---------------------------------------------------------------- distributed plumbing

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def reduce_max(value: float, world: int, device) -> float:
    """Max over ranks of a per-rank float (identity on one rank)."""
    if world <= 1:
        return value
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------- clocks

CLOCK_FIELDS = ["index", "clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
                "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
                "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]


class ClockSampler:
    """nvidia-smi sampled every 200 ms during the timed region."""

    def __init__(self, gpu_index: int, enabled: bool = True):
        self.p = None
        self.gpu = gpu_index
        if enabled:
            try:
                self.p = subprocess.Popen(
                    ["nvidia-smi", "-i", str(gpu_index), "--query-gpu=" + ",".join(CLOCK_FIELDS),
                     "--format=csv,noheader,nounits", "-lms", "200"],
                    stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            except OSError:
                self.p = None

    def stop(self) -> dict:
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["not sampled"]}
        time.sleep(0.25)
        self.p.terminate()
        out, _ = self.p.communicate(timeout=10)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < len(CLOCK_FIELDS):
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


PEAK_RULE = ("burst unless the timed region lasted >= 1 s and nvidia-smi saw sw_power_cap during it "
             "(then the power-capped sustained peak)")


def roofline_peak_kind(wall_s: float, clk: dict) -> str:
    """Which measured peak is the roofline denominator: the burst peak for a
    short timed region at full clocks, the sustained (power-capped) one only
    when the region was long enough to reach the power cap and the clock
    samples show it."""
    capped = "sw_power_cap" in (clk.get("reasons") or [])
    return "sustained" if (wall_s >= 1.0 and capped) else "burst"


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# ---------------------------------------------------------------- the GPU arm

class Workload:
    """Device-resident inputs and buffers of one workload."""

    def __init__(self, cfg, device, stage1_opts):
        import combine_counting_sort_gb300 as moe
        from combine_counting_sort_gb300 import inputs
        self.moe, self.cfg, self.dev = moe, cfg, device
        T, H, E, G, k, N = cfg.T, cfg.H, cfg.E, cfg.G, cfg.k, cfg.N
        self.R = T * k
        self.x = inputs.make_x(T, H, cfg.seed).to(device)
        logits = inputs.make_logits(T, E, cfg.zipf, cfg.seed).to(device)
        self.ids = torch.empty(T, k, dtype=torch.int32, device=device)
        self.w = torch.empty(T, k, dtype=torch.float32, device=device)
        moe.moe_router_topk(logits, k, self.ids, self.w)
        W = inputs.make_weights(E, N, H, cfg.seed, device=device)
        self.Wq = torch.empty(E, N, H, dtype=torch.uint8, device=device)
        self.Ws = torch.empty(E, N // 128, H // 128, dtype=torch.float32, device=device)
        moe.moe_quant_weights(W, self.Wq, self.Ws)
        # the MXFP8 variant's weights (e8m0 scales per 32 values), timed beside the fp32-scale path
        self.Wq_mx = torch.empty(E, N, H, dtype=torch.uint8, device=device)
        self.W_sf = torch.empty(moe.mx_sf_w_shape(E, N, H), dtype=torch.uint8, device=device)
        moe.moe_quant_weights_mx(W, self.Wq_mx, self.W_sf)
        torch.cuda.synchronize(device)
        del W
        self.L = moe.Layout(T, k, E, G, device=device)
        self.A = torch.empty(self.R, H, dtype=torch.uint8, device=device)
        self.As = torch.empty(H // 128, self.R, dtype=torch.float32, device=device)
        self.Y = torch.empty(self.R, N, dtype=torch.bfloat16, device=device)
        self.out = torch.empty(T, N, dtype=torch.bfloat16, device=device)
        self.ws = torch.empty(int(self.L.sizes.stage1_ws_bytes), dtype=torch.uint8, device=device)
        self.ws_gc = torch.empty(int(self.L.sizes.gemm_combine_ws_bytes), dtype=torch.uint8, device=device)
        self.runs = moe.SendRuns(self.L, device=device)
        self.A_send = torch.empty(self.runs.max_rows, H, dtype=torch.uint8, device=device)
        self.As_send = torch.empty(H // 128, self.runs.max_rows, dtype=torch.float32, device=device)
        self.A_mx = torch.empty(self.R, H, dtype=torch.uint8, device=device)
        self.A_sf = torch.empty(moe.mx_sf_a_shape(self.L, H), dtype=torch.uint8, device=device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        self.opts = stage1_opts
        self.flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
        torch.cuda.empty_cache()

    def calls(self, s, variant, ids=None, w=None):
        """The step's calls in order, as (part name, thunk) pairs, on stream s:
        fused    layout | stage1 (one launch: quant + dispatch + GEMM1) | combine
        unfused  layout | dispatch | GEMM1 | combine
        overlap  layout | dispatch | GEMM1 with the combine overlapped (one launch)"""
        moe = self.moe
        ids = self.ids if ids is None else ids
        w = self.w if w is None else w
        layout = ("layout", lambda: moe.moe_route_layout(ids, w, self.L, self.status, stream=s))
        dispatch = ("dispatch", lambda: moe.moe_dispatch_quant(self.x, self.L, self.A, self.As, self.status, stream=s))
        gemm1 = ("gemm1", lambda: moe.moe_grouped_gemm1(self.A, self.As, self.Wq, self.Ws, self.L, self.Y, self.status,
                                                        stream=s))
        combine = ("combine", lambda: moe.moe_combine(self.Y, self.L, self.out, self.status, stream=s))
        if variant == "fused":
            return [layout, ("stage1", lambda: moe.moe_stage1(self.x, self.L, self.Wq, self.Ws, self.A, self.As, self.Y,
                                                              self.ws, self.status, self.opts, stream=s)), combine]
        if variant == "unfused":
            return [layout, dispatch, gemm1, combine]
        if variant == "overlap":
            return [layout, dispatch, ("gemm1_combine", lambda: moe.moe_grouped_gemm1_combine(
                self.A, self.As, self.Wq, self.Ws, self.L, self.Y, self.out, self.ws_gc, self.status, stream=s))]
        raise ValueError(variant)

    def step(self, s, variant, ev=None, ids=None, w=None):
        """One pass of the hot path on stream s; ev: one event before each call and one after the last."""
        calls = self.calls(s, variant, ids, w)
        for i, (_, fn) in enumerate(calls):
            if ev: ev[i].record(s)
            fn()
        if ev: ev[len(calls)].record(s)

    def flush_l2(self, s):
        with torch.cuda.stream(s):
            self.flush.zero_()

    # algorithmic work per launch
    def gemm_flops(self):
        return 2.0 * self.R * self.cfg.N * self.cfg.H

    def dispatch_bytes(self):
        c = self.cfg
        return 2.0 * c.T * c.H + self.R * c.H + 4.0 * self.R * c.H / 128

    def dispatch_bytes_mx(self):
        c = self.cfg
        return 2.0 * c.T * c.H + self.R * c.H + self.R * c.H / 32

    def combine_bytes(self):
        c = self.cfg
        return 2.0 * self.R * c.N + 2.0 * c.T * c.N + 8.0 * self.R


VARIANTS = ["fused", "unfused", "overlap"]
ROOFLINE_PART = {"fused": ("stage1", "stage1_kernel"), "unfused": ("gemm1", "grouped_gemm1_kernel"),
                 "overlap": ("gemm1_combine", "grouped_gemm1_combine_kernel")}


def timed_loop(wl, s, steps, variant):
    """`steps` steps of `variant`, the L2 flushed before each (outside the events).
    Returns (per-step ms, {part: [ms per step]})."""
    names = [n for n, _ in wl.calls(s, variant)]
    evs = []
    for _ in range(steps):
        wl.flush_l2(s)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)]
        wl.step(s, variant, ev)
        evs.append(ev)
    torch.cuda.synchronize()
    step_ms = [e[0].elapsed_time(e[-1]) for e in evs]
    parts = {n: [e[i].elapsed_time(e[i + 1]) for e in evs] for i, n in enumerate(names)}
    return step_ms, parts


def run_gpu(args):
    import combine_counting_sort_gb300 as moe
    from combine_counting_sort_gb300 import inputs
    import __graft_entry__ as ge

    rank, world, local = dist_env()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    ge.build()
    cfg = inputs.CONFIGS[args.workload]
    opts = moe.stage1_opts(comm_sms=args.comm_sms, flags=args.flags, schedule=args.schedule,
                           producers_join=args.join)
    wl = Workload(cfg, device, opts)
    s = torch.cuda.Stream(device)
    variant = args.variant

    for v in VARIANTS:            # every variant warmed up (each is timed below)
        for _ in range(args.warmup):
            wl.flush_l2(s)
            wl.step(s, v)
    torch.cuda.synchronize()
    if wl.status.item() != 0:
        raise RuntimeError(f"device status {moe.status_string(wl.status.item())} after warm-up")

    # ---- timed region: exactly K steps, barrier + sync on both sides
    barrier(world)
    torch.cuda.synchronize()
    clocks = ClockSampler(local, enabled=not args.no_clocks)
    t_wall = time.perf_counter()
    step_ms, parts = timed_loop(wl, s, args.steps, variant)
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall
    barrier(world)
    clk = clocks.stop()
    if wl.status.item() != 0:
        raise RuntimeError(f"device status {moe.status_string(wl.status.item())} in the timed region")
    total_ms = reduce_max(sum(step_ms), world, device)
    ms_per_step = total_ms / args.steps
    value = world * cfg.T / (ms_per_step / 1e3)

    # ---- the other step variants on the same inputs, for comparison (not part of `value`)
    med = lambda xs: statistics.median(xs)
    variants = {variant: {"ms_per_step": round(statistics.mean(step_ms), 4),
                          "parts_us": {n: round(med(v) * 1e3, 1) for n, v in parts.items()}}}
    vparts = {variant: parts}
    for v in VARIANTS:
        if v == variant:
            continue
        sm, pt = timed_loop(wl, s, max(3, args.steps // 2), v)
        variants[v] = {"ms_per_step": round(statistics.mean(sm), 4),
                       "parts_us": {n: round(med(x) * 1e3, 1) for n, x in pt.items()}}
        vparts[v] = pt
    if wl.status.item() != 0:
        raise RuntimeError(f"device status {moe.status_string(wl.status.item())} in the variant runs")
    u = vparts["unfused"]
    u_disp, u_gemm, u_comb = med(u["dispatch"]), med(u["gemm1"]), med(u["combine"])
    st1 = med(vparts["fused"]["stage1"])
    gc = med(vparts["overlap"]["gemm1_combine"])

    # ---- the MXFP8 variant on the same step's layout: dispatch and block-scaled GEMM1
    mx = run_mx_variant(wl, s, max(3, args.steps // 2))
    # ---- the per-(token, group) send runs: their dispatch and GEMM1 gathering A rows
    runs = run_runs_variant(wl, s, max(3, args.steps // 2))
    # ---- GEMM1 on CTA pairs (cta_group::2) on the same dispatch buffer
    pair = run_pair_variant(wl, s, max(3, args.steps // 2))

    # ---- end to end through the public API with host buffers: H2D inputs, D2H output
    e2e = run_e2e(wl, s, args, world, device)

    peaks = measured_peaks()
    fp8_burst = peaks["bf16_tflops"] * FP8_OVER_BF16
    fp8_sustained = peaks["bf16_tflops_sustained"] * FP8_OVER_BF16
    peak_kind = roofline_peak_kind(t_wall, clk)
    fp8_peak = fp8_sustained if peak_kind == "sustained" else fp8_burst
    part, kernel = ROOFLINE_PART[variant]
    roof_ms = statistics.mean(parts[part])
    variant_key = variant if variant != "fused" else "fused/comm%d/%s/%s/join%d" % (
        args.comm_sms, ["per_tile", "per_expert"][args.flags], ["expert_major", "ready_first"][args.schedule],
        args.join)
    traffic = args.traffic if args.traffic is not None else \
        TRAFFIC.get((cfg.name, variant_key, kernel_source_hash()))
    achieved = wl.gemm_flops() / (roof_ms / 1e3) / 1e12
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "fp8_e4m3 (fp32 accumulate, bf16 out)",
        "data": "synthetic (seeded: x~N(0,1) bf16, logits~N(0,1)+Zipf bias, W1~N(0,1/H) quantised on device)",
        "config": {"workload": cfg.name, "T": cfg.T, "H": cfg.H, "E": cfg.E, "G": cfg.G, "k": cfg.k, "N": cfg.N,
                   "zipf": cfg.zipf, "variant": variant,
                   "step": " | ".join(n for n, _ in wl.calls(s, variant)),
                   "stage1_opts": {"comm_sms": args.comm_sms, "flags": ["per_tile", "per_expert"][args.flags],
                                   "schedule": ["expert_major", "ready_first"][args.schedule],
                                   "producers_join": args.join},
                   "l2": "flushed between steps (512 MiB write, outside the step events)",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": {"kernel": kernel, "bound": "tensor",
                     "achieved": round(achieved, 1), "peak": round(fp8_peak, 1), "unit": "TFLOP/s",
                     "frac": round(achieved / fp8_peak, 4),
                     "work": "2*T*k*N*H GEMM1 flops (valid rows) / mean duration of the %s call" % part,
                     "peak_kind": peak_kind,
                     "peak_source": f"{peaks['source']} bf16 {peak_kind} x {FP8_OVER_BF16} (fp8/bf16 nominal); "
                                    + PEAK_RULE,
                     "peak_burst": round(fp8_burst, 1), "frac_of_burst": round(achieved / fp8_burst, 4),
                     "peak_sustained": round(fp8_sustained, 1),
                     "frac_of_sustained": round(achieved / fp8_sustained, 4),
                     "traffic": traffic,
                     "traffic_source": "ncu dram__bytes_read.sum + dram__bytes_write.sum, one full-size launch"
                     if traffic is not None else None},
        "parts_us": variants[variant]["parts_us"],
        "variants": variants,
        "layout_us": round(med(parts["layout"]) * 1e3, 1),
        "stage1_us": round(st1 * 1e3, 1),
        "unfused_us": {"dispatch": round(u_disp * 1e3, 1), "gemm1": round(u_gemm * 1e3, 1),
                       "sum": round((u_disp + u_gemm) * 1e3, 1)},
        "combine_us": round(u_comb * 1e3, 1),
        "gemm1_combine_us": round(gc * 1e3, 1),
        "gemm1_plus_combine_us": round((u_gemm + u_comb) * 1e3, 1),
        "gemm1_tflops": round(wl.gemm_flops() / (u_gemm / 1e3) / 1e12, 1),
        "stage1_tflops": round(wl.gemm_flops() / (st1 / 1e3) / 1e12, 1),
        "dispatch_gbs": round(wl.dispatch_bytes() / (u_disp / 1e3) / 1e9, 1),
        "combine_gbs": round(wl.combine_bytes() / (u_comb / 1e3) / 1e9, 1),
        "hbm_peak_gbs": peaks["hbm_gbs"],
        "mx": dict(mx, gemm1_tflops=round(wl.gemm_flops() / (mx["gemm1_us"] / 1e6) / 1e12, 1),
                   gemm1_frac_of_burst=round(wl.gemm_flops() / (mx["gemm1_us"] / 1e6) / 1e12 / fp8_burst, 4),
                   dispatch_gbs=round(wl.dispatch_bytes_mx() / (mx["dispatch_us"] / 1e6) / 1e9, 1)),
        "send_runs": runs,
        "gemm1_pair": dict(pair, gemm1_tflops=round(wl.gemm_flops() / (pair["gemm1_us"] / 1e6) / 1e12, 1),
                           gemm1_frac_of_burst=round(wl.gemm_flops() / (pair["gemm1_us"] / 1e6) / 1e12 / fp8_burst,
                                                     4)),
        "e2e": e2e,
        "gpu_launches": len(parts) * args.steps,
        "clocks": clk,
        "wall_s_timed_region": round(t_wall, 3),
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(cfg, args.cpu_budget_s)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_runs_variant(wl, s, reps):
    """The per-(token, group) send runs on the step's layout: the send-run
    layout, the dispatch into the runs and GEMM1 gathering its A rows from
    them (median CUDA-event times, the L2 flushed before every launch), with
    the dispatch's algorithmic bytes beside the dense dispatch's."""
    moe, c = wl.moe, wl.cfg
    moe.moe_route_layout(wl.ids, wl.w, wl.L, wl.status, stream=s)
    lay = _time_events(lambda: moe.moe_send_layout(wl.ids, wl.L, wl.runs, wl.status, stream=s), s, reps, wl.flush)
    d = _time_events(lambda: moe.moe_dispatch_quant_runs(wl.x, wl.L, wl.runs, wl.A_send, wl.As_send, wl.status,
                                                         stream=s), s, reps, wl.flush)
    g = _time_events(lambda: moe.moe_grouped_gemm1_gather(wl.A_send, wl.As_send, wl.Wq, wl.Ws, wl.L, wl.runs, wl.Y,
                                                          wl.status, stream=s), s, reps, wl.flush)
    torch.cuda.synchronize()
    if wl.status.item() != 0:
        raise RuntimeError(f"device status {moe.status_string(wl.status.item())} in the send-run variant")
    rows = int(wl.runs["run_offset"][-1].item())
    bytes_runs = 2.0 * c.T * c.H + rows * c.H + 4.0 * rows * c.H / 128
    return {"send_rows": rows, "send_rows_per_token": round(rows / c.T, 3), "layout_us": round(lay, 1),
            "dispatch_us": round(d, 1), "dispatch_bytes": bytes_runs,
            "dense_dispatch_bytes": wl.dispatch_bytes(),
            "dispatch_bytes_ratio": round(wl.dispatch_bytes() / bytes_runs, 3),
            "dispatch_gbs": round(bytes_runs / (d / 1e6) / 1e9, 1),
            "gemm1_gather_us": round(g, 1),
            "gemm1_gather_tflops": round(wl.gemm_flops() / (g / 1e6) / 1e12, 1)}


def run_mx_variant(wl, s, reps):
    """The MXFP8 variant (e8m0 scales per 32 values, block-scaled tcgen05 MMA)
    on the step's layout: median CUDA-event times of its dispatch and its
    GEMM1 over `reps` launches each, the L2 flushed before every launch."""
    moe = wl.moe
    moe.moe_route_layout(wl.ids, wl.w, wl.L, wl.status, stream=s)
    d = _time_events(lambda: moe.moe_dispatch_quant_mx(wl.x, wl.L, wl.A_mx, wl.A_sf, wl.status, stream=s),
                     s, reps, wl.flush)
    g = _time_events(lambda: moe.moe_grouped_gemm1_mx(wl.A_mx, wl.A_sf, wl.Wq_mx, wl.W_sf, wl.L, wl.Y, wl.status,
                                                       stream=s), s, reps, wl.flush)
    torch.cuda.synchronize()
    if wl.status.item() != 0:
        raise RuntimeError(f"device status {moe.status_string(wl.status.item())} in the MX variant")
    return {"dispatch_us": round(d, 1), "gemm1_us": round(g, 1),
            "scales": "e8m0 per 32 values (amax/448 rounded up to a power of two), applied by the tensor core"}


def run_pair_variant(wl, s, reps):
    """GEMM1 on CTA pairs (tcgen05 cta_group::2, M = 256 over two SMs) on the
    step's dispatch buffer: median CUDA-event time over `reps` launches, the L2
    flushed before every launch; its Y must be the single-CTA kernel's."""
    moe = wl.moe
    moe.moe_route_layout(wl.ids, wl.w, wl.L, wl.status, stream=s)
    moe.moe_dispatch_quant(wl.x, wl.L, wl.A, wl.As, wl.status, stream=s)
    moe.moe_grouped_gemm1(wl.A, wl.As, wl.Wq, wl.Ws, wl.L, wl.Y, wl.status, stream=s)
    with torch.cuda.stream(s):
        Y1 = wl.Y.clone()
    g = _time_events(lambda: moe.moe_grouped_gemm1(wl.A, wl.As, wl.Wq, wl.Ws, wl.L, wl.Y, wl.status, stream=s,
                                                    pair=True), s, reps, wl.flush)
    torch.cuda.synchronize()
    if wl.status.item() != 0:
        raise RuntimeError(f"device status {moe.status_string(wl.status.item())} in the pair GEMM1")
    same = bool(torch.equal(Y1.view(torch.int16), wl.Y.view(torch.int16)))
    del Y1
    return {"gemm1_us": round(g, 1), "same_Y_as_single_cta": same,
            "pairs": "two M-tiles of one expert x 256 columns per 2-CTA cluster (odd tile counts leave one CTA empty)"}


def run_e2e(wl, s, args, world, device):
    """Same step through the public API with pinned host buffers: every step
    copies its x and the router's pairs host->device, runs the path and copies
    the combined output device->host, all inside the timed region.  Serving
    pipeline: two buffer sets; the H2D of step i+1 (copy stream) and the D2H of
    step i-1 (second copy stream) overlap step i's kernels, with events
    ordering every reuse of a buffer.  Timed: K steps end to end, from an event
    before the first H2D to one after the last D2H.  No L2 flush: a step's
    working set (weights of the used experts, x, A, Y) is ~6 GB, far above L2."""
    T, H, k, N = wl.cfg.T, wl.cfg.H, wl.cfg.k, wl.cfg.N
    hx = [wl.x.cpu().pin_memory() for _ in range(2)]
    hids = [wl.ids.cpu().pin_memory() for _ in range(2)]
    hw = [wl.w.cpu().pin_memory() for _ in range(2)]
    hout = [torch.empty(T, N, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    dx = [torch.empty_like(wl.x) for _ in range(2)]
    dids = [torch.empty_like(wl.ids) for _ in range(2)]
    dw = [torch.empty_like(wl.w) for _ in range(2)]
    dout = [wl.out, torch.empty_like(wl.out)]
    c_in, c_out = torch.cuda.Stream(device), torch.cuda.Stream(device)
    saved = (wl.x, wl.out)

    def pipeline(steps):
        ev = lambda: torch.cuda.Event()
        in_done = [ev() for _ in range(steps)]
        comp_done = [ev() for _ in range(steps)]
        out_done = [ev() for _ in range(steps)]
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        c_in.wait_event(e0)

        def h2d(i):
            b = i % 2
            if i >= 2:
                c_in.wait_event(comp_done[i - 2])     # step i-2 has read this buffer set
            with torch.cuda.stream(c_in):
                dx[b].copy_(hx[b], non_blocking=True)
                dids[b].copy_(hids[b], non_blocking=True)
                dw[b].copy_(hw[b], non_blocking=True)
            in_done[i].record(c_in)

        h2d(0)
        for i in range(steps):
            b = i % 2
            if i + 1 < steps:
                h2d(i + 1)
            s.wait_event(in_done[i])
            if i >= 2:
                s.wait_event(out_done[i - 2])         # out[b] of step i-2 is on the host
            wl.x, wl.out = dx[b], dout[b]
            wl.step(s, args.variant, ids=dids[b], w=dw[b])
            comp_done[i].record(s)
            c_out.wait_event(comp_done[i])
            with torch.cuda.stream(c_out):
                hout[b].copy_(dout[b], non_blocking=True)
            out_done[i].record(c_out)
        s.wait_event(out_done[steps - 1])
        e1.record(s)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1)

    try:
        pipeline(3)                                    # warm-up
        steps = max(3, args.steps)
        ms = reduce_max(pipeline(steps) / steps, world, device)
    finally:
        wl.x, wl.out = saved
    bi = hx[0].numel() * 2 + hids[0].numel() * 4 + hw[0].numel() * 4
    bo = hout[0].numel() * 2
    return {"value": round(world * T / (ms / 1e3), 1), "unit": UNIT, "h2d_bytes_per_step": bi,
            "d2h_bytes_per_step": bo, "ms_per_step": round(ms, 4),
            "pipeline": "double-buffered: H2D of step i+1 and D2H of step i-1 overlap step i", "l2": "not flushed"}


# ---------------------------------------------------------------- CPU oracle (baseline / reference arm)

class CpuSample:
    """The oracle, as it stands, on a bounded sample of the workload, scaled to
    a whole step of T tokens.

    Untimed set-up: inputs, the router's top-k pairs (input preparation, not a
    step of the path), one layout and one quantisation of every token (to hand
    GEMM1 its operands), random bf16 expert outputs for the combine sample,
    and one expert's weights as random finite e4m3 codes
    with fp32 block scales, used for every sampled expert (weights are
    quantised offline and the oracle's time does not depend on their values).  Timed pieces:
      * fixed(): the routing layout of all T tokens (whole), then quant +
        dispatch and combine of a seeded sample of tokens (each x T / sample);
      * expert(): GEMM1 over all rows of one non-empty expert, the experts
        taken in a seeded random order without repetition (cycling once all
        are done); the mean over the experts timed, x the number of non-empty
        experts, estimates the whole GEMM1 call (exact once every expert has
        been timed)."""
    TOKENS = 64

    def __init__(self, cfg):
        import numpy as np
        import oracle
        from combine_counting_sort_gb300 import inputs
        self.np, self.oracle, self.cfg = np, oracle, cfg
        self.x = inputs.bf16_bits(inputs.make_x(cfg.T, cfg.H, cfg.seed))
        logits = inputs.make_logits(cfg.T, cfg.E, cfg.zipf, cfg.seed).numpy()
        self.ids, self.w = oracle.router_topk(logits, cfg.k)
        self.L = oracle.route_layout(self.ids, self.w, cfg.E, cfg.G)
        self.q, self.sc = oracle.quantize_rows(self.x)
        eo = self.L["expert_offset"]
        self.rng = np.random.default_rng(cfg.seed)
        self.order = self.rng.permutation(np.nonzero(eo[1:] > eo[:-1])[0])
        self.tokens = min(self.TOKENS, cfg.T)
        self.t_fixed, self.t_experts = [], []
        self.codes = self.rng.integers(0, 0x7E, size=(1, cfg.N, cfg.H), dtype=np.uint8)
        self.codes |= self.rng.integers(0, 2, size=self.codes.shape, dtype=np.uint8) << 7
        self.scales = np.full((1, cfg.N // 128, cfg.H // 128), 1.0 / (448.0 * math.sqrt(cfg.H)), np.float32)
        self.Y = oracle.f64_to_bf16(self.rng.standard_normal((self.tokens * cfg.k, cfg.N)))   # GEMM1 rows to combine

    def fixed(self) -> float:
        np, oracle, cfg = self.np, self.oracle, self.cfg
        S = self.tokens
        t0 = time.perf_counter()
        oracle.route_layout(self.ids, self.w, cfg.E, cfg.G)
        t_layout = time.perf_counter() - t0

        toks = self.rng.choice(cfg.T, S, replace=False)
        t0 = time.perf_counter()
        q, sc = oracle.quantize_rows(self.x[toks])
        oracle.dispatch(q, sc, np.arange(S * cfg.k), cfg.k)
        t_quant = time.perf_counter() - t0

        toks = self.rng.choice(cfg.T, S, replace=False)
        t0 = time.perf_counter()
        oracle.combine(self.Y, np.arange(S * cfg.k), self.w[toks])
        t_comb = time.perf_counter() - t0
        self.t_fixed.append(t_layout + (t_quant + t_comb) * cfg.T / S)
        return t_layout + t_quant + t_comb

    def expert(self) -> float:
        np, oracle, cfg, L = self.np, self.oracle, self.cfg, self.L
        e = int(self.order[len(self.t_experts) % len(self.order)])
        eo = L["expert_offset"]
        toks = L["row_pair"][eo[e]:eo[e + 1]] // cfg.k
        A, As = self.q[toks], np.ascontiguousarray(self.sc[toks].T)
        t0 = time.perf_counter()
        oracle.grouped_gemm1(A, As, self.codes, self.scales, np.array([0, len(toks)]))
        t = time.perf_counter() - t0
        self.t_experts.append(t)
        return t

    def step_ms(self) -> float:
        """Estimated oracle time of one whole step, from every piece timed so far."""
        return 1e3 * (statistics.mean(self.t_fixed) + statistics.mean(self.t_experts) * len(self.order))

    def describe(self) -> str:
        cfg = self.cfg
        return (f"{len(self.t_fixed)} x (layout of all {cfg.T} tokens; quant+dispatch and combine of "
                f"{self.tokens} sampled tokens) and GEMM1 of {len(self.t_experts)} sampled experts (all their rows, "
                f"of {len(self.order)} non-empty); each piece scaled to a whole step, value = T / that time")


def cpu_baseline(cfg, budget_s):
    sample = CpuSample(cfg)
    timed = sample.fixed()
    while not sample.t_experts or timed < budget_s:
        timed += sample.expert()
    return {"value": round(cfg.T / (sample.step_ms() / 1e3), 2), "unit": UNIT, "cores": cpu_threads(),
            "kind": "oracle", "sample": sample.describe(), "seconds": round(timed, 2)}


def cpu_threads() -> int:
    """Threads the oracle's numpy kernels may use: the BLAS pool if one is
    reported, else the cores this process may run on."""
    try:
        from threadpoolctl import threadpool_info
        n = [p["num_threads"] for p in threadpool_info() if p.get("user_api") == "blas"]
        if n:
            return max(n)
    except ImportError:
        pass
    return len(os.sched_getaffinity(0))


def run_reference(args):
    """Reference arm of this tier: the CPU oracle timed on the host cores.  Each
    step times the fixed pieces of a sampled step (CpuSample.fixed, ~0.1 s)
    and then experts' GEMM1 while the step's share of --ref-budget-s (with
    what earlier steps left unspent) lasts, so that a run takes about that
    budget plus 0.1 s per step."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    from combine_counting_sort_gb300 import inputs
    cfg = inputs.CONFIGS[args.workload]
    sample = CpuSample(cfg)
    for _ in range(args.warmup):         # untimed warm-up of the fixed pieces
        sample.fixed()
    sample.t_fixed.clear()
    share, bank, secs = args.ref_budget_s / max(1, args.steps), 0.0, 0.0
    for _ in range(args.steps):
        bank += share
        secs += sample.fixed()
        while bank > 0:
            t = sample.expert()
            bank -= t
            secs += t
    if not sample.t_experts:
        secs += sample.expert()
    full_step_ms = sample.step_ms()
    value = cfg.T / (full_step_ms / 1e3)
    # each timed step is a bounded sample of the workload: ms_per_step is what a
    # step took, the whole T-token step it stands for is estimated beside it
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * secs / args.steps, 1),
            "ms_per_full_step_estimate": round(full_step_ms, 3),
            "step": "a bounded sample of the T-token step (see cpu_baseline.sample); value = T / the estimated "
                    "time of the whole step",
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64 (fp32 quant)",
            "data": "synthetic (seeded)", "config": {"workload": cfg.name, "T": cfg.T, "H": cfg.H, "E": cfg.E,
                                                      "G": cfg.G, "k": cfg.k, "N": cfg.N, "zipf": cfg.zipf},
            "cpu_baseline": {"value": round(value, 2), "unit": UNIT, "cores": cpu_threads(), "kind": "oracle",
                             "sample": sample.describe(), "seconds_timed": round(secs, 2)},
            "e2e": {"value": round(value, 2), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- sweeps (one JSON line per case)

def _time_events(fn, s, reps, flush):
    ts = []
    for i in range(reps + 2):
        if flush is not None:
            with torch.cuda.stream(s):
                flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        fn()
        e1.record(s)
        torch.cuda.synchronize()
        if i >= 2:
            ts.append(e0.elapsed_time(e1) * 1e3)
    return statistics.median(ts)


def run_bw_sweep(args):
    """Dispatch + combine with the identity expert (no GEMM): GB/s per kernel vs HBM."""
    import combine_counting_sort_gb300 as moe
    from combine_counting_sort_gb300 import inputs
    import __graft_entry__ as ge
    ge.build()
    dev = torch.device("cuda", 0)
    s = torch.cuda.Stream(dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    peak = measured_peaks()["hbm_gbs"]
    for T in (2048, 4096, 8192, 16384):
        cfg = inputs.CONFIGS[f"bw_t{T}"]
        x = inputs.make_x(T, cfg.H, cfg.seed).to(dev)
        logits = inputs.make_logits(T, cfg.E, cfg.zipf, cfg.seed).to(dev)
        ids = torch.empty(T, cfg.k, dtype=torch.int32, device=dev)
        w = torch.empty(T, cfg.k, dtype=torch.float32, device=dev)
        moe.moe_router_topk(logits, cfg.k, ids, w)
        L = moe.Layout(T, cfg.k, cfg.E, cfg.G, device=dev)
        st = torch.zeros(1, dtype=torch.int32, device=dev)
        moe.moe_route_layout(ids, w, L, st)
        R = T * cfg.k
        A = torch.empty(R, cfg.H, dtype=torch.uint8, device=dev)
        As = torch.empty(cfg.H // 128, R, dtype=torch.float32, device=dev)
        Y = torch.empty(R, cfg.H, dtype=torch.bfloat16, device=dev)
        out = torch.empty(T, cfg.H, dtype=torch.bfloat16, device=dev)
        lay = _time_events(lambda: moe.moe_route_layout(ids, w, L, st, stream=s), s, args.steps, flush)
        d_us = _time_events(lambda: moe.moe_dispatch_quant(x, L, A, As, st, stream=s), s, args.steps, flush)
        moe.moe_dequant_rows(A, As, L, Y, stream=s)
        c_us = _time_events(lambda: moe.moe_combine(Y, L, out, st, stream=s), s, args.steps, flush)
        torch.cuda.synchronize()
        assert st.item() == 0
        d_bytes = 2.0 * T * cfg.H + R * cfg.H + 4.0 * R * cfg.H / 128
        c_bytes = 2.0 * R * cfg.H + 2.0 * T * cfg.H + 8.0 * R
        print(json.dumps({"sweep": "dispatch_combine_bw", "T": T, "H": cfg.H, "E": cfg.E, "k": cfg.k,
                          "layout_us": round(lay, 1), "dispatch_us": round(d_us, 1),
                          "dispatch_gbs": round(d_bytes / d_us / 1e3, 1), "dispatch_frac": round(d_bytes / d_us / 1e3 / peak, 3),
                          "combine_us": round(c_us, 1), "combine_gbs": round(c_bytes / c_us / 1e3, 1),
                          "combine_frac": round(c_bytes / c_us / 1e3 / peak, 3), "hbm_peak_gbs": peak}), flush=True)
        del x, A, As, Y, out, L


def run_layout_sweep(args):
    """Routing layout call latency vs batch (E=256, k=8, Zipf 1.2 routing): one
    block in a plain launch up to T = 32, the cooperative grid above; the
    no-plan layout beside it up to T*k = 16384 pairs."""
    import combine_counting_sort_gb300 as moe
    from combine_counting_sort_gb300 import inputs
    import __graft_entry__ as ge
    ge.build()
    dev = torch.device("cuda", 0)
    s = torch.cuda.Stream(dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    E, G, k = 256, 8, 8
    for T in (8, 32, 33, 128, 256, 512, 1024, 2048, 8192, 16384):
        logits = inputs.make_logits(T, E, 1.2, 0).to(dev)
        ids = torch.empty(T, k, dtype=torch.int32, device=dev)
        w = torch.empty(T, k, dtype=torch.float32, device=dev)
        moe.moe_router_topk(logits, k, ids, w)
        L = moe.Layout(T, k, E, G, device=dev)
        st = torch.zeros(1, dtype=torch.int32, device=dev)
        us = _time_events(lambda: moe.moe_route_layout(ids, w, L, st, stream=s), s, args.steps, flush)
        line = {"sweep": "layout", "T": T, "k": k, "E": E, "pairs": T * k, "layout_us": round(us, 1),
                "blocks": "one (plain launch)" if T <= 32 else "grid (cooperative)"}
        if T * k <= moe.MOE_NOPLAN_MAX_PAIRS:
            # the no-plan layout: reservation atomics in one block, rows in reservation order
            line["noplan_us"] = round(_time_events(lambda: moe.moe_route_layout_noplan(ids, w, L, st, stream=s),
                                                   s, args.steps, flush), 1)
        torch.cuda.synchronize()
        assert st.item() == 0
        print(json.dumps(line), flush=True)


def run_stage1_sweep(args):
    """Fused stage1 (default workload T=16384 Zipf(1.0)): producer SMs x flag granularity x schedule vs the
    unfused sum."""
    import combine_counting_sort_gb300 as moe
    from combine_counting_sort_gb300 import inputs
    import __graft_entry__ as ge
    ge.build()
    dev = torch.device("cuda", 0)
    cfg = inputs.CONFIGS[args.sweep_workload]
    wl = Workload(cfg, dev, moe.stage1_opts())
    s = torch.cuda.Stream(dev)
    moe.moe_route_layout(wl.ids, wl.w, wl.L, wl.status, stream=s)
    disp = _time_events(lambda: moe.moe_dispatch_quant(wl.x, wl.L, wl.A, wl.As, wl.status, stream=s), s,
                        args.steps, wl.flush)
    gemm = _time_events(lambda: moe.moe_grouped_gemm1(wl.A, wl.As, wl.Wq, wl.Ws, wl.L, wl.Y, wl.status, stream=s),
                        s, args.steps, wl.flush)
    print(json.dumps({"sweep": "stage1", "workload": cfg.name, "variant": "unfused", "dispatch_us": round(disp, 1),
                      "gemm1_us": round(gemm, 1), "sum_us": round(disp + gemm, 1)}), flush=True)
    for comm in (int(c) for c in args.sweep_comm.split(",")):
        for flags in (moe.MOE_FLAGS_PER_TILE, moe.MOE_FLAGS_PER_EXPERT):
            for sched in (moe.MOE_SCHED_EXPERT_MAJOR, moe.MOE_SCHED_READY_FIRST):
                opts = moe.stage1_opts(comm_sms=comm, flags=flags, schedule=sched, trace=1)
                us = _time_events(lambda: moe.moe_stage1(wl.x, wl.L, wl.Wq, wl.Ws, wl.A, wl.As, wl.Y, wl.ws,
                                                         wl.status, opts, stream=s), s, args.steps, wl.flush)
                tr = moe.stage1_trace(wl.ws)
                print(json.dumps({"sweep": "stage1", "workload": cfg.name, "comm_sms": comm,
                                  "flags": ["per_tile", "per_expert"][flags],
                                  "schedule": ["expert_major", "ready_first"][sched], "stage1_us": round(us, 1),
                                  "vs_unfused_sum": round(us / (disp + gemm), 3),
                                  "produced_us": round(tr["produced_us"], 1),
                                  "consumer_wait_us_total": round(tr["wait_us_total"], 1)}), flush=True)
    assert wl.status.item() == 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)   # ~1 s timed: several clock samples under load
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="t8192_zipf1.2")
    ap.add_argument("--variant", choices=VARIANTS, default="unfused",
                    help="the step timed for `value` (default: the fastest measured on this workload); the "
                         "others are timed beside it")
    ap.add_argument("--comm-sms", type=int, default=36)
    ap.add_argument("--flags", type=int, default=0, help="0 per-tile, 1 per-expert")
    ap.add_argument("--schedule", type=int, default=0, help="0 expert-major, 1 ready-first")
    ap.add_argument("--join", type=int, default=1, help="producer CTAs take GEMM work when done")
    ap.add_argument("--traffic", type=float, default=None,
                    help="dram bytes per launch of the roofline kernel from an ncu capture (else null)")
    ap.add_argument("--cpu-budget-s", type=float, default=15.0, help="seconds of oracle work of the cpu_baseline")
    ap.add_argument("--ref-budget-s", type=float, default=40.0,
                    help="seconds of sampled oracle GEMM1 in a whole --impl reference run")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--sweep", choices=["bw", "stage1", "layout"], default=None,
                    help="instead of the bench line: the dispatch/combine bandwidth sweep (identity expert, "
                         "T=2048..16384), the fused stage1 sweep or the layout latency sweep, one JSON line per case")
    ap.add_argument("--sweep-workload", default="stage1_t16384_zipf1.0",
                    help="workload of the stage1 sweep (a name from combine_counting_sort_gb300.inputs.CONFIGS)")
    ap.add_argument("--sweep-comm", default="8,16,24,36,48", help="producer SM counts of the stage1 sweep")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    elif args.sweep == "bw":
        run_bw_sweep(args)
    elif args.sweep == "stage1":
        run_stage1_sweep(args)
    elif args.sweep == "layout":
        run_layout_sweep(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
