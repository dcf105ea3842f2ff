#!/usr/bin/env python
"""Benchmark of the selective-SSM forward hot path on GB300.

One step = ssd_fwd on the Mamba-2 SSD workload b=4, L=8192, 80 heads, H=64, S=128, G=1,
chunk 256, bf16 inputs / fp32 accumulation, h0 ~ N(0, 0.1^2) (4 kernels), followed by
linscan_fwd on the scalar scan workload 384 rows x 65,536 fp32 (1 kernel).  Inputs are
seeded synthetic values, resident in HBM before the timed region; L2 (129 MB) is flushed
by a 256 MiB write before every timed step, outside the timed events.

Prints ONE JSON line (rank 0).  value = SSD forward tokens/s (batch*seqlen per SSD call,
summed over ranks, divided by the max over ranks of the SSD device time); the scan's GB/s,
per-kernel times, the roofline of the dominant kernel, clocks, the end-to-end leg through the
public API with host buffers, and the float64 oracle timed on the host cores ride along.  The
decode step (ssd_step: one token for each of 128 sequences of the same model shape, f32 state
carried in place) is timed on its own and reported under "decode", and the scan page's
baseline levels next to the production scan under "scan_baselines".

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
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from selective_state_space_mamba_gb300 import synth  # noqa: E402

METRIC = "SSD fwd tokens/s + % of roofline; linear-scan GB/s vs GB300 HBM peak"
SSD = synth.SSD_B4_L8192
SCAN = synth.SCAN_384x65536
STEP = synth.STEP_B128
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# GB300 HBM3e bandwidth from NVIDIA's public GB300 NVL72 specification: 576 TB/s for the rack's 72
# Blackwell Ultra GPUs, i.e. 8 TB/s per GPU.  The gates are also reported against this figure;
# the measured copy bandwidth (MEASURED_PEAKS.json) stays the roofline denominator.
DATASHEET_HBM_GBS = 8000.0
DATASHEET_SOURCE = "NVIDIA GB300 NVL72 specification: 576 TB/s HBM3e over 72 GPUs = 8 TB/s per GPU"
KERNELS = ("linscan_lookback", "ssd_chunk_cumsum", "ssd_chunk_state", "ssd_state_passing", "ssd_chunk_scan",
           "ssd_state_fused")  # the headline step's kernels; the decode step is timed on its own


# ----------------------------------------------------------------------------------------
# algorithmic byte / FLOP models (per launch)
# ----------------------------------------------------------------------------------------
def ssd_sizes(s):
    b, L, nh, H, S, G, T = s.batch, s.seqlen, s.nheads, s.headdim, s.dstate, s.ngroups, s.chunk
    nc = -(-L // T)
    e = 2 if s.dtype == "bf16" else 4
    return dict(x=b * L * nh * H * e, dt=b * L * nh * e, BC=b * L * G * S * e, AD=2 * nh * 4,
                state=b * nh * H * S * 4, chunk_states_f32=b * nc * nh * H * S * 4,
                hin=b * nc * nh * H * S * e, gd=2 * b * nh * nc * T * 4, y=b * L * nh * H * e)


def kernel_bytes(s):
    z = ssd_sizes(s)
    return {
        "ssd_chunk_cumsum": z["dt"] + z["AD"] // 2 + z["gd"],
        "ssd_chunk_state": z["x"] + z["BC"] + z["gd"] + z["chunk_states_f32"],
        "ssd_state_passing": z["chunk_states_f32"] + z["state"] + z["hin"] + z["state"],
        "ssd_chunk_scan": z["x"] + 2 * z["BC"] + z["gd"] + z["hin"] + z["AD"] // 2 + z["y"],
        # chunk states and state passing in one pass: x, B, G/dt and h0 in; h_in and h_final out
        "ssd_state_fused": z["x"] + z["BC"] + z["gd"] + z["hin"] + 2 * z["state"],
    }


def ssd_model_b_bytes(s):
    """Inputs once + outputs once + per-chunk fp32 states written once and read once."""
    z = ssd_sizes(s)
    return z["x"] + z["dt"] + 2 * z["BC"] + z["AD"] + z["state"] + z["y"] + z["state"] + 2 * z["chunk_states_f32"]


def ssd_flops(s):
    b, L, nh, H, S, G, T = s.batch, s.seqlen, s.nheads, s.headdim, s.dstate, s.ngroups, s.chunk
    nc = -(-L // T)
    state = 2 * b * nc * nh * T * H * S                 # X~^T B per (b, c, h)
    scan = b * nc * nh * (2 * T * T * H + 2 * T * S * H) + b * nc * G * 2 * T * T * S  # CB once per group
    return {"ssd_chunk_state": state, "ssd_state_fused": state, "ssd_chunk_scan": scan, "total": state + scan}


def step_bytes(s):
    """Decode step: the f32 state read and written once, x in, y out, dt, B, C, A, D."""
    e = 2 if s.dtype == "bf16" else 4
    state = s.batch * s.nheads * s.headdim * s.dstate * 4
    return 2 * state + 2 * s.batch * s.nheads * s.headdim * e + s.batch * s.nheads * e \
        + 2 * s.batch * s.ngroups * s.dstate * e + 2 * s.nheads * 4


def scan_bytes(rows, length):
    return 12 * rows * length  # read a, read b, write h


# ----------------------------------------------------------------------------------------
def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured (MEASURED_PEAKS.json)"
    return dict(FALLBACK_PEAKS), "fallback (6.8 TB/s, 1.9 PFLOP/s)"


def kernel_traffic(kernel):
    """ncu DRAM bytes per launch from profiles/ncu_traffic.json, if taken on the current source."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get(kernel)
    if not d:
        return None
    src = os.path.join(ROOT, "selective_state_space_mamba_gb300", "csrc", d["source"])
    if not os.path.exists(src) or hashlib.sha256(open(src, "rb").read()).hexdigest()[:16] != d["source_sha"]:
        return None
    return d["bytes_per_launch"]


class ClockSampler:
    """nvidia-smi clock / throttle sampling (every 10 ms); summary() keeps the samples taken
    inside [t0, t1] (host wall-clock bounds of the timed region)."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.out = ""

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "10"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()
        return False

    def summary(self, t0=None, t1=None):
        import datetime
        sm, mx, reasons, power = [], 0.0, set(), []
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in self.out.strip().splitlines():
            f = [v.strip() for v in line.split(",")]
            if len(f) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                ts = None
            if t0 is not None and ts is not None and not (t0 - 0.025 <= ts <= t1 + 0.025):
                continue
            try:
                sm.append(float(f[2]))
                mx = max(mx, float(f[3]))
                power.append(float(f[4]))
            except ValueError:
                continue
            for n, v in zip(names, f[6:10]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx or None,
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(power) if power else None}


# ----------------------------------------------------------------------------------------
def dist_setup(args):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(world, v):
    """The largest v over all ranks (NCCL reduces device tensors, gloo host tensors)."""
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_value(world, units_per_rank, ms_per_rank_max):
    """Whole-job throughput: the units every rank processed, over the slowest rank's time."""
    return world * units_per_rank / (ms_per_rank_max * 1e-3)


def device_inputs(torch, inp, dtype):
    out = {}
    for k, v in inp.items():
        t = torch.from_numpy(v).cuda()
        out[k] = t.to(torch.bfloat16) if (dtype == "bf16" and k in ("x", "dt", "B", "C")) else t
    return out


def run_ours(args, world, rank, local):
    import torch
    import selective_state_space_mamba_gb300 as ssm

    peaks, peak_src = load_peaks()
    ssd_np = synth.ssd_inputs(SSD)
    scan_np = synth.scan_inputs(SCAN.rows, SCAN.length, seed=synth.WORKLOAD_SEED[SCAN.name])
    d = device_inputs(torch, ssd_np, SSD.dtype)
    a = torch.from_numpy(scan_np["a"]).cuda()
    bsc = torch.from_numpy(scan_np["b"]).cuda()
    y = torch.empty_like(d["x"])
    hf = torch.empty(SSD.batch, SSD.nheads, SSD.headdim, SSD.dstate, dtype=torch.float32, device="cuda")
    h = torch.empty_like(a)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()

    def ssd_call():
        ssm.ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["h0"], chunk=SSD.chunk, y=y, h_final=hf)

    # per-shape plan, chosen by measurement once before anything is timed (as a user would);
    # "rules" keeps the library's rules of thumb (for profiler runs, where timings are skewed)
    if args.plan == "tune":
        plan, plan_ms = ssm.tune_ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["h0"],
                                         chunk=SSD.chunk, reps=5, y=y, h_final=hf)
        plan_how = "ssm_ssd_fwd_tune before the warm-up: every candidate plan timed, the fastest kept"
    else:
        ssm.set_ssd_fwd_plan(d["x"], d["B"], SSD.chunk, -1)
        plan, plan_ms, plan_how = 0, 0.0, "the library's rules of thumb (no tuning)"

    def scan_call():
        ssm.linscan_fwd(a, bsc, h=h)

    # the scan's CTA shape, chosen the same way (ssm_linscan_fwd_tune)
    if args.plan == "tune":
        scan_shape, scan_shape_ms = ssm.tune_linscan_fwd(a, bsc, h=h, reps=5)
    else:
        ssm.set_linscan_shape(SCAN.rows, SCAN.length, -1)
        scan_shape, scan_shape_ms = -1, 0.0

    for _ in range(args.warmup):
        flush.fill_(1)
        ssd_call()
        scan_call()
    torch.cuda.synchronize()
    if ssm.check_device_status(kind="ssd") or ssm.check_device_status(kind="linscan"):
        raise RuntimeError("device status error during warm-up")

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        time.sleep(0.1)  # let the sampler start
        t_wall0 = time.time()
        t_wall = time.perf_counter()
        for i in range(args.steps):
            flush.fill_(i & 0xff)
            ev[i][0].record(stream)
            ssd_call()
            ev[i][1].record(stream)
            scan_call()
            ev[i][2].record(stream)
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall
        barrier(world)
        # Per-kernel breakdown: the same steps again, with the library's events around every
        # launch.  Those events keep consecutive launches from overlapping (programmatic
        # dependent launch), so this second timed pass gives the per-kernel times and the
        # roofline, not the headline.  The clock record covers both passes.
        torch.cuda.synchronize()
        with ssm.KernelTimer(max_launches=8 * args.steps + 8) as kt:
            for i in range(args.steps):
                flush.fill_(i & 0xff)
                ssd_call()
                scan_call()
            torch.cuda.synchronize()
        t_wall1 = time.time()
        time.sleep(0.05)
    barrier(world)
    if ssm.check_device_status(kind="ssd") or ssm.check_device_status(kind="linscan"):
        raise RuntimeError("device status error during the timed region")
    decode = run_decode(args, peaks)
    scan_baselines = run_scan_baselines(args, peaks)

    # the median of the per-step samples (the scan page reports the median of interleaved
    # samples); min and max beside it
    ssd_s = [e[0].elapsed_time(e[1]) for e in ev]
    scan_s = [e[1].elapsed_time(e[2]) for e in ev]
    step_s = [e[0].elapsed_time(e[2]) for e in ev]
    ssd_ms, scan_ms, step_ms = (statistics.median(v) for v in (ssd_s, scan_s, step_s))
    ssd_ms_max = max_over_ranks(world, ssd_ms)
    scan_ms_max = max_over_ranks(world, scan_ms)
    step_ms_max = max_over_ranks(world, step_ms)
    tokens = SSD.batch * SSD.seqlen
    value = weak_scaling_value(world, tokens, ssd_ms_max)
    sbytes = scan_bytes(SCAN.rows, SCAN.length)
    scan_gbs = world * sbytes / (scan_ms_max * 1e-3) / 1e9

    # per-kernel
    kb = kernel_bytes(SSD)
    kb["linscan_lookback"] = sbytes
    kflops = ssd_flops(SSD)
    kernels = {}
    for k in KERNELS:
        n = kt.launches.get(k, 0)
        ms = kt.ms.get(k, 0.0) / max(n, 1)
        gbs = kb[k] / (ms * 1e-3) / 1e9 if ms > 0 else None
        ent = {"launches": n, "ms_per_launch": round(ms, 5), "alg_bytes": kb[k],
               "GB/s": round(gbs, 1) if gbs else None,
               "hbm_frac": round(gbs / peaks["hbm_gbs"], 4) if gbs else None}
        if k in kflops:
            tf = kflops[k] / (ms * 1e-3) / 1e12 if ms > 0 else None
            ent["alg_flops"] = kflops[k]
            ent["TFLOP/s"] = round(tf, 1) if tf else None
            ent["tensor_frac"] = round(tf / peaks["bf16_tflops"], 4) if tf else None
        kernels[k] = ent
    ssd_kernels = [k for k in KERNELS if k.startswith("ssd_")]
    dom = max(ssd_kernels, key=lambda k: kt.ms.get(k, 0.0))
    dk = kernels[dom]
    tensor_time = kflops.get(dom, 0) / (peaks["bf16_tflops"] * 1e12)
    hbm_time = kb[dom] / (peaks["hbm_gbs"] * 1e9)
    if dom in kflops and tensor_time > hbm_time:
        roof = {"kernel": dom, "bound": "tensor", "achieved": dk["TFLOP/s"], "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "frac": dk["tensor_frac"]}
    else:
        roof = {"kernel": dom, "bound": "hbm", "achieved": dk["GB/s"], "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": dk["hbm_frac"]}
    tr = kernel_traffic(dom)
    roof["traffic"] = tr
    roof["peak_source"] = peak_src + " (burst copy / burst cuBLAS)"

    model_b = ssd_model_b_bytes(SSD)
    ssd_roof_ms = max(model_b / (peaks["hbm_gbs"] * 1e9), kflops["total"] / (peaks["bf16_tflops"] * 1e12)) * 1e3
    out = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(step_ms_max, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded numpy PCG64; distributions of the pages' workloads)",
        "config": {
            "workload": workload_name(),
            "step": "ssd_fwd (4 kernels) then linscan_fwd (1 kernel); value from the ssd_fwd events",
            "per_kernel": "a second timed pass of the same steps with per-launch events",
            "l2": "inputs larger than L2, and L2 flushed by a 256 MiB write before each timed step",
            "parallelism": f"replicas x{world} (independent problems, no collective)",
            "plan": {"id": plan, "fused_state_path": (plan & 3) - 1, "sequential_state_passing": ((plan >> 2) & 3) - 1,
                     "scan_heads_per_cta": (plan >> 4) & 0xffff, "fused_ring_split": ("rule", "4+3", "3+4", "5+2")[
                         (plan >> 20) & 3], "tuning_median_ms": round(plan_ms, 4), "how": plan_how},
            "scan_shape": {"id": scan_shape, "tuning_median_ms": round(scan_shape_ms, 4),
                           "how": "ssm_linscan_fwd_tune before the warm-up (-1: the rule of thumb)"},
        },
        "timing": f"median of {args.steps} per-step CUDA-event samples (min / median / max below)",
        "ssd": {"tokens_per_s": round(value, 1), "ms": round(ssd_ms_max, 4), "ms_min_median_max": spread(ssd_s),
                "model_B_bytes": model_b, "roofline_ms": round(ssd_roof_ms, 4),
                "roofline_frac": round(ssd_roof_ms / ssd_ms_max, 4),
                "roofline_frac_datasheet": round(model_b / (DATASHEET_HBM_GBS * 1e9) * 1e3 / ssd_ms_max, 4),
                "io_only_bytes": model_b - 2 * ssd_sizes(SSD)["chunk_states_f32"]},
        "linscan": {"value": round(scan_gbs, 1), "unit": "GB/s", "ms": round(scan_ms_max, 4),
                    "ms_min_median_max": spread(scan_s), "alg_bytes": sbytes,
                    "frac": round(scan_gbs / world / peaks["hbm_gbs"], 4),
                    "frac_datasheet": round(scan_gbs / world / DATASHEET_HBM_GBS, 4)},
        "step_ms_min_median_max": spread(step_s),
        "datasheet_hbm": {"GB/s": DATASHEET_HBM_GBS, "source": DATASHEET_SOURCE},
        "kernels": kernels,
        "decode": decode,
        "scan_baselines": scan_baselines,
        "roofline": roof,
        "gpu_launches": sum(kt.launches.values()),
        "clocks": clocks.summary(t_wall0, t_wall1),
        "wall_s_timed": round(t_wall, 3),
    }
    return out, ssd_np, scan_np


def spread(samples):
    return [round(min(samples), 4), round(statistics.median(samples), 4), round(max(samples), 4)]


def run_decode(args, peaks):
    """The decode step (ssm_ssd_step) on its own workload: one token for each of 128 sequences,
    state updated in place, so every step starts from the state the previous one left.  The
    state (335.5 MB) is larger than L2; CUDA events around every launch on its stream."""
    import torch
    import selective_state_space_mamba_gb300 as ssm
    inp = synth.step_inputs(STEP)
    d = device_inputs(torch, inp, STEP.dtype)
    y = torch.empty_like(d["x"])
    stream = torch.cuda.current_stream()

    def call():
        ssm.ssd_step(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["state"], y=y, inplace=True)

    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    ev[0].record(stream)
    for i in range(args.steps):
        call()
        ev[i + 1].record(stream)
    torch.cuda.synchronize()
    per = [ev[i].elapsed_time(ev[i + 1]) for i in range(args.steps)]
    ms = statistics.median(per)
    nbytes = step_bytes(STEP)
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"workload": f"ssd_step b{STEP.batch} nh{STEP.nheads} H{STEP.headdim} S{STEP.dstate} G{STEP.ngroups} "
                        f"bf16, f32 state in place",
            "launches": args.steps, "ms_per_launch": round(ms, 5), "ms_min_median_max": spread(per),
            "ms_mean": round(sum(per) / len(per), 5),
            "tokens_per_s": round(STEP.batch / (ms * 1e-3), 1), "alg_bytes": nbytes, "GB/s": round(gbs, 1),
            "hbm_frac": round(gbs / peaks["hbm_gbs"], 4), "hbm_frac_datasheet": round(gbs / DATASHEET_HBM_GBS, 4),
            "traffic": kernel_traffic("ssd_step"),
            "timing": "median of per-launch CUDA events"}


# bytes each scan level moves per element (the reference page's traffic model): levels 1, 3,
# 3b and the production scan read a, b and write h; level 2 also writes and re-reads the local
# states and decay products
SCAN_LEVEL_BYTES = {"blelloch": 12, "three_pass": 28, "lookback_serial": 12, "lookback_warp": 12,
                    "linscan_fwd": 12}
# Hillis-Steele: per pass, two arrays read at t and t - d, two written (the last pass: one)


def hs_bytes(length):
    passes = max(0, (length - 1).bit_length())
    return 24 * passes - 4 if passes else 8


def run_scan_baselines(args, peaks):
    """The reference page's scan levels next to the production scan, on its own study shapes:
    96 MiB per array as 12288 rows x 2048 and 384 rows x 65536 (L2 flushed before each call,
    median of per-call CUDA events)."""
    import torch
    import selective_state_space_mamba_gb300 as ssm
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    out = {}
    for rows, length in ((12288, 2048), (SCAN.rows, SCAN.length)):
        inp = synth.scan_inputs(rows, length, seed=synth.BASE_SEED + 6)
        a = torch.from_numpy(inp["a"]).cuda()
        b = torch.from_numpy(inp["b"]).cuda()
        h = torch.empty_like(a)
        res = {}
        for algo in ("blelloch", "three_pass", "lookback_serial", "lookback_warp", "hillis_steele", "linscan_fwd"):
            if algo == "blelloch" and length > 2048:
                continue
            if algo == "linscan_fwd":
                def call():
                    ssm.linscan_fwd(a, b, h=h)
            else:
                def call(algo=algo):
                    ssm.linscan_baseline(a, b, algo, h=h)
            for _ in range(max(args.warmup, 3)):
                call()
            torch.cuda.synchronize()
            per = []
            for _ in range(15):
                flush.fill_(1)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                call()
                e1.record()
                torch.cuda.synchronize()
                per.append(e0.elapsed_time(e1))
            ms = statistics.median(per)
            n = rows * length
            per_elem = hs_bytes(length) if algo == "hillis_steele" else SCAN_LEVEL_BYTES[algo]
            moved = per_elem * n / (ms * 1e-3) / 1e9
            res[algo] = {"ms": round(ms, 4), "GB/s_3_array_model": round(12 * n / (ms * 1e-3) / 1e9, 1),
                         "GB/s_moved": round(moved, 1), "hbm_frac_moved": round(moved / peaks["hbm_gbs"], 4)}
        out[f"{rows}x{length}"] = res
    if ssm.check_device_status(kind="scan_lookback_serial") or ssm.check_device_status(kind="scan_lookback_warp"):
        raise RuntimeError("device status error in the baseline scans")
    return out


def run_e2e(args):
    """Same metric through the public API with pinned host buffers: H2D of the inputs, the call,
    D2H of y and h_final inside the timed region, every step.  The steps are pipelined the way a
    caller streaming batches would run them: three streams (H2D, compute, D2H) and two sets of
    device buffers, so that step i+1's inputs go in while step i computes and step i-1's results
    come out."""
    import torch
    import selective_state_space_mamba_gb300 as ssm
    inp = synth.ssd_inputs(SSD)
    host = {}
    for k, v in inp.items():
        t = torch.from_numpy(v)
        if SSD.dtype == "bf16" and k in ("x", "dt", "B", "C"):
            t = t.to(torch.bfloat16)
        host[k] = t.pin_memory()
    dev = [{k: torch.empty_like(v, device="cuda") for k, v in host.items()} for _ in range(2)]
    y_dev = [torch.empty_like(dev[0]["x"]) for _ in range(2)]
    hf_dev = [torch.empty(SSD.batch, SSD.nheads, SSD.headdim, SSD.dstate, dtype=torch.float32, device="cuda")
              for _ in range(2)]
    y_host = [torch.empty_like(host["x"]).pin_memory() for _ in range(2)]
    hf_host = [torch.empty(SSD.batch, SSD.nheads, SSD.headdim, SSD.dstate, dtype=torch.float32).pin_memory()
               for _ in range(2)]
    s_in, s_comp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: [torch.cuda.Event() for _ in range(2)]
    in_done, comp_done, out_done = ev(), ev(), ev()
    ws = ssm.Workspace()

    def step(i):
        j = i & 1
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(comp_done[j])  # buffer set j no longer read by step i-2
            for k in host:
                dev[j][k].copy_(host[k], non_blocking=True)
            in_done[j].record(s_in)
        with torch.cuda.stream(s_comp):
            s_comp.wait_event(in_done[j])
            if i >= 2:
                s_comp.wait_event(out_done[j])  # step i-2's results have left y_dev[j]
            d = dev[j]
            ssm.ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["h0"], chunk=SSD.chunk,
                        y=y_dev[j], h_final=hf_dev[j], workspace=ws)
            comp_done[j].record(s_comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(comp_done[j])
            y_host[j].copy_(y_dev[j], non_blocking=True)
            hf_host[j].copy_(hf_dev[j], non_blocking=True)
            out_done[j].record(s_out)

    for i in range(max(2, args.warmup)):
        step(i)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n = max(4, args.steps)  # the pipeline's fill and drain are inside the timed region
    start.record(s_in)
    for i in range(n):
        step(i)
    s_in.wait_stream(s_out)
    end.record(s_in)
    torch.cuda.synchronize()
    ms = start.elapsed_time(end) / n
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = y_host[0].numel() * y_host[0].element_size() + hf_host[0].numel() * 4
    return {"value": round(SSD.batch * SSD.seqlen / (ms * 1e-3), 1), "unit": "tokens/s", "ms_per_step": round(ms, 4),
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "pipeline": "H2D, compute and D2H on three streams with two buffer sets"}


def oracle_sample(ssd_np, scan_np, budget_s, unit_batch):
    """Time the float64 C oracle, as it stands, on a bounded sample of the SSD workload (whole
    (batch, head) units over the full sequence) and of the scan workload (whole rows)."""
    from oracle import native
    threads = native.max_threads()
    total_units = SSD.batch * SSD.nheads
    done, t_ssd = 0, 0.0
    order = np.random.default_rng(0).permutation(total_units)
    while done < total_units and t_ssd < budget_s:
        units = order[done:done + unit_batch]
        t0 = time.perf_counter()
        native.ssd_fwd(ssd_np["x"], ssd_np["dt"], ssd_np["A"], ssd_np["B"], ssd_np["C"], ssd_np["D"], ssd_np["h0"],
                       units=units)
        t_ssd += time.perf_counter() - t0
        done += len(units)
    ssd_tokens_equiv = done / SSD.nheads * SSD.seqlen  # tokens whose every head was computed
    # the same oracle on one host core: a few whole units
    one_units = order[:2]
    t0 = time.perf_counter()
    native.ssd_fwd(ssd_np["x"], ssd_np["dt"], ssd_np["A"], ssd_np["B"], ssd_np["C"], ssd_np["D"], ssd_np["h0"],
                   units=one_units, threads=1)
    t_one = time.perf_counter() - t0
    # the scan oracle on every row of the workload, repeated until at least 0.5 s have passed
    reps, t_scan = 0, 0.0
    while t_scan < 0.5:
        t0 = time.perf_counter()
        native.linscan(scan_np["a"], scan_np["b"])
        t_scan += time.perf_counter() - t0
        reps += 1
    # decode step: the one-token forward from the carried state, on every unit of the workload
    st = synth.step_inputs(STEP)
    t0 = time.perf_counter()
    native.ssd_fwd(st["x"][:, None], st["dt"][:, None], st["A"], st["B"][:, None], st["C"][:, None], st["D"],
                   st["state"].astype(np.float64))
    t_step = time.perf_counter() - t0
    return {
        "step_tokens_per_s": STEP.batch / t_step, "step_s": t_step,
        "ssd_tokens_per_s": ssd_tokens_equiv / t_ssd, "ssd_units": done, "ssd_s": t_ssd,
        "ssd_1core_tokens_per_s": len(one_units) / SSD.nheads * SSD.seqlen / t_one, "ssd_1core_units": len(one_units),
        "ssd_1core_s": t_one,
        "scan_gbs": reps * scan_bytes(SCAN.rows, SCAN.length) / t_scan / 1e9, "scan_reps": reps, "scan_s": t_scan,
        "cores": threads,
    }


def workload_name() -> str:
    """The one workload string both arms report."""
    return (f"ssd_fwd b{SSD.batch} L{SSD.seqlen} nh{SSD.nheads} H{SSD.headdim} S{SSD.dstate} "
            f"G{SSD.ngroups} chunk{SSD.chunk} bf16/fp32-acc + linscan {SCAN.rows}x{SCAN.length} f32")


def run_reference(args):
    """The float64 oracle timed on the host cores, on this bench's workload, metric and unit:
    each step is a bounded sample (a few whole (batch, head) units of the SSD workload)."""
    ssd_np = synth.ssd_inputs(SSD)
    from oracle import native
    threads = native.max_threads()
    per_step = max(1, threads)
    res = []
    for i in range(args.warmup + args.steps):
        units = np.arange(i * per_step, (i + 1) * per_step) % (SSD.batch * SSD.nheads)
        t0 = time.perf_counter()
        native.ssd_fwd(ssd_np["x"], ssd_np["dt"], ssd_np["A"], ssd_np["B"], ssd_np["C"], ssd_np["D"], ssd_np["h0"],
                       units=units)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            res.append(dt)
    step_s = sum(res) / len(res)
    tokens_equiv = per_step / SSD.nheads * SSD.seqlen
    value = tokens_equiv / step_s
    sample = (f"{per_step} whole (batch, head) units of the SSD workload per step "
              f"({per_step}/{SSD.batch * SSD.nheads} of the work of one SSD call)")
    return {"impl": "reference", "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(step_s * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded numpy PCG64)",
            "config": {"workload": workload_name(),
                       "timed": "float64 oracle on sampled whole (batch, head) units of the ssd_fwd part; "
                                "value is the ssd_fwd tokens/s, as in the CUDA arm"},
            "cpu_baseline": {"value": round(value, 1), "unit": "tokens/s", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 1), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def run_ssd_configs(args, steps=None):
    """Every bf16 SSD workload (b8 L2048 nh24, b4 L8192 nh80, b1 L131072 nh32 G8) timed alone
    with its tuned plan (or --plan rules / --plan-id), L2 flushed before each forward.  Median of
    `steps` forwards (min and max beside it); per-kernel times from the library's events.
    Returns one entry per workload."""
    import torch
    import selective_state_space_mamba_gb300 as ssm
    peaks, _ = load_peaks()
    steps = steps or args.steps
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    entries = []
    for shape in (synth.SSD_B8_L2048, synth.SSD_B4_L8192, synth.SSD_B1_L131072):
        if args.ssd_workload and shape.name != args.ssd_workload:
            continue
        d = device_inputs(torch, synth.ssd_inputs(shape), shape.dtype)
        y = torch.empty_like(d["x"])
        hf = torch.empty(shape.batch, shape.nheads, shape.headdim, shape.dstate, dtype=torch.float32, device="cuda")

        def call():
            ssm.ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["h0"], chunk=shape.chunk, y=y, h_final=hf)

        if args.plan_id is not None:  # a fixed plan (profiler runs of one path)
            plan = args.plan_id
            ssm.set_ssd_fwd_plan(d["x"], d["B"], shape.chunk, plan)
        elif args.plan == "tune":
            plan, _ = ssm.tune_ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["h0"], chunk=shape.chunk,
                                       reps=5, y=y, h_final=hf)
        else:
            plan = -1
            ssm.set_ssd_fwd_plan(d["x"], d["B"], shape.chunk, -1)
        for _ in range(max(3, args.warmup)):
            flush.fill_(1)
            call()
        ms = []
        for i in range(steps):
            flush.fill_(i & 0xff)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            call()
            e1.record()
            torch.cuda.synchronize()
            ms.append(e0.elapsed_time(e1))
        with ssm.KernelTimer(max_launches=8 * steps + 8) as kt:
            for i in range(steps):
                flush.fill_(i & 0xff)
                call()
            torch.cuda.synchronize()
        if ssm.check_device_status(kind="ssd"):
            raise RuntimeError(f"device status error in {shape.name}")
        med = float(np.median(ms))
        roof_ms = ssd_model_b_bytes(shape) / (peaks["hbm_gbs"] * 1e9) * 1e3
        entries.append({"workload": shape.name, "plan": plan, "ms": round(med, 4), "ms_min_median_max": spread(ms),
                        "tokens_per_s": round(shape.batch * shape.seqlen / (med * 1e-3), 1),
                        "model_B_roofline_ms": round(roof_ms, 4), "roofline_frac": round(roof_ms / med, 4),
                        "roofline_frac_datasheet": round(roof_ms * peaks["hbm_gbs"] / DATASHEET_HBM_GBS / med, 4),
                        "per_kernel_us": {k: round(kt.ms[k] / kt.launches[k] * 1e3, 1)
                                          for k in kt.ms if kt.launches.get(k)}})
        del d, y, hf
        torch.cuda.empty_cache()
    return entries


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--cpu-budget-s", type=float, default=15.0, help="time budget of the oracle CPU baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-ssd-configs", action="store_true", help="leave out the per-workload SSD block")
    ap.add_argument("--ssd-configs", action="store_true",
                    help="instead of the bench line: time every bf16 SSD workload alone, one JSON line each")
    ap.add_argument("--ssd-workload", default=None, help="with --ssd-configs: only the workload of this name")
    ap.add_argument("--plan-id", type=int, default=None,
                    help="with --ssd-configs: this ssd_fwd plan id instead of tuning (see ssm_ssd_fwd_set_plan)")
    ap.add_argument("--plan", choices=("tune", "rules"), default="tune",
                    help="ssd_fwd plan: tuned by measurement first (default) or the rules of thumb")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        print("note: fewer than 3 warm-up steps", file=sys.stderr)

    if args.impl == "reference":
        if int(os.environ.get("RANK", "0")) != 0:
            return
        print(json.dumps(run_reference(args)))
        return

    if args.ssd_configs:
        for e in run_ssd_configs(args):
            print(json.dumps(e), flush=True)
        return
    world, rank, local = dist_setup(args)
    out, ssd_np, scan_np = run_ours(args, world, rank, local)
    if not args.no_ssd_configs:
        # every bf16 SSD workload alone (tuned plan each), for the per-workload rooflines
        out["ssd_configs"] = run_ssd_configs(args, steps=max(15, min(args.steps, 30)))
    if not args.no_e2e:
        e2e = run_e2e(args)
        e2e["value"] = round(max_over_ranks(world, -e2e["value"]) * -1 * world, 1) if world > 1 else e2e["value"]
        out["e2e"] = e2e
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cb = oracle_sample(ssd_np, scan_np, args.cpu_budget_s, unit_batch=16)
        out["cpu_baseline"] = {
            "value": round(cb["ssd_tokens_per_s"], 1), "unit": "tokens/s", "cores": cb["cores"], "kind": "oracle",
            "sample": (f"{cb['ssd_units']} of {SSD.batch * SSD.nheads} whole (batch, head) units of the SSD workload "
                       f"in {cb['ssd_s']:.1f} s; tokens/s counts a token once all its heads are done"),
            "one_core": {"value": round(cb["ssd_1core_tokens_per_s"], 1), "unit": "tokens/s", "cores": 1,
                         "sample": f"{cb['ssd_1core_units']} whole (batch, head) units on one thread in "
                                   f"{cb['ssd_1core_s']:.2f} s"},
            "linscan": {"value": round(cb["scan_gbs"], 2), "unit": "GB/s", "cores": cb["cores"],
                        "sample": f"all {SCAN.rows} rows, {cb['scan_reps']} times, in {cb['scan_s']:.2f} s"},
            "decode": {"value": round(cb["step_tokens_per_s"], 1), "unit": "tokens/s",
                       "sample": f"one whole decode step ({STEP.batch} tokens) in {cb['step_s']:.2f} s"},
        }
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(out))


if __name__ == "__main__":
    main()
