#!/usr/bin/env python
"""PSA self-attention backward throughput on GB300.

One step = one psa_attn_bwd call (every backward kernel: D preprocess, the
dK/dV/dQ contractions, the dQ write-out) over one batch of synthetic inputs
already resident in HBM, for the bf16 B=8, heads=2, N=6400 (80x80 map),
head_dim=32 workload.  The forward (psa_attn_fwd) produces O and LSE once,
before timing.  Before every timed step L2 (129 MB) is flushed by writing a
256 MB buffer and then reading a second 256 MB buffer, so that the step starts
with none of its data in L2 and no dirty line of the flush left to be written
back while it runs (--l2-flush write: the write alone); each step is timed with
CUDA events on the launching stream.  Per-kernel times come from a second pass
of the same steps with events around each kernel.

Metric: TFLOP/s counting 12*N^2*d per (batch, head) -- 4*N^2*d for the shared
S recompute plus 2 * 4*N^2*d for the per-V-half dP/dV and dQ/dK terms.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun (N > 1) every rank runs the whole workload on its own GPU
(independent batches, weak scaling, no collective on the data path); the
slowest rank's time sets the aggregate.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "PSA attn-bwd TFLOP/s (1 GB300, N=400/1600/6400) and % of roofline"
UNIT = "TFLOP/s"
HEADLINE = "psa_bf16_b8_h2_n6400_d32"
SECONDARY = ["psa_bf16_b32_h8_n400_d64", "psa_bf16_b16_h4_n1600_d64", "psa_f32_b8_h4_n400_d64"]
FLUSH_BYTES = 256 << 20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ------------------------------------------------------------------ accounting
def metric_flops(w) -> float:
    """Counted FLOPs of one backward over the whole workload."""
    return 12.0 * w.N * w.N * w.d * w.BH


# Per-launch FLOPs of each kernel, in units of N^2*d per (batch, head).  The
# fused tensor-core kernel does the whole backward: the metric's 12 (it
# executes 14).  The two-pass dK/dV kernel executes S (2), dP (4), dV (4) and
# dK (2); the dQ pass S (2), dP (4) and dQ (2).  The CUDA-core dK/dV and dQ
# kernels are credited with the metric's terms they produce.
KERNEL_FLOPS = {
    "tc": {"bwd_main": 12.0},
    "tc2": {"bwd_main": 12.0, "bwd_dq": 8.0},
    "simt": {"bwd_main": 10.0, "bwd_dq": 2.0},
}
# executed FLOPs of one backward, same units
EXECUTED = {"tc": 14.0, "tc2": 20.0, "simt": 20.0}


def resolved_algo(B, name: str, w) -> str:
    """The kernel family a run with --algo `name` uses on workload w."""
    if name != "auto":
        return name
    tc = B.psa_attn_bwd_workspace_bytes(1, 1, 16, w.d, 1 if w.dtype == "bf16" else 0, B.PSA_ALGO_TC) > 0
    return "tc" if tc else "simt"


def alg_bytes(w) -> float:
    """Algorithmic HBM bytes of one backward: read Q, K, V_lo, V_hi, O_lo, O_hi,
    dO_lo, dO_hi and LSE (fp32); write dQ, dK, dV_lo, dV_hi."""
    s = 2 if w.dtype == "bf16" else 4
    return float(w.BH) * (12.0 * w.N * w.d * s + 4.0 * w.N)


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def tensor_peak(peaks, dtype: str, sustained=False) -> float:
    bf16 = peaks["bf16_tflops_sustained" if sustained else "bf16_tflops"]
    # fp32 storage runs on CUDA cores / tf32-class rates: nominal tf32 : bf16 = 1 : 2
    return bf16 if dtype == "bf16" else bf16 / 2.0


def roofline_time_s(w, peaks) -> tuple[float, str]:
    t_t = metric_flops(w) / (tensor_peak(peaks, w.dtype) * 1e12)
    t_m = alg_bytes(w) / (peaks["hbm_gbs"] * 1e9)
    return (t_t, "tensor") if t_t >= t_m else (t_m, "hbm")


# Sources each kernel family's code comes from (the traffic record is tied to
# their contents; a change elsewhere, such as the forward, leaves it valid).
TRAFFIC_SOURCES = {
    "tc": ["tc_bwd.cu", "tc_tmap.cu", "tc_ptx.cuh", "tc_sync.cuh", "common.cuh", "psa_internal.h"],
    "tc2": ["tc_pair.cu", "tc_bwd.cu", "tc_dq.cu", "tc_tmap.cu", "tc_ptx.cuh", "tc_sync.cuh", "common.cuh",
            "psa_internal.h"],
    "simt": ["simt_kernels.cuh", "psa_attn.cu", "common.cuh", "psa_internal.h"],
}


def source_hash(algo: str) -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "self_attention_backward_gb300", "csrc")
    for name in sorted(TRAFFIC_SOURCES.get(algo, os.listdir(csrc))):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel_slot: str, workload: str, algo: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except Exception:
        return None
    e = rec.get(workload, {}).get(algo, {}).get(kernel_slot)
    if not e or e.get("source_hash") != source_hash(algo):
        return None
    return float(e["dram_bytes_per_launch"])


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out = ""
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        if not getattr(self, "lines", None):
            return None
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ distributed
def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def max_over_ranks(x: float, world: int, device=None) -> float:
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------------ cpu oracle
def oracle_sample(w, budget_s: float, max_slices: int | None = None):
    """Time the fp64 oracle on whole (batch, head) slices of workload w until
    `budget_s` has elapsed (at least one slice).  Returns (TFLOP/s, slices, s)."""
    import numpy as np
    import oracle
    from self_attention_backward_gb300.inputs import make_inputs
    inp = make_inputs(w, BH=max_slices or w.BH)
    done, t_total = 0, 0.0
    while done < inp.packed.shape[0]:
        p = inp.packed[done:done + 1].astype(np.float64)
        vs = np.ascontiguousarray(p[:, 2:4].transpose(1, 0, 2, 3))
        dos = np.stack([inp.do_lo[done:done + 1], inp.do_hi[done:done + 1]]).astype(np.float64)
        t0 = time.perf_counter()
        oracle.attn_bwd(p[:, 0], p[:, 1], vs, dos, inp.scale)
        t_total += time.perf_counter() - t0
        done += 1
        if t_total >= budget_s:
            break
    flops = 12.0 * w.N * w.N * w.d * done
    return flops / t_total / 1e12, done, t_total


# ------------------------------------------------------------------ arms
def run_reference(args, w):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    if args.warmup > 0:                       # one untimed slice warms caches and threads
        oracle_sample(w, 0.0, max_slices=1)
    vals, t_all, slices = [], 0.0, 0
    for _ in range(args.steps):
        v, n, t = oracle_sample(w, 0.0, max_slices=1)
        vals.append(v)
        t_all += t
        slices += n
    value = 12.0 * w.N * w.N * w.d * slices / t_all / 1e12
    sample = f"{slices} of {w.BH} (batch, head) slices of {w.name}, one per step, fp64"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t_all / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(w, args.l2_flush),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def workload_config(w, flush_mode="write+read"):
    how = (f"{FLUSH_BYTES >> 20} MB write" if flush_mode == "write"
           else f"{FLUSH_BYTES >> 20} MB write, then a {FLUSH_BYTES >> 20} MB read of a second buffer")
    return {"workload": w.name, "B": w.B, "heads": w.heads, "N": w.N, "feature_map": w.fmap,
            "head_dim": w.d, "storage": w.dtype, "scale": w.scale, "seed": w.seed,
            "l2": f"flushed ({how}) before every timed step"}


class L2Flush:
    """Evicts L2 before a timed step: writes a buffer twice the size of L2 and,
    in mode "write+read", then reads a second one of that size, which writes
    the first buffer's dirty lines back before the step instead of during it."""

    def __init__(self, device, mode="write+read"):
        import torch
        self.mode = mode
        self.w = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=device)
        # fp32, whose sum is one reduction kernel (an int32 sum first casts to int64)
        self.r = torch.ones(FLUSH_BYTES // 4, dtype=torch.float32, device=device) if mode != "write" else None

    def __call__(self):
        self.w.zero_()
        if self.r is not None:
            self.r.sum()


def device_inputs(w, device):
    import torch
    from self_attention_backward_gb300 import binding as B
    from self_attention_backward_gb300.inputs import make_inputs
    inp = make_inputs(w)
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    dev = lambda a: torch.from_numpy(a).to(device).to(tdt).contiguous()  # noqa: E731
    packed, do_lo, do_hi = dev(inp.packed), dev(inp.do_lo), dev(inp.do_hi)
    o_lo, o_hi, lse = B.attn_fwd(packed, w.scale)
    torch.cuda.synchronize()
    return packed, o_lo, o_hi, lse, do_lo, do_hi


def time_steps(w, bufs, steps, flush, device, algo):
    """Per-step CUDA-event times (ms) of psa_attn_bwd on the current stream."""
    import torch
    from self_attention_backward_gb300 import binding as B
    packed, o_lo, o_hi, lse, do_lo, do_hi = bufs
    d_packed = torch.empty_like(packed)
    ws = B.BwdWorkspace(device)
    st = torch.cuda.current_stream()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for a, b in evs:
        flush()
        a.record(st)
        B.attn_bwd(packed, o_lo, o_hi, lse, do_lo, do_hi, w.scale, d_packed=d_packed, workspace=ws, algo=algo)
        b.record(st)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


def run_ours(args, w):
    import torch
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    from self_attention_backward_gb300.build import build
    build()
    from self_attention_backward_gb300 import binding as B
    algo = {"auto": B.PSA_ALGO_AUTO, "simt": B.PSA_ALGO_SIMT, "tc": B.PSA_ALGO_TC,
            "tc2": B.PSA_ALGO_TC_2PASS}[args.algo]
    peaks, peaks_src = read_peaks()

    bufs = device_inputs(w, device)
    flush = L2Flush(device, args.l2_flush)
    time_steps(w, bufs, max(args.warmup, 3), flush, device, algo)       # warm-up
    B.psa_attn_sync_status()

    with ClockSampler(torch.cuda.current_device() if "CUDA_VISIBLE_DEVICES" not in os.environ else local) as cs:
        barrier(world)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        step_ms = time_steps(w, bufs, args.steps, flush, device, algo)
        torch.cuda.synchronize()
        barrier(world)
        wall = time.perf_counter() - t0
        # per-kernel times: the same steps once more, with events around each
        # kernel (the library then starts each kernel after the one before it)
        B.psa_attn_profile_read()
        B.psa_attn_profile_enable(True)
        prof_step_ms = time_steps(w, bufs, args.steps, flush, device, algo)
        B.psa_attn_profile_enable(False)
        prof = B.psa_attn_profile_read()
    B.psa_attn_sync_status()

    ms_local = sum(step_ms) / len(step_ms)
    ms = max_over_ranks(ms_local, world, device)
    value = metric_flops(w) * world / (ms * 1e-3) / 1e12
    launches = sum(n for _, n in prof.values())
    # dominant kernel: largest total time in the timed region
    dom = max((k for k in prof if prof[k][1] > 0), key=lambda k: prof[k][0])
    dom_ms = prof[dom][0] / prof[dom][1]
    t_roof, bound = roofline_time_s(w, peaks)
    # algorithmic work of the dominant kernel per launch
    used_algo = resolved_algo(B, args.algo, w)
    if bound == "tensor":
        share = KERNEL_FLOPS[used_algo].get(dom, 0.0)
        achieved = share * w.BH * w.N * w.N * w.d / (dom_ms * 1e-3) / 1e12
        peak, unit = tensor_peak(peaks, w.dtype), "TFLOP/s"
        peak_note = f"bf16_tflops (burst) of {peaks_src}"
    else:
        achieved = alg_bytes(w) / (dom_ms * 1e-3) / 1e9
        peak, unit = peaks["hbm_gbs"], "GB/s"
        peak_note = f"hbm_gbs of {peaks_src}"
    traffic = recorded_traffic(dom, w.name, used_algo)

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if w.dtype == "bf16" else "f32", "data": "synthetic",
        "config": dict(workload_config(w, args.l2_flush),
                       parallelism=f"replicas x{world}" if world > 1 else "single GPU", algo=used_algo),
        "roofline": {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
                     "frac": achieved / peak, "traffic": traffic, "kernel": dom, "peak_source": peak_note},
        "step_roofline_frac": t_roof / (ms * 1e-3),
        "executed_tflops": value * EXECUTED[used_algo] / 12.0,
        "kernels_ms_per_step": {k: v[0] / args.steps for k, v in prof.items() if v[1]},
        "kernel_timing": ("a second pass of the same steps with CUDA events around each kernel, the kernels "
                          "started one after another; that pass's ms per step: "
                          f"{statistics.mean(prof_step_ms):.4f}"),
        "gpu_launches": launches,
        "wall_s_timed_region": wall,
    }
    clocks = cs.summary()
    line["clocks"] = clocks

    if rank == 0 and not args.no_secondary:
        sec = {}
        for name in SECONDARY:
            from self_attention_backward_gb300.inputs import WORKLOADS
            w2 = WORKLOADS[name]
            # a kernel family the workload's storage type lacks falls back to AUTO
            dt2 = 1 if w2.dtype == "bf16" else 0
            algo2 = algo if B.psa_attn_bwd_workspace_bytes(1, 1, 16, w2.d, dt2, algo) > 0 else B.PSA_ALGO_AUTO
            b2 = device_inputs(w2, device)
            time_steps(w2, b2, 3, flush, device, algo2)
            t2 = statistics.mean(time_steps(w2, b2, max(5, args.steps // 2), flush, device, algo2))
            tr, bd = roofline_time_s(w2, peaks)
            sec[name] = {"tflops": metric_flops(w2) / (t2 * 1e-3) / 1e12, "ms": t2, "bound": bd,
                         "roofline_frac": tr / (t2 * 1e-3), "storage": w2.dtype,
                         "algo": resolved_algo(B, {B.PSA_ALGO_AUTO: "auto", B.PSA_ALGO_SIMT: "simt",
                                                   B.PSA_ALGO_TC: "tc", B.PSA_ALGO_TC_2PASS: "tc2"}[algo2], w2)}
            del b2
        line["other_workloads"] = sec

    if rank == 0 and not args.no_extras:
        line["e2e"] = run_e2e(w, args, device, algo)
        line["forward"] = time_forward(w, bufs, flush, args.steps)
        line["merge"] = time_merge(w, bufs, flush, args.steps, algo)
    if rank == 0 and world == 1 and not args.no_cpu:
        v, n, t = oracle_sample(w, args.cpu_budget)
        import oracle
        line["cpu_baseline"] = {"value": v, "unit": UNIT, "cores": oracle.threads(), "kind": "oracle",
                                "sample": f"{n} of {w.BH} (batch, head) slices of {w.name}, fp64, {t:.1f} s"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def time_forward(w, bufs, flush, steps):
    """psa_attn_fwd on the same workload (support for the backward, outside the
    timed step): CUDA-event time per call, L2 flushed before each call, and
    TFLOP/s counting 6 N^2 d per (batch, head) (S and the two P V products)."""
    import torch
    from self_attention_backward_gb300 import binding as B
    packed = bufs[0]
    st = torch.cuda.current_stream()
    for _ in range(3):
        B.attn_fwd(packed, w.scale)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for a, b in evs:
        flush()
        a.record(st)
        B.attn_fwd(packed, w.scale)
        b.record(st)
    torch.cuda.synchronize()
    ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
    return {"ms": ms, "tflops": 6.0 * w.BH * w.N * w.N * w.d / (ms * 1e-3) / 1e12, "flops_per_bh": "6 N^2 d"}


def time_merge(w, bufs, flush, steps, algo):
    """The merge op's backward with the attention backward on the same
    workload, dO_lo / dO_hi given as one merged [B, 2*heads*d, H, W] gradient
    (synthetic, drawn like dO): fused (psa_merge_attn_bwd reads dO out of it)
    against separate (psa_merge_bwd into contiguous dO, then psa_attn_bwd).
    CUDA events per call, L2 flushed before each."""
    import torch
    from self_attention_backward_gb300 import binding as B
    packed, o_lo, o_hi, lse = bufs[0], bufs[1], bufs[2], bufs[3]
    H, Wd = (int(x) for x in w.fmap.split("x"))
    g = torch.randn((w.B, 2 * w.heads * w.d, H, Wd), generator=torch.Generator().manual_seed(w.seed + 100))
    gm = g.to(packed.device).to(packed.dtype)
    d_packed = torch.empty_like(packed)
    ws = B.BwdWorkspace(packed.device)
    d_lo = torch.empty_like(o_lo)
    d_hi = torch.empty_like(o_lo)

    def fused():
        B.merge_attn_bwd(packed, o_lo, o_hi, lse, gm, w.heads, w.scale, d_packed=d_packed, workspace=ws, algo=algo)

    def separate():
        B.psa_merge_bwd(gm, d_lo, d_hi, w.B, w.heads, H, Wd, w.d, 1 if w.dtype == "bf16" else 0)
        B.attn_bwd(packed, o_lo, o_hi, lse, d_lo, d_hi, w.scale, d_packed=d_packed, workspace=ws, algo=algo)

    st = torch.cuda.current_stream()
    out = {}
    for name, fn in (("fused", fused), ("separate", separate)):
        for _ in range(3):
            fn()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for a, b in evs:
            flush()
            a.record(st)
            fn()
            b.record(st)
        torch.cuda.synchronize()
        out[name + "_ms"] = statistics.mean(a.elapsed_time(b) for a, b in evs)
    B.psa_attn_sync_status()
    out["d_merged"] = list(gm.shape)
    return out


def run_e2e(w, args, device, algo):
    """Same metric through the public API on HOST buffers: per step the inputs
    are copied host->device from pinned memory and d_packed device->host."""
    import torch
    from self_attention_backward_gb300 import binding as B
    from self_attention_backward_gb300.inputs import make_inputs
    inp = make_inputs(w)
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    pin = lambda a: torch.from_numpy(a).to(tdt).pin_memory()  # noqa: E731
    packed, do_lo, do_hi = pin(inp.packed), pin(inp.do_lo), pin(inp.do_hi)
    o_lo_d, o_hi_d, lse_d = B.attn_fwd(packed.to(device), w.scale)
    o_lo, o_hi, lse = o_lo_d.cpu().pin_memory(), o_hi_d.cpu().pin_memory(), lse_d.cpu().pin_memory()
    out = torch.empty(packed.shape, dtype=tdt).pin_memory()
    dt = B.PSA_BF16 if w.dtype == "bf16" else B.PSA_F32
    runner = B.HostBwd(w.BH, w.N, w.d, dt, device=device, algo=algo)
    st = torch.cuda.current_stream()
    for _ in range(3):
        runner(packed, o_lo, o_hi, lse, do_lo, do_hi, w.scale, out)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(st)
    for _ in range(args.steps):
        runner(packed, o_lo, o_hi, lse, do_lo, do_hi, w.scale, out)
    b.record(st)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / args.steps
    return {"value": metric_flops(w) / (ms * 1e-3) / 1e12, "unit": UNIT, "ms_per_step": ms,
            "h2d_bytes_per_step": runner.h2d_bytes(), "d2h_bytes_per_step": runner.d2h_bytes()}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=HEADLINE)
    ap.add_argument("--algo", choices=["auto", "simt", "tc", "tc2"], default="auto")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle time for cpu_baseline")
    ap.add_argument("--l2-flush", choices=["write+read", "write"], default="write+read",
                    help="L2 eviction before each timed step (see the module docstring)")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the end-to-end, forward and merge legs (profiling runs)")
    args = ap.parse_args(argv)
    from self_attention_backward_gb300.inputs import WORKLOADS
    w = WORKLOADS[args.workload]
    if args.impl == "reference":
        return run_reference(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
