"""Benchmark: context-parallel causal GQA prefill attention on GB300.

One step = one ``slope_cp_prefill`` call over the whole workload: every ring
step's partial (output + log-sum-exp per rank and step) followed by the exact
log-sum-exp merge.  Default workload: S = 32768, 64 query / 8 KV heads, head
dim 64, bf16, zigzag ring of 8 simulated ranks.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--window W] [--impl reference]

Prints one JSON line (rank 0).  ``value`` is algorithmic TFLOP/s (visible
query-key pairs x Hq x 2 x (dqk + dv)) of the whole job.  ``e2e`` is the same
metric through ``slope_cp_prefill_host`` with pinned host buffers: every step
copies Q/K/V in and out/lse back inside the timed region, two device-buffer
sets letting each step's copies overlap its neighbours' compute.
``fused_single_launch`` is the same attention as one launch over the whole
sequence (no partials, no merge); ``bf16_partials`` is the step with the
partial outputs kept in bf16 (``slope_cp_prefill_ex``); ``ulysses`` is the
head-sharded layout (one KV head group per rank, no merge).  ``--impl reference`` times the fp64 CPU
oracle on a bounded sample of the same workload (rank 0 only).
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

import slope_workloads as wl  # noqa: E402

METRIC = "causal prefill-attention TFLOP/s & tokens/s at 32K–100K; % of GB300 BF16 tensor peak"
UNIT = "TFLOP/s"
DEFAULT_WORKLOAD = "causal_gqa_s32k_zigzag8"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# every source file the attention kernel is compiled from (its ncu summary is valid for this hash only)
K1_SOURCES = [os.path.join(ROOT, "ring_attention_slope_gb300", "csrc", f)
              for f in ("attn_partial.cu", "sm103_ptx.cuh", "kernels.cuh", "waits.cuh")]


# ---------------------------------------------------------------- helpers

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def k1_source_hash():
    h = hashlib.sha256()
    for path in K1_SOURCES:
        with open(path, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


TRAFFIC_FILE = os.path.join(ROOT, "profiles", "attn_partial_traffic.json")


def profiled_traffic(workload_name, window=0):
    """DRAM bytes per attention launch from the committed ncu record (profiles/attn_partial_traffic.json),
    if that record was taken on the current kernel source; else None."""
    try:
        with open(TRAFFIC_FILE) as f:
            records = json.load(f)
    except (OSError, ValueError):
        return None
    rec = records.get(f"{workload_name}/w{window}")
    if not rec or rec.get("kernel_source_sha256_16") != k1_source_hash():
        return None
    return float(rec["dram_bytes_per_launch"])


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

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
        self.thread.join(timeout=2)
        sm, mx, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
                power.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm), "power_w_max": max(power) if power else None}


def workload_flops(w, window=0):
    return wl.flops(w, window)


def max_over_ranks(x: float, dist=None, device="cpu") -> float:
    """Largest value of x over all ranks (the job's time is its slowest rank's)."""
    import torch

    if dist is None or not dist.is_initialized():
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(flops_per_step: float, steps: int, world: int, ms: float) -> float:
    """Whole-job throughput: every rank runs its own replica of the step (weak scaling)."""
    return flops_per_step * steps * world / (ms * 1e-3) / 1e12


# ---------------------------------------------------------------- CPU oracle legs

def oracle_sample(w, target_s, seed=0):
    """Time the fp64 oracle on a bounded row sample of one KV group; returns (TFLOP/s, seconds, desc, cores)."""
    import torch

    import oracle

    oracle.build()
    q, k, v = wl.workload_qkv(w, device="cpu")
    heads = wl.sample_heads(w)
    rng = np.random.default_rng(w.seed + 101 + seed)
    # calibrate on a small sample, then size the timed sample to ~target_s
    n_rows = 16
    t_cal = 0.0
    while True:
        rows = np.sort(rng.integers(0, w.S, size=n_rows))
        t0 = time.perf_counter()
        oracle.attention(q, k, v, causal=True, rows=rows, heads=heads)
        t_cal = time.perf_counter() - t0
        if t_cal > 0.5 or n_rows >= w.S:
            break
        n_rows = min(w.S, n_rows * 4)
    n_rows = int(min(w.S, max(16, n_rows * target_s / max(t_cal, 1e-3))))
    rows = np.sort(rng.integers(0, w.S, size=n_rows))
    t0 = time.perf_counter()
    oracle.attention(q, k, v, causal=True, rows=rows, heads=heads)
    dt = time.perf_counter() - t0
    pairs = float(np.sum(rows + 1))  # causal: row i sees i + 1 keys
    flops = pairs * len(heads) * 2 * (w.dqk + w.dv)
    desc = (f"{n_rows} random query rows x {len(heads)} heads (one KV group) of {w.name}, "
            f"causal over all earlier keys; fp64 OpenMP oracle")
    del torch
    return flops / dt / 1e12, dt, desc, oracle.num_threads()


def run_reference(args, w):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    per_step = max(2.0, min(20.0, 90.0 / max(1, args.steps)))
    vals, times = [], []
    for s in range(args.warmup):
        oracle_sample(w, min(per_step, 2.0), seed=1000 + s)
    desc, cores = "", 1
    for s in range(args.steps):
        v, dt, desc, cores = oracle_sample(w, per_step, seed=s)
        vals.append(v)
        times.append(dt)
    value = float(np.mean(vals))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * float(np.mean(times)),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "S": w.S, "Hq": w.Hq, "Hkv": w.Hkv, "dqk": w.dqk, "dv": w.dv,
                   "layout": w.layout, "n_chunks": wl.n_chunks(w)},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line))
    return 0


# ---------------------------------------------------------------- GPU leg

# The other full-size configurations, timed in the same default run after the headline workload
# (each with its own clock record): the 64K chunked prefill, the 100K zigzag ring in full causal and
# sliding-window-128 form, and the MLA-shaped chunked prefill.
EXTRA_CONFIGS = [("chunked_prefill_s64k_c12k", 0), ("long_s100k_zigzag16_full_and_w128", 0),
                 ("long_s100k_zigzag16_full_and_w128", 128), ("mla_s64k_d192_192_128_chunked_var", 0)]
EXTRA_TIME_TARGET_MS = 1500.0  # timed work per extra configuration


class Ctx:
    """What every measurement of one bench run shares."""

    def __init__(self, torch, slope, dist, local, peaks, peak_src, args):
        self.torch, self.slope, self.dist, self.local = torch, slope, dist, local
        self.peaks, self.peak_src, self.args = peaks, peak_src, args
        self.world = dist.get_world_size() if dist is not None else 1
        self.stream = torch.cuda.current_stream()

    def barrier(self):
        if self.dist is not None:
            self.dist.barrier()


def k1_roofline(ctx, w, window, flops_step, steps, k1_ms, k1_n, k1_bytes, clocks):
    """The attention kernel against its roof: the measured burst bf16 peak under a full causal mask (the
    kernel is timed in launches of milliseconds, inside short steps at the sampled clock); the measured HBM
    copy rate with a sliding window, where each tile sees a few key tiles only."""
    peaks = ctx.peaks
    k1_tflops = flops_step * steps / (k1_ms * 1e-3) / 1e12
    k1_gbs = k1_bytes * k1_n / (k1_ms * 1e-3) / 1e9
    common = {"traffic": profiled_traffic(w.name, window), "kernel": "attn_partial_kernel", "launches": k1_n,
              "avg_launch_ms": k1_ms / max(1, k1_n), "bytes_per_launch": k1_bytes,
              # one exponential per visible (query, key) pair and query head
              "exp_per_s": flops_step / (2.0 * (w.dqk + w.dv)) * steps / (k1_ms * 1e-3),
              "sm_mhz": clocks.get("sm_mhz")}
    if window == 0:
        r = {"bound": "tensor", "achieved": k1_tflops, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
             "frac": k1_tflops / peaks["bf16_tflops"], "peak_source": f"{ctx.peak_src} bf16_tflops (burst)",
             "achieved_gbs": k1_gbs, **common}
        mhz, mx = clocks.get("sm_mhz"), clocks.get("sm_max_mhz")
        if mhz and mx:
            # note only: the burst peak was measured at the maximum clock
            r["frac_of_peak_at_sampled_clock"] = k1_tflops / (peaks["bf16_tflops"] * mhz / mx)
        return r
    return {"bound": "hbm", "achieved": k1_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": k1_gbs / peaks["hbm_gbs"], "peak_source": f"{ctx.peak_src} hbm_gbs",
            "achieved_tflops": k1_tflops, **common}


def measure_job(ctx, w, window, q, k, v, steps, warmup, flags=()):
    """Times `steps` whole slope_cp_prefill calls (all attention launches + the merge) after `warmup`
    untimed ones, with CUDA events around every launch on the launching stream and the clocks sampled
    during the timed region.  Returns the measured record."""
    torch, slope = ctx.torch, ctx.slope
    sizes = wl.chunk_sizes(w)
    n = wl.n_chunks(w)
    out = torch.empty((w.S, w.Hq, w.dv), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((w.Hq, w.S), dtype=torch.float32, device="cuda")
    ws = torch.empty((slope.cp_prefill_workspace_size(w.S, w.Hq, w.dv, n, w.layout, sizes),), dtype=torch.uint8,
                     device="cuda")
    stream = ctx.stream

    def step():
        slope.cp_prefill(q, k, v, n, w.layout, chunk_sizes=sizes, window=window, out=out, lse=lse, workspace=ws)

    _, launches_per_step, _ = slope.cp_prefill_plan(w.S, n, w.layout, chunk_sizes=sizes, window=window)
    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    st, site = slope.device_status()
    if st != 0:
        raise RuntimeError(f"device status {st} at site {site}")

    # ---- the job: `steps` plain calls between two events (consecutive attention launches of a call
    # overlap their tails, which per-launch events would prevent)
    sampler = ClockSampler(ctx.local)
    sampler.start()
    time.sleep(0.15)
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ctx.barrier()
    torch.cuda.synchronize()
    t_start.record(stream)
    for _ in range(steps):
        step()
    t_end.record(stream)
    torch.cuda.synchronize()
    ctx.barrier()
    clocks = sampler.stop()
    elapsed_ms = max_over_ranks(t_start.elapsed_time(t_end), ctx.dist, "cuda")
    st, site = slope.device_status()
    if st != 0:
        raise RuntimeError(f"device status {st} at site {site}")

    # ---- each kernel's own duration: the same steps again with CUDA events around every launch
    n_pairs = launches_per_step + 8
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_pairs)]
          for _ in range(steps)]
    for step_ev in ev:
        for a, b in step_ev:  # materialise the CUDA events
            a.record(stream)
            b.record(stream)
    torch.cuda.synchronize()
    kinds_all, counts = [], []
    for s in range(steps):
        _, _, nl, kinds = slope.cp_prefill_timed(q, k, v, n, w.layout, ev[s], chunk_sizes=sizes, window=window,
                                                 out=out, lse=lse, workspace=ws)
        counts.append(nl)
        kinds_all.append(kinds)
    torch.cuda.synchronize()
    st, site = slope.device_status()
    if st != 0:
        raise RuntimeError(f"device status {st} at site {site}")

    k1_ms, k2_ms, kf_ms, k1_n, k2_n, kf_n = 0.0, 0.0, 0.0, 0, 0, 0
    for s in range(steps):
        for i in range(counts[s]):
            a, b = ev[s][i]
            d = a.elapsed_time(b)
            if kinds_all[s][i] == 0:  # attention
                k1_ms += d
                k1_n += 1
            elif kinds_all[s][i] == 1:  # merge
                k2_ms += d
                k2_n += 1
            else:  # the -inf fill of the live partial lse planes
                kf_ms += d
                kf_n += 1
    flops_step = workload_flops(w, window)
    merge_bytes = merge_bytes_per_launch(slope, w, n, sizes, window)
    k2_gbs = merge_bytes * k2_n / (k2_ms * 1e-3) / 1e9 if k2_ms > 0 else None
    k1_bytes, k1_launches_per_step = k1_bytes_per_launch(slope, w, n, sizes, window)
    if k1_n != k1_launches_per_step * steps:
        raise RuntimeError(f"attention launches {k1_n} != {k1_launches_per_step} per step x {steps}")
    peaks = ctx.peaks
    roof = k1_roofline(ctx, w, window, flops_step, steps, k1_ms, k1_n, k1_bytes, clocks)
    # The attention launches as they run inside the job, where consecutive launches of a call overlap
    # their tails (programmatic dependent launch), which events around every launch prevent: the job's
    # time less its fill and merge launches (which run the ordinary way in both passes), per launch.
    # Reported beside the per-launch figure, which stays the roofline's `achieved`.
    att_ms = elapsed_ms - k2_ms - kf_ms
    if k1_n and att_ms > 0 and roof.get("achieved"):
        per_launch = att_ms / k1_n
        roof["avg_launch_ms_in_job"] = per_launch
        roof["achieved_in_job"] = roof["achieved"] * roof["avg_launch_ms"] / per_launch
        roof["frac_in_job"] = roof["achieved_in_job"] / roof["peak"]
    rec = {
        "value": job_tflops(flops_step, steps, ctx.world, elapsed_ms), "unit": UNIT,
        "ms_per_step": elapsed_ms / steps, "steps": steps, "warmup": warmup,
        "tokens_per_s": w.S * steps * ctx.world / (elapsed_ms * 1e-3),
        "roofline": roof,
        "roofline_merge": {"bound": "hbm", "achieved": k2_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                           "frac": (k2_gbs / peaks["hbm_gbs"]) if k2_gbs else None,
                           "peak_source": f"{ctx.peak_src} hbm_gbs",
                           "bytes_per_launch": merge_bytes, "kernel": "lse_merge_kernel",
                           "avg_launch_ms": k2_ms / max(1, k2_n),
                           "lse_fill": {"kernel": "lse_fill_kernel", "launches": kf_n,
                                        "avg_launch_ms": kf_ms / max(1, kf_n),
                                        "bytes_per_launch": fill_bytes_per_launch(slope, w, n, sizes, window)}},
        "gpu_launches": int(sum(counts)),
        "clocks": clocks,
        "timing": "value: steps x slope_cp_prefill between two CUDA events; kernel durations: a second pass of "
                  "the same steps through slope_cp_prefill_timed (events around every launch)",
        "config": {"workload": w.name, "S": w.S, "Hq": w.Hq, "Hkv": w.Hkv, "dqk": w.dqk, "dv": w.dv,
                   "layout": w.layout, "n_chunks": n, "window": window, "batch": 1,
                   "l2": f"inputs larger than L2 (Q+K+V {q.numel() * 2 + k.numel() * 2 + v.numel() * 2} B, "
                         f"partials {ws.numel()} B > {L2_BYTES} B); no flush",
                   "flops_per_step": flops_step},
    }
    return rec, ws


def steps_for(ctx, step, target_ms, max_steps, warmup):
    """Number of timed steps that fill about target_ms (at least 3), from the warm-up steps' time."""
    torch = ctx.torch
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(ctx.stream)
    for _ in range(warmup):
        step()
    b.record(ctx.stream)
    torch.cuda.synchronize()
    per = a.elapsed_time(b) / max(1, warmup)
    return int(max(3, min(max_steps, round(target_ms / max(per, 1e-3)))))


def run_gpu(args, w):
    import torch

    import ring_attention_slope_gb300 as slope

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    slope.build()
    slope.load()
    peaks, peak_src = load_peaks()
    ctx = Ctx(torch, slope, dist, local, peaks, peak_src, args)
    window = args.window
    q, k, v = wl.workload_qkv(w, device="cuda")
    sizes = wl.chunk_sizes(w)
    n = wl.n_chunks(w)

    head, ws = measure_job(ctx, w, window, q, k, v, args.steps, args.warmup)
    out = torch.empty((w.S, w.Hq, w.dv), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((w.Hq, w.S), dtype=torch.float32, device="cuda")
    stream = ctx.stream
    variants = {}
    if not args.no_variants:
        # the same attention as one launch (bf16 out, no partials, no merge): the fused single-GPU form
        variants["fused_single_launch"] = run_fused(slope, torch, w, window, q, k, v, stream, args, ctx.barrier,
                                                    dist)
        # the ring / chunked layout with each rank's queries run over all their visible keys in one item
        variants["fused_layout"] = run_fused_layout(slope, torch, w, n, sizes, window, q, k, v, out, lse, stream,
                                                    args, ctx.barrier, dist)
        # the same step with the partials kept in bf16 between the attention launches and the merge
        variants["bf16_partials"] = run_bf16_partials(slope, torch, w, n, sizes, window, q, k, v, out, lse, stream,
                                                      args, ctx.barrier, dist)
        variants["bf16_partials"]["gpu_launches_per_step"] = head["gpu_launches"] // args.steps
        # the same attention in the head-sharded (Ulysses) layout
        variants["ulysses"] = run_ulysses(slope, torch, w, window, q, k, v, out, lse, stream, args, ctx.barrier,
                                          dist)
    # end to end through the public call with pinned host buffers
    e2e = None if args.no_e2e else run_e2e(slope, torch, w, n, sizes, window, q, k, v, ws, stream, args,
                                           ctx.barrier, dist)
    del q, k, v, ws, out, lse
    torch.cuda.empty_cache()

    result = {
        "metric": METRIC, "value": head["value"], "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {**head["config"], "parallelism": f"replicas{world}" if world > 1 else "single"},
        "tokens_per_s": head["tokens_per_s"],
        "pct_of_bf16_peak": 100.0 * head["value"] / world / peaks["bf16_tflops"],
        "roofline": head["roofline"],
        "roofline_merge": head["roofline_merge"],
        "e2e": e2e,
        **variants,
        "gpu_launches": head["gpu_launches"],
        "clocks": head["clocks"],
    }

    # ---- the other full-size configurations, each with its own clock record
    if not args.only_workload:
        configs = {}
        for name, win in EXTRA_CONFIGS:
            wx = wl.BY_NAME[name]
            configs[f"{name}/w{win}"] = run_extra(ctx, wx, win, args)
            torch.cuda.empty_cache()
        result["configs"] = configs
        result["gate"] = gate_summary(result)

    if rank == 0 and not args.no_cpu_baseline:
        v_cpu, dt, desc, cores = oracle_sample(w, args.cpu_seconds)
        result["cpu_baseline"] = {"value": v_cpu, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc,
                                  "seconds": dt}
    if rank == 0:
        print(json.dumps(result))
    if dist is not None:
        dist.destroy_process_group()
    return 0


def run_extra(ctx, w, window, args):
    """One more full-size configuration: the whole job (attention launches + merge) with its attention and
    merge rooflines, its fused-layout form and, for the MLA-shaped workload, the host-buffer end to end."""
    torch, slope = ctx.torch, ctx.slope
    q, k, v = wl.workload_qkv(w, device="cuda")
    sizes = wl.chunk_sizes(w)
    n = wl.n_chunks(w)
    out = torch.empty((w.S, w.Hq, w.dv), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((w.Hq, w.S), dtype=torch.float32, device="cuda")
    ws0 = torch.empty((slope.cp_prefill_workspace_size(w.S, w.Hq, w.dv, n, w.layout, sizes),), dtype=torch.uint8,
                      device="cuda")

    def step():
        slope.cp_prefill(q, k, v, n, w.layout, chunk_sizes=sizes, window=window, out=out, lse=lse, workspace=ws0)

    steps = steps_for(ctx, step, EXTRA_TIME_TARGET_MS, args.steps, args.warmup)
    del ws0
    rec, ws = measure_job(ctx, w, window, q, k, v, steps, args.warmup)
    sub = argparse.Namespace(**{**vars(args), "steps": steps})
    if not args.no_variants:
        rec["fused_layout"] = run_fused_layout(slope, torch, w, n, sizes, window, q, k, v, out, lse, ctx.stream, sub,
                                               ctx.barrier, ctx.dist)
    if w.layout == "chunked" and not args.no_variants:
        rec["dck"] = run_dck(slope, torch, w, window, q, k, v, out, lse, ctx.stream, sub, ctx.barrier, ctx.dist)
    if not args.no_e2e and w.dqk != w.dv:
        rec["e2e"] = run_e2e(slope, torch, w, n, sizes, window, q, k, v, ws, ctx.stream,
                             argparse.Namespace(**{**vars(args), "steps": max(steps, 10)}), ctx.barrier, ctx.dist)
    del q, k, v, out, lse, ws
    return rec


def gate_summary(result):
    """Each configuration's attention-kernel fraction and merge fraction of its measured roof."""
    rows = {f"{result['config']['workload']}/w{result['config']['window']}": result}
    rows.update(result.get("configs", {}))
    return {key: {"k1_frac": r["roofline"]["frac"], "k1_bound": r["roofline"]["bound"],
                  "k1_frac_in_job": r["roofline"].get("frac_in_job"),
                  "merge_frac": r["roofline_merge"]["frac"], "job_tflops": r["value"],
                  "sm_mhz": r["clocks"].get("sm_mhz"), "reasons": r["clocks"].get("reasons")}
            for key, r in rows.items()}


def merge_bytes_per_launch(slope, w, n, sizes, window):
    """Algorithmic DRAM bytes of one merge launch, exact, from the launch plan.

    The merge reads, for every row and head, the lse of each merged plane and the fp32
    partial output of the planes in which that row saw at least one key, and writes the
    bf16 output and fp32 lse.  A plane none of whose rows sees a key is not merged.  In
    the ring and chunked layouts a row's position is its row index, so a row of a plan
    item is live when one of the item's key ranges, cut to the causal limit (key <= row)
    and the window (row - key < window), is not empty.
    """
    items, _, n_planes = slope.cp_prefill_plan(w.S, n, w.layout, chunk_sizes=sizes, causal=True, window=window)
    live_rows = np.zeros(n_planes, dtype=np.int64)
    plane_live = np.zeros(n_planes, dtype=bool)
    plane_live[0] = True
    for it in items:
        if it["kv"]:
            plane_live[it["plane"]] = True
        q = np.arange(it["q_row0"], it["q_row0"] + it["q_len"], dtype=np.int64)
        seen = np.zeros(q.shape, dtype=bool)
        for k0, ln in it["kv"]:
            lo = np.maximum(k0, q - window + 1) if window > 0 else np.full(q.shape, k0)
            hi = np.minimum(k0 + ln - 1, q)
            seen |= lo <= hi
        live_rows[it["plane"]] += int(seen.sum())
    reads = int(plane_live.sum()) * w.S * 4 + int(live_rows[plane_live].sum()) * w.dv * 4
    return float(w.Hq * (reads + w.S * (w.dv * 2 + 4)))


def fill_bytes_per_launch(slope, w, n, sizes, window):
    """Bytes the lse fill writes per call: -inf into every live partial plane's lse ([S, Hq] fp32)."""
    items, _, n_planes = slope.cp_prefill_plan(w.S, n, w.layout, chunk_sizes=sizes, causal=True, window=window)
    live = {0} | {it["plane"] for it in items if it["kv"]}
    return float(len(live) * w.S * w.Hq * 4)


def launch_groups(items, n_launch):
    """Plan launches (ring steps, chunks, ranks) grouped into kernel launches by the library's rule:
    consecutive ones share a launch while their items fit in 32; a partial plane none of whose items sees
    a key is dropped (plane 0 is always kept)."""
    live_planes = {0} | {it["plane"] for it in items if it["kv"]}
    by_launch = {}
    for it in items:
        if it["plane"] in live_planes:
            by_launch.setdefault(it["launch"], []).append(it)
    groups, cur = [], []
    for lch in range(n_launch):
        step = by_launch.get(lch, [])
        if cur and len(cur) + len(step) > 32:
            groups.append(cur)
            cur = []
        cur = cur + step
    if cur:
        groups.append(cur)
    return groups


def k1_bytes_per_launch(slope, w, n, sizes, window):
    """Algorithmic DRAM bytes of an average attention launch of one step, from the plan.

    Plan launches (ring steps, chunks) are grouped into kernel launches by the library's rule:
    consecutive steps share a launch while their live items fit in 32 (a plane none of whose
    items sees a key is dropped).  Per kernel launch: each distinct Q row that sees a key and
    each distinct K/V row is read once, and every item writes its fp32 partial out + lse for
    rows that see a key, or its lse alone for rows that see none.
    Returns (bytes per launch, launches per step).
    """
    items, n_launch, _ = slope.cp_prefill_plan(w.S, n, w.layout, chunk_sizes=sizes, causal=True, window=window)
    groups = launch_groups(items, n_launch)
    total = 0.0
    for g in groups:
        qrows = np.zeros(w.S, dtype=bool)
        kvrows = np.zeros(w.S, dtype=bool)
        writes = 0
        for it in g:
            q = np.arange(it["q_row0"], it["q_row0"] + it["q_len"], dtype=np.int64)
            seen = np.zeros(q.shape, dtype=bool)
            for k0, ln in it["kv"]:
                lo = np.maximum(k0, q - window + 1) if window > 0 else np.full(q.shape, k0)
                seen |= lo <= np.minimum(k0 + ln - 1, q)
                kvrows[k0:k0 + ln] = True
            qrows[q[seen]] = True
            n_seen = int(seen.sum())
            writes += n_seen * w.Hq * (w.dv * 4 + 4) + (it["q_len"] - n_seen) * w.Hq * 4
        total += int(qrows.sum()) * w.Hq * w.dqk * 2 + int(kvrows.sum()) * w.Hkv * (w.dqk + w.dv) * 2 + writes
    return total / len(groups), len(groups)


def run_fused(slope, torch, w, window, q, k, v, stream, args, barrier, dist):
    """The whole causal attention as one attention launch over the full sequence (bf16 out): every query
    tile runs the online softmax over all of its visible keys, with no partials and no merge."""
    out = torch.empty((w.S, w.Hq, w.dv), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((w.Hq, w.S), dtype=torch.float32, device="cuda")

    def step():
        slope.attn_partial(q, k, v, causal=True, window=window, out=out, lse=lse)

    for _ in range(max(1, args.warmup)):
        step()
    torch.cuda.synchronize()
    barrier()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(args.steps):
        step()
    b.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(a.elapsed_time(b), dist, "cuda")
    world = dist.get_world_size() if dist is not None else 1
    return {"value": job_tflops(workload_flops(w, window), args.steps, world, ms), "unit": UNIT,
            "ms_per_step": ms / args.steps, "api": "slope_attn_partial over the whole sequence, bf16 out",
            "gpu_launches_per_step": 1}


def run_fused_layout(slope, torch, w, n, sizes, window, q, k, v, out, lse, stream, args, barrier, dist):
    """The workload's own layout with SLOPE_CP_FUSED: every rank's (or chunk's) query rows attend to all of
    their visible keys in one work item, merged online in the kernel (no partial planes, no merge launch)."""
    nbytes = slope.cp_prefill_workspace_size(w.S, w.Hq, w.dv, n, w.layout, sizes, fused=True)
    wsf = torch.empty((max(nbytes, 256),), dtype=torch.uint8, device="cuda")

    def step():
        slope.cp_prefill(q, k, v, n, w.layout, chunk_sizes=sizes, window=window, out=out, lse=lse, workspace=wsf,
                         fused=True)

    ms, world = time_variant(torch, step, stream, args, barrier, dist)
    items, n_launch, _ = slope.cp_prefill_plan(w.S, n, w.layout, chunk_sizes=sizes, window=window, fused=True)
    return {"value": job_tflops(workload_flops(w, window), args.steps, world, ms), "unit": UNIT,
            "ms_per_step": ms / args.steps, "api": "slope_cp_prefill_ex(SLOPE_CP_FUSED)",
            "gpu_launches_per_step": len(launch_groups(items, n_launch))}


def run_dck(slope, torch, w, window, q, k, v, out, lse, stream, args, barrier, dist):
    """The chunked workload with dynamic chunk sizes (slope_dck_chunk_sizes: initial 12288, smoothing 0.65),
    as partials + merge and in the fused form."""
    sizes = slope.dck_chunk_sizes(w.S, 12288, 0.65)
    n = len(sizes)
    res = {"chunks": n, "first": sizes[0], "last_full": sizes[-2] if n > 1 else sizes[0],
           "api": "slope_dck_chunk_sizes(S, 12288, 0.65) -> slope_cp_prefill(SLOPE_LAYOUT_CHUNKED)"}
    ws = torch.empty((slope.cp_prefill_workspace_size(w.S, w.Hq, w.dv, n, "chunked", sizes),), dtype=torch.uint8,
                     device="cuda")

    def step():
        slope.cp_prefill(q, k, v, n, "chunked", chunk_sizes=sizes, window=window, out=out, lse=lse, workspace=ws)

    ms, world = time_variant(torch, step, stream, args, barrier, dist)
    res["value"] = job_tflops(workload_flops(w, window), args.steps, world, ms)
    res["unit"] = UNIT
    res["ms_per_step"] = ms / args.steps
    del ws
    res["fused_layout"] = run_fused_layout(slope, torch, w, n, sizes, window, q, k, v, out, lse, stream, args,
                                           barrier, dist)
    return res


def time_variant(torch, step, stream, args, barrier, dist):
    """(ms per step, world size) of `step` run args.steps times after its warm-up, device-timed on `stream`."""
    for _ in range(max(1, args.warmup)):
        step()
    torch.cuda.synchronize()
    barrier()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(args.steps):
        step()
    b.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(a.elapsed_time(b), dist, "cuda")
    return ms, dist.get_world_size() if dist is not None else 1


def run_bf16_partials(slope, torch, w, n, sizes, window, q, k, v, out, lse, stream, args, barrier, dist):
    """The benchmark step with SLOPE_CP_BF16_PARTIALS: the same launches, the partial outputs written and
    merged as bf16 (half the workspace, half the merge's partial reads)."""
    nbytes = slope.cp_prefill_workspace_size(w.S, w.Hq, w.dv, n, w.layout, sizes, bf16_partials=True)
    ws16 = torch.empty((nbytes,), dtype=torch.uint8, device="cuda")

    def step():
        slope.cp_prefill(q, k, v, n, w.layout, chunk_sizes=sizes, window=window, out=out, lse=lse, workspace=ws16,
                         bf16_partials=True)

    ms, world = time_variant(torch, step, stream, args, barrier, dist)
    return {"value": job_tflops(workload_flops(w, window), args.steps, world, ms), "unit": UNIT,
            "ms_per_step": ms / args.steps, "api": "slope_cp_prefill_ex(SLOPE_CP_BF16_PARTIALS)",
            "workspace_bytes": nbytes}


def run_ulysses(slope, torch, w, window, q, k, v, out, lse, stream, args, barrier, dist):
    """The same attention in the head-sharded (Ulysses) layout at the largest degree GQA allows
    (one KV head per rank): every rank's whole-sequence attention of its head group, no merge."""
    U = w.Hkv if w.Hkv <= 32 else 32
    while w.Hkv % U:
        U -= 1
    nbytes = slope.cp_prefill_workspace_size(w.S, w.Hq, w.dv, U, "ulysses")
    wsu = torch.empty((nbytes,), dtype=torch.uint8, device="cuda")

    def step():
        slope.cp_prefill(q, k, v, U, "ulysses", window=window, out=out, lse=lse, workspace=wsu)

    ms, world = time_variant(torch, step, stream, args, barrier, dist)
    return {"value": job_tflops(workload_flops(w, window), args.steps, world, ms), "unit": UNIT,
            "ms_per_step": ms / args.steps, "api": f"slope_cp_prefill(SLOPE_LAYOUT_ULYSSES, n_chunks={U})",
            "ranks": U, "gpu_launches_per_step": (U + 31) // 32}


def run_e2e(slope, torch, w, n, sizes, window, q, k, v, ws, stream, args, barrier, dist):
    """The metric through the host-buffer call: every step copies its inputs from pinned host memory and its
    result back.  Two device-buffer sets alternate over three streams, so the copies of one step overlap the
    compute of its neighbours (the library orders each buffer set's reuse); a timed window runs from the
    first step's input copies to the last step's output copies, and the median of three windows is kept."""
    hq = torch.empty(q.shape, dtype=q.dtype, pin_memory=True)
    hk = torch.empty(k.shape, dtype=k.dtype, pin_memory=True)
    hv = torch.empty(v.shape, dtype=v.dtype, pin_memory=True)
    hq.copy_(q)
    hk.copy_(k)
    hv.copy_(v)
    sets = []
    for _ in range(2):
        sets.append({"q": torch.empty_like(q), "k": torch.empty_like(k), "v": torch.empty_like(v),
                     "out": torch.empty((w.S, w.Hq, w.dv), dtype=torch.bfloat16, device="cuda"),
                     "lse": torch.empty((w.Hq, w.S), dtype=torch.float32, device="cuda"),
                     "hout": torch.empty((w.S, w.Hq, w.dv), dtype=torch.bfloat16, pin_memory=True),
                     "hlse": torch.empty((w.Hq, w.S), dtype=torch.float32, pin_memory=True)})
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()

    def step(i):
        b = sets[i % 2]
        slope.cp_prefill_host(hq, hk, hv, b["hout"], b["hlse"], b["q"], b["k"], b["v"], b["out"], b["lse"], n,
                              w.layout, chunk_sizes=sizes, window=window, workspace=ws, copy_in_stream=s_in,
                              compute_stream=stream, copy_out_stream=s_out)

    for i in range(max(1, args.warmup)):
        step(i)
    torch.cuda.synchronize()
    barrier()
    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    time.sleep(0.15)
    # three timed windows of `steps` steps each; the host link is shared with the machine's other
    # jobs and an occasional window runs slower, so the median window is the reported one
    windows = []
    for _ in range(3):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(s_in)
        for i in range(args.steps):
            step(i)
        b.record(s_out)
        torch.cuda.synchronize()
        windows.append(max_over_ranks(a.elapsed_time(b), dist, "cuda"))
    clocks = sampler.stop()
    ms = sorted(windows)[1]
    world = dist.get_world_size() if dist is not None else 1
    val = job_tflops(workload_flops(w, window), args.steps, world, ms)
    h2d = int(hq.numel() * 2 + hk.numel() * 2 + hv.numel() * 2)
    d2h = int(sets[0]["hout"].numel() * 2 + sets[0]["hlse"].numel() * 4)

    # the copies alone, on the same buffers and streams: with the copies overlapped, a step takes about
    # the longest of the input copies, the compute and the output copies
    def copy_ms(fn, st, reps=3):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        for _ in range(reps):
            fn()
        e1.record(st)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps

    b0 = sets[0]

    def h2d_copy():
        with torch.cuda.stream(s_in):
            b0["q"].copy_(hq, non_blocking=True)
            b0["k"].copy_(hk, non_blocking=True)
            b0["v"].copy_(hv, non_blocking=True)

    def d2h_copy():
        with torch.cuda.stream(s_out):
            b0["hout"].copy_(b0["out"], non_blocking=True)
            b0["hlse"].copy_(b0["lse"], non_blocking=True)

    h2d_ms, d2h_ms = copy_ms(h2d_copy, s_in), copy_ms(d2h_copy, s_out)
    return {"value": val, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": ms / args.steps, "windows_ms_per_step": [x / args.steps for x in windows],
            "api": "slope_cp_prefill_host",
            "overlap": "2 device-buffer sets; input copies, compute and output copies on 3 streams",
            "h2d_alone_ms": h2d_ms, "h2d_gbs": h2d / (h2d_ms * 1e-3) / 1e9,
            "d2h_alone_ms": d2h_ms, "d2h_gbs": d2h / (d2h_ms * 1e-3) / 1e9, "clocks": clocks}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["slope", "reference"], default="slope")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(wl.BY_NAME))
    ap.add_argument("--window", type=int, default=0)
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg (profiling runs)")
    ap.add_argument("--no-variants", action="store_true",
                    help="skip the fused, bf16-partial and Ulysses legs (profiling runs)")
    ap.add_argument("--only-workload", action="store_true",
                    help="time the chosen workload alone, not the other full-size configurations after it")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("at least 3 warm-up steps")
    w = wl.BY_NAME[args.workload]
    if args.impl == "reference":
        return run_reference(args, w)
    return run_gpu(args, w)


if __name__ == "__main__":
    sys.exit(main())
