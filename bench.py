#!/usr/bin/env python3
"""FP32 GEMM bench on one GB300 (or N replicas, one per GPU).

One step = one call of the library's GEMM (gemm_f32_ex, mode AUTO unless
--mode) on the workload's inputs, which are resident in HBM.  Timing follows
the course page's cudaEvent method ("Project - tiled matrix multiply",
section "Starter scaffolding": warm-up outside the measurement, events on
the launching stream, transfers excluded) with W warm-up steps and K timed
steps; inputs are rotated over several buffer sets whose total size exceeds
the 129 MB L2, so each step starts with cold inputs.

Prints one JSON line (rank 0).  --impl reference times the CPU oracle on a
bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "FP32 GEMM TFLOP/s (2MNK/t) at N=4096/8192 and % of GB300 FP32/TF32/HBM roofline"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# dense TF32 / dense BF16 tensor rate on GB300 (nominal 1.1 vs 2.25 PFLOP/s)
TF32_OVER_BF16 = 1.1 / 2.25


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="sq4096")
    ap.add_argument("--mode", default="auto")
    ap.add_argument("--no-extras", action="store_true", help="skip per-mode and reference points")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--calibrate-only", action="store_true",
                    help="run only the HBM copy calibration (2 x 1 GiB buffers) and print GB/s")
    return ap.parse_args()


# --------------------------------------------------------------- helpers

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(x: float, world: int, dev) -> float:
    """The largest of every rank's `x` (a time), identical on all ranks."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(flops_per_step: float, steps: int, world: int, ms_max: float) -> float:
    """Aggregate throughput: every rank ran `steps` steps of `flops_per_step`
    (replicas, weak scaling), timed by the slowest rank."""
    return world * steps * flops_per_step / (ms_max * 1e-3) / 1e12


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 200 ms."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        smax = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in rows:
            for i, n in enumerate(names):
                if r[5 + i].lower().startswith("active"):
                    reasons.add(n)
        power = [num(r[3]) for r in rows if num(r[3]) is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(rows),
                "power_w_max": max(power) if power else None}


def code_only(text: str) -> str:
    """C/CUDA source with comments and blank lines removed, so that editing
    a comment does not mark a kernel's counters stale."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    lines = (re.sub(r"//.*$", "", l).rstrip() for l in text.splitlines())
    return "\n".join(l for l in lines if l)


def source_hash(paths):
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), encoding="utf-8") as f:
            h.update(code_only(f.read()).encode())
    return h.hexdigest()[:16]


# Sources whose change invalidates a kernel's recorded DRAM counters: the
# kernel itself, what it includes, and the planner that picks its launch.
TRAFFIC_SOURCES = {
    "tc": ["roofline_gb300/csrc/tc_tf32x3.cu", "roofline_gb300/csrc/tc_common.cuh",
           "roofline_gb300/csrc/common.cuh", "roofline_gb300/csrc/plan.cu"],
    "simt": ["roofline_gb300/csrc/simt.cu", "roofline_gb300/csrc/common.cuh",
             "roofline_gb300/csrc/plan.cu"],
}


def kernel_instance(plan, b_stored_nk=False) -> str:
    """The template instantiation and launch shape a plan runs, e.g.
    ``tc_tf32x3_kernel<128,256,16,5,2,0,3,0> grid=152 stream_k=1``.  The
    last template value says how B is split: 0 by the pass, 1 on chip as
    stored N x K, 2 on chip transposed from K x N (the bench's row-major B)."""
    k = plan["kernel_name"]
    if k in ("tc_tf32x3", "tc_tf32"):
        ak = 0 if not plan["a_split_in_kernel"] else (2 if plan["a_hi_tmem"] else 1)
        nprod = 1 if k == "tc_tf32" else 3
        br = 0 if not plan.get("b_split_in_kernel", 0) else (1 if b_stored_nk else 2)
        inst = (f"tc_tf32x3_kernel<{plan['bm']},{plan['bn']},{plan['bk']},{plan['stages']},"
                f"{ak},{int(plan['b_concat'])},{nprod},{br}>")
    elif k == "simt":
        inst = (f"simt_packed_kernel<{plan['bm']},{plan['bn']},{plan['bk']},{plan['stages']},"
                f"{int(plan['vec'])},0,0>")
    else:
        inst = k
    return f"{inst} grid={plan['grid_ctas']} split_k={plan['split_k']} stream_k={plan['stream_k']}"


def ncu_traffic(plan, workload: str):
    """DRAM bytes per launch of exactly this instantiation and launch shape on
    this workload, from the committed ncu summaries, or None when absent or
    when a source it depends on changed after the counters were taken."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    key = f"{kernel_instance(plan)} @ {workload}"
    try:
        with open(path) as f:
            d = json.load(f)
    except Exception:
        return None, f"no profiles/traffic.json entry for {key}"
    e = d.get(key)
    if e is None:
        return None, f"no profiles/traffic.json entry for {key}"
    if e.get("source_hash") != source_hash(e["sources"]):
        return None, f"stale: sources of {key} changed after the capture"
    return float(e["dram_bytes_per_launch"]), e.get("note", "")


class Stamps:
    """Device int64 pairs for gemm_set_profile_stamps: pair i receives the
    earliest start and latest end (GPU %globaltimer, ns) of the main kernel
    of the call made while it was set."""

    def __init__(self, n, dev):
        import torch
        self.t = torch.empty((n, 2), dtype=torch.int64, device=dev)
        self.reset()

    def reset(self):
        self.t[:, 0] = -1  # all ones: the atomic minimum's identity
        self.t[:, 1] = 0

    def ptr(self, i):
        return self.t.data_ptr() + 16 * i

    def ms(self, n=None):
        v = self.t[:n].cpu().numpy().view("uint64").astype("float64")
        return [(e - b) * 1e-6 for b, e in v]


# --------------------------------------------------------------- oracle timing

def time_oracle_rows(A, B, C0, w, rows: int):
    """Runs the oracle on the first `rows` output rows; returns seconds."""
    import oracle
    c0 = None if C0 is None else C0[:rows, :w.N]
    t0 = time.perf_counter()
    oracle.gemm(A[:rows, :w.K], B[:, :w.N], w.alpha, w.beta, c0, M=rows)
    return time.perf_counter() - t0


def oracle_sample_rows(A, B, C0, w, target_s: float):
    import oracle
    cores = oracle.max_threads()
    r0 = min(w.M, max(2 * cores, 16))
    t0 = time_oracle_rows(A, B, C0, w, r0)
    rows = int(r0 * target_s / max(t0, 1e-6))
    rows = max(r0, min(w.M, rows))
    return rows, cores


def single_core_512():
    """The oracle on one core over the whole 512^3 product: seconds."""
    import oracle
    from workloads import WORKLOADS
    w = WORKLOADS["sq512"]
    A, B, _ = w.make()
    t0 = time.perf_counter()
    oracle.gemm(A[:, :w.K], B[:, :w.N], 1.0, 0.0, None, nthreads=1)
    return time.perf_counter() - t0


def cpu_baseline(A, B, C0, w, target_s=12.0):
    rows, cores = oracle_sample_rows(A, B, C0, w, target_s / 4)
    t = time_oracle_rows(A, B, C0, w, rows)
    flops = 2.0 * rows * w.N * w.K
    t1 = single_core_512()
    return {"value": flops / t / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"first {rows} of {w.M} output rows of {w.name} (all N={w.N}, K={w.K}), "
                      f"fp64 accumulation, {t:.2f} s",
            "single_core_512": {"seconds": t1, "gflops": 2 * 512 ** 3 / t1 / 1e9}}


# --------------------------------------------------------------- reference arm

def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    from workloads import WORKLOADS
    w = WORKLOADS[args.workload]
    A, B, C0 = w.make()
    per_step = min(3.0, 150.0 / max(1, args.steps + args.warmup))
    rows, cores = oracle_sample_rows(A, B, C0, w, per_step)
    for _ in range(args.warmup):
        time_oracle_rows(A, B, C0, w, rows)
    ts = [time_oracle_rows(A, B, C0, w, rows) for _ in range(args.steps)]
    total = sum(ts)
    flops = 2.0 * rows * w.N * w.K * args.steps
    value = flops / total / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": total / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w, args.mode, rotation_of(w)[2]),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": f"each step: first {rows} of {w.M} output rows of {w.name} "
                                   f"(all N, all K), fp64 accumulation"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------- our arm

# Main-kernel durations averaged for each roofline entry (at least this many
# launches whatever --steps is).
KERNEL_SAMPLES = 50


def workload_config(w, mode, rotation):
    cfg = {"workload": f"{w.name}: {w.description}", "M": w.M, "N": w.N, "K": w.K,
           "alpha": w.alpha, "beta": w.beta, "layout": "row-major", "mode": mode}
    if rotation is not None:
        cfg["l2"] = rotation
    return cfg


class Caller:
    """One library call per step on rotating device input sets, through the
    C ABI with the pointers and stream resolved once (gemm_f32_ex)."""

    def __init__(self, w, mode, sets):
        import torch

        from roofline_gb300 import gemm
        self.gemm = gemm
        self.lib = gemm.load()
        self.w = w
        self.mode = gemm._mode(mode)
        lda, ldb, ldc = w.lds()
        self.args = [(a.data_ptr(), b.data_ptr(), c.data_ptr()) for a, b, c in sets]
        self.lds = (lda, ldb, ldc)
        self.stream = torch.cuda.current_stream()
        self.handle = self.stream.cuda_stream

    def __call__(self, i):
        a, b, c = self.args[i % len(self.args)]
        lda, ldb, ldc = self.lds
        w = self.w
        rc = self.lib.gemm_f32_ex(w.M, w.N, w.K, w.alpha, a, lda, b, ldb, w.beta, c, ldc,
                                  self.mode, None, 0, self.handle)
        if rc != 0:
            raise self.gemm.GemmError(rc, "gemm_f32_ex")


def stamped_run(call, stamps, first, count):
    """Calls first .. first+count-1, main kernel of call i stamped into pair i."""
    from roofline_gb300 import gemm
    lib = gemm.load()
    for i in range(first, first + count):
        lib.gemm_set_profile_stamps(stamps.ptr(i))
        call(i)
    lib.gemm_set_profile_stamps(None)


def event_kernel_ms(call, n):
    """Cross-check in another launch mode: CUDA events recorded by the library
    around the main kernel (which puts that kernel in plain stream order),
    mean over n calls."""
    import torch

    from roofline_gb300 import gemm
    s = torch.cuda.current_stream()
    eb = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    ea = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    for e in eb + ea:  # torch creates the underlying cudaEvent on first record
        e.record(s)
    torch.cuda.synchronize()
    for i in range(n):
        gemm.set_profile_events(eb[i], ea[i])
        call(i)
    gemm.set_profile_events(None, None)
    torch.cuda.synchronize()
    return statistics.mean(eb[i].elapsed_time(ea[i]) for i in range(n))


def run_ours(args):
    import torch
    import torch.distributed as dist

    from roofline_gb300 import gemm
    from workloads import WORKLOADS

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    gemm.load()
    info = gemm.device_info(local)
    peaks, peaks_src = measured_peaks()

    w = WORKLOADS[args.workload]
    lda, ldb, ldc = w.lds()
    A, B, C0 = w.make()
    sets, set_bytes = device_sets(w, dev, (A, B, C0))
    rotation = rotation_of(w)[2]

    plan = gemm.plan(w.M, w.N, w.K, lda, ldb, ldc, args.mode, 0, w.beta != 0.0)
    stream = torch.cuda.current_stream()
    step = Caller(w, args.mode, sets)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()

    sampler = ClockSampler(local)
    sampler.start()
    # a little untimed load so the clock record reflects the loaded state
    t_pre = time.perf_counter()
    i = 0
    while time.perf_counter() - t_pre < 0.5:
        step(i)
        i += 1
        if i % 16 == 0:
            torch.cuda.synchronize()
    torch.cuda.synchronize()

    # The timed region: K steps in the library's production launch order.
    # Each step's main kernel also stamps its start and end into its own pair
    # (%globaltimer, atomics in the kernel; the launch order is unchanged),
    # and the stamping continues, untimed, for the steps that follow until
    # there are KERNEL_SAMPLES pairs, all in one back-to-back stream of calls.
    n_stamped = max(args.steps, KERNEL_SAMPLES)
    stamps = Stamps(n_stamped, dev)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    start.record(stream)
    stamped_run(step, stamps, 0, args.steps)
    end.record(stream)
    stamped_run(step, stamps, args.steps, n_stamped - args.steps)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    ms_total = start.elapsed_time(end)
    if gemm.check_status() != gemm.OK:
        raise RuntimeError("device status reported an error during the timed region")
    main_ms = stamps.ms()

    t_max = max_over_ranks(ms_total, world, dev)
    flops = float(w.flops)
    value = whole_job_tflops(flops, args.steps, world, t_max)
    ms_step = t_max / args.steps

    # roofline of the dominant (main GEMM) kernel
    main_avg = statistics.mean(main_ms)
    roof = roofline_for(plan, w, main_avg, info, peaks, peaks_src)
    roof["kernel_timing"] = (
        f"mean of {len(main_ms)} launches: the main kernel's first-CTA start to last-CTA end "
        f"(%globaltimer stamps written by the kernel) in the {args.steps} timed steps and the "
        f"{n_stamped - args.steps} steps issued right after them, same launch order "
        f"(programmatic dependent launch on)")
    roof["kernel_ms_timed_steps"] = statistics.mean(main_ms[:args.steps])
    roof["kernel_ms_best"] = min(main_ms)
    roof["achieved_best"] = roof["achieved"] * main_avg / min(main_ms)
    roof["kernel_ms_events_plain_order"] = event_kernel_ms(step, KERNEL_SAMPLES)

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded SplitMix64 inputs, workload shapes and distributions)",
        "config": workload_config(w, args.mode, rotation),
        "plan": {k: plan[k] for k in ("kernel_name", "bm", "bn", "bk", "stages", "split_k",
                                      "stream_k", "a_split_in_kernel", "b_concat", "vec",
                                      "launches", "grid_ctas", "ctas_per_sm", "bound_name")},
        "gpu_launches": args.steps * int(plan["launches"]),
        "roofline": roof,
        "clocks": clocks,
        "device": {"name": info["name"], "sm_count": info["sm_count"],
                   "max_sm_mhz": info["clock_khz"] / 1e3,
                   "fp32_peak_tflops": info["fp32_peak_tflops"]},
        "peaks_source": peaks_src,
    }
    if clocks and clocks.get("sm_mhz"):
        line["roofline"]["frac_at_observed_clock"] = (
            roof["frac"] * (clocks["sm_max_mhz"] or info["clock_khz"] / 1e3) / clocks["sm_mhz"]
            if roof["bound"] != "hbm" else None)

    # end to end: host buffers in, result back to the host, every step
    if not args.no_e2e:
        line["e2e"] = e2e(args, w, A, B, C0, dev, world)

    if rank == 0 and not args.no_extras:
        line["extras"] = extras(args, w, sets, info, peaks, peaks_src)
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(A, B, C0, w)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def link_ms(h2d_bytes, d2h_bytes, dev, reps=5):
    """Time to move h2d_bytes host->device and d2h_bytes device->host between
    pinned host buffers and device memory, the two directions concurrently on
    two streams (the copy engines the library's host call uses): best of
    `reps`, CUDA events.  Also each direction alone."""
    import torch
    hi = torch.empty(h2d_bytes // 4, dtype=torch.float32).pin_memory()
    di = torch.empty_like(hi, device=dev)
    do = torch.empty(d2h_bytes // 4, dtype=torch.float32, device=dev)
    ho = torch.empty(do.numel(), dtype=torch.float32).pin_memory()
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    cur = torch.cuda.current_stream(dev)

    def timed(fn):
        best = None
        for _ in range(reps + 1):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize(dev)
            e0.record(cur)
            fn()
            e1.record(cur)
            torch.cuda.synchronize(dev)
            t = e0.elapsed_time(e1)
            best = t if best is None else min(best, t)
        return best

    def both():
        s_in.wait_stream(cur)
        s_out.wait_stream(cur)
        with torch.cuda.stream(s_in):
            di.copy_(hi, non_blocking=True)
        with torch.cuda.stream(s_out):
            ho.copy_(do, non_blocking=True)
        cur.wait_stream(s_in)
        cur.wait_stream(s_out)

    res = {"both_ms": timed(both),
           "h2d_ms": timed(lambda: di.copy_(hi, non_blocking=True)),
           "d2h_ms": timed(lambda: ho.copy_(do, non_blocking=True))}
    del hi, di, do, ho
    return res


def e2e(args, w, A, B, C0, dev, world):
    """The metric measured through the host-buffer C-ABI call gemm_f32_host:
    A, B (and C when beta != 0) in pinned host memory, copied in, multiplied
    and copied back inside the call (blocks pipelined over copy and compute
    streams).  Timed on the host around whole blocking calls.  Its roof is the
    host link: the same bytes moved in both directions at once, measured in
    the same run."""
    import torch
    import torch.distributed as dist

    from roofline_gb300 import gemm
    lda, ldb, ldc = w.lds()
    hA = torch.from_numpy(A).pin_memory()
    hB = torch.from_numpy(B).pin_memory()
    hC = torch.from_numpy(C0).pin_memory() if C0 is not None else \
        torch.empty((w.M, ldc), dtype=torch.float32).pin_memory()
    steps = max(3, min(args.steps, 30))

    def one():
        rc = gemm.gemm_f32_host(w.M, w.N, w.K, w.alpha, hA.data_ptr(), lda, hB.data_ptr(), ldb,
                                w.beta, hC.data_ptr(), ldc, args.mode, 0)
        if rc != gemm.OK:
            raise gemm.GemmError(rc, "gemm_f32_host")

    for _ in range(3):
        one()
    if world > 1:
        dist.barrier()
    t0 = time.perf_counter()
    for _ in range(steps):
        one()
    ms = max_over_ranks((time.perf_counter() - t0) * 1e3, world, dev)
    h2d = 4 * (w.M * w.K + w.K * w.N + (w.M * w.N if w.beta != 0 else 0))
    d2h = 4 * w.M * w.N
    out = {"value": whole_job_tflops(float(w.flops), steps, world, ms), "unit": "TFLOP/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
           "ms_per_step": ms / steps,
           "path": "pinned host -> gemm_f32_host (blocks: H2D copy stream, GEMM stream, "
                   "D2H copy stream) -> pinned host; host wall clock around blocking calls"}
    try:
        lk = link_ms(h2d, d2h, dev)
        call_ms = ms / steps
        out["roofline"] = {
            "bound": "host_link", "achieved": (h2d + d2h) / (call_ms * 1e-3) / 1e9,
            "peak": (h2d + d2h) / (lk["both_ms"] * 1e-3) / 1e9, "unit": "GB/s",
            "frac": lk["both_ms"] / call_ms,
            "link_ms": lk["both_ms"], "h2d_alone_gbs": h2d / (lk["h2d_ms"] * 1e-3) / 1e9,
            "d2h_alone_gbs": d2h / (lk["d2h_ms"] * 1e-3) / 1e9,
            "peak_source": "the call's own input and output bytes copied between pinned host "
                           "buffers and device memory, both directions at once on two streams, "
                           "measured in this run (best of 5)"}
    except Exception as e:  # pragma: no cover
        out["roofline"] = {"failed": str(e)}
    return out


def time_steps(fn, steps, warmup):
    import torch
    for i in range(warmup):
        fn(i)
    torch.cuda.synchronize()
    s = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    for i in range(steps):
        fn(i)
    e1.record(s)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


def roofline_for(plan, w, kernel_ms, info, peaks, peaks_src):
    """Roofline record of the main kernel of `plan` on workload `w`."""
    from roofline_gb300 import roofline as rf
    flops = float(w.flops)
    alg_bytes = rf.gemm_bytes(w.M, w.N, w.K, w.beta != 0.0)
    kname = plan["kernel_name"]
    if plan["bound_name"] == "hbm":
        roof = {"bound": "hbm", "achieved": rf.gbps(alg_bytes, kernel_ms),
                "peak": peaks["hbm_gbs"], "unit": "GB/s"}
    elif kname == "tc_tf32x3":
        roof = {"bound": "tensor", "achieved": rf.tflops(flops, kernel_ms),
                "peak": peaks["bf16_tflops"] * TF32_OVER_BF16 / 3.0, "unit": "TFLOP/s"}
    elif kname == "tc_tf32":
        roof = {"bound": "tensor", "achieved": rf.tflops(flops, kernel_ms),
                "peak": peaks["bf16_tflops"] * TF32_OVER_BF16, "unit": "TFLOP/s"}
    else:
        roof = {"bound": "alu", "achieved": rf.tflops(flops, kernel_ms),
                "peak": info["fp32_peak_tflops"], "unit": "TFLOP/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    traffic, tnote = ncu_traffic(plan, w.name)
    roof["traffic"] = traffic
    roof["kernel"] = kname
    roof["instance"] = kernel_instance(plan)
    roof["kernel_ms"] = kernel_ms
    roof["algorithmic"] = (f"{alg_bytes} B" if roof["unit"] == "GB/s" else f"{flops:.0f} FLOP") + \
        " per launch"
    tensor_src = f"{peaks_src} bf16 burst x {TF32_OVER_BF16:.3f} (dense TF32/BF16 nominal ratio)"
    if kname == "tc_tf32x3":
        tensor_src += " / 3 (three TF32 products per FP32 product)"
    roof["peak_source"] = {"alu": "SMs x 128 FP32 lanes x 2 x max SM clock (device attributes)",
                           "tensor": tensor_src,
                           "hbm": f"{peaks_src} copy bandwidth"}[roof["bound"]]
    roof["traffic_note"] = tnote
    return roof


def measure(w, mode, sets, info, peaks, peaks_src, steps=KERNEL_SAMPLES, warmup=3):
    """One config: mean step time over `steps` back-to-back calls (CUDA events
    on the launching stream), then the same calls again with the main kernel
    stamped (same launch order) for its mean duration and roofline."""
    import torch

    from roofline_gb300 import gemm
    plan = gemm.plan(w.M, w.N, w.K, *w.lds(), mode, 0, w.beta != 0.0)
    call = Caller(w, mode, sets)
    step_ms = time_steps(call, steps, warmup)
    stamps = Stamps(steps, torch.device("cuda"))
    stamped_run(call, stamps, 0, steps)
    torch.cuda.synchronize()
    kernel_ms = statistics.mean(stamps.ms())
    r = roofline_for(plan, w, kernel_ms, info, peaks, peaks_src)
    return {"tflops": float(w.flops) / (step_ms * 1e-3) / 1e12, "ms": step_ms,
            "kernel": plan["kernel_name"], "kernel_ms": kernel_ms, "calls": steps,
            "plan": {k: plan[k] for k in ("bm", "bn", "bk", "stages", "split_k", "stream_k",
                                          "grid_ctas", "launches")},
            "roofline": {k: r[k] for k in ("bound", "achieved", "peak", "unit", "frac",
                                           "traffic", "instance", "peak_source")}}


def rotation_of(w, min_sets=2):
    """(input sets, bytes per set, description) of the L2 rotation the timed
    loop uses: enough sets to exceed L2 three times (2 to 64)."""
    lda, ldb, ldc = w.lds()
    set_bytes = 4 * (w.M * lda + w.K * ldb + w.M * ldc)
    nsets = max(min_sets, min(64, -(-3 * L2_BYTES // set_bytes)))
    return nsets, set_bytes, (f"inputs rotated over {nsets} buffer sets "
                              f"({nsets * set_bytes / 2**20:.0f} MiB > L2)")


def device_sets(w, dev, arrays=None, min_sets=2):
    """Device copies of the workload's inputs, enough sets to exceed L2 three times."""
    import torch
    A, B, C0 = arrays if arrays is not None else w.make()
    lda, ldb, ldc = w.lds()
    nsets, set_bytes, _ = rotation_of(w, min_sets)
    hA, hB = torch.from_numpy(A), torch.from_numpy(B)
    hC = torch.from_numpy(C0) if C0 is not None else None
    sets = []
    for _ in range(nsets):
        dA, dB = hA.to(dev), hB.to(dev)
        dC = hC.to(dev) if hC is not None else torch.zeros((w.M, ldc), dtype=torch.float32,
                                                           device=dev)
        sets.append((dA[:, :w.K], dB[:, :w.N], dC[:, :w.N]))
    return sets, set_bytes


def graph_replay(w, reps=50):
    """Per-call time of workload `w` (mode AUTO, caller workspace) issued one
    call at a time and replayed from a CUDA graph holding one call per input
    set; both timed with CUDA events over the same calls."""
    import torch

    from roofline_gb300 import gemm
    sets, _ = device_sets(w, torch.device("cuda"))
    sets = sets[:8]
    p = gemm.plan(w.M, w.N, w.K, *w.lds(), "auto", 0, w.beta != 0.0)
    ws = torch.empty(max(int(p["workspace_bytes"]), 256), dtype=torch.uint8, device="cuda")

    def calls():
        for a, b, c in sets:
            gemm.matmul(a, b, c, w.alpha, w.beta, "auto", workspace=ws)

    calls()
    torch.cuda.synchronize()
    stream = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        calls()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    res = {"calls_per_replay": len(sets), "kernel": p["kernel_name"], "launches": p["launches"]}
    for tag, fn in [("eager_us", calls), ("graph_us", g.replay)]:
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        e0.record()
        for _ in range(reps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        res[tag] = e0.elapsed_time(e1) * 1e3 / (reps * len(sets))
    res["graph_tflops"] = float(w.flops) / (res["graph_us"] * 1e-6) / 1e12
    return res


# Every workload of the measured configuration list, with the modes timed for
# each (the headline workload's AUTO line is the main result).
EXTRA_CONFIGS = [("sq4096", ["fp32_simt", "tf32x3", "tf32"]),
                 ("sq8192", ["auto", "fp32_simt"]),
                 ("skinny", ["auto"]),
                 ("ragged", ["auto", "fp32_simt"]),
                 ("sq512", ["auto", "tf32x3"]),
                 ("sq512_int", ["auto"])]


def extras(args, w, sets, info, peaks, peaks_src):
    """Every config with its roofline (mean of KERNEL_SAMPLES calls each), the
    FMA and HBM copy roofs, and cuBLAS reference points (timed beside the
    library, never inside it)."""
    import torch

    from roofline_gb300 import gemm
    from workloads import WORKLOADS
    out = {"configs": {}}
    n = len(sets)
    for name, modes in EXTRA_CONFIGS:
        wl = WORKLOADS[name]
        try:
            wsets = sets if name == w.name else device_sets(wl, torch.device("cuda"))[0]
            res = {}
            for mode in modes:
                try:
                    res[mode] = measure(wl, mode, wsets, info, peaks, peaks_src)
                except gemm.GemmError as e:
                    res[mode] = {"unavailable": str(e)}
            out["configs"][name] = res
            if name != w.name:
                del wsets
                torch.cuda.empty_cache()
        except Exception as e:  # pragma: no cover
            out["configs"][name] = {"failed": str(e)}
    # launch overhead: 512^3 calls one by one against the same calls replayed
    # from a CUDA graph (one capture of one call per input set)
    try:
        out["sq512_graph"] = graph_replay(WORKLOADS["sq512"])
    except Exception as e:  # pragma: no cover
        out["sq512_graph"] = {"failed": str(e)}
    # FP32 FMA roof, measured ("Bandwidths and peak rate - exercises", exercise 5)
    try:
        out["fp32_fma_peak_tflops"] = {"scalar": gemm.fp32_fma_peak(1 << 16, False),
                                       "packed": gemm.fp32_fma_peak(1 << 16, True),
                                       "derived": info["fp32_peak_tflops"]}
    except Exception as e:  # pragma: no cover
        out["fp32_fma_peak_tflops"] = f"failed: {e}"
    # HBM copy calibration: 2 x 256M floats (1 GiB each), 50 timed copies
    try:
        src = torch.ones(256 << 20, dtype=torch.float32, device="cuda")
        dst = torch.empty_like(src)
        out["hbm_copy_gbs"] = gemm.hbm_copy_calibrate(src, dst, iters=50)
        del src, dst
    except Exception as e:  # pragma: no cover
        out["hbm_copy_gbs"] = f"failed: {e}"
    # cuBLAS through torch, FP32 (no TF32) and TF32, same inputs
    old = torch.backends.cuda.matmul.allow_tf32
    try:
        for tag, tf32 in [("torch_fp32", False), ("torch_tf32", True)]:
            torch.backends.cuda.matmul.allow_tf32 = tf32
            ms = time_steps(lambda i: torch.matmul(sets[i % n][0], sets[i % n][1]), 20, 3)
            out[tag + "_tflops"] = float(w.flops) / (ms * 1e-3) / 1e12
        torch.backends.cuda.matmul.allow_tf32 = True
        x = torch.randn(8192, 8192, device="cuda")
        y = torch.randn(8192, 8192, device="cuda")
        best = min(time_steps(lambda i: torch.matmul(x, y), 1, 1) for _ in range(10))
        out["tf32_dense_tflops_measured"] = 2 * 8192 ** 3 / (best * 1e-3) / 1e12
        del x, y
    finally:
        torch.backends.cuda.matmul.allow_tf32 = old
    return out


def run_calibration(args):
    """The C1 copy calibration alone: out[i] = in[i] over 256M floats, one
    untimed copy, then `args.steps` (at least 50) timed copies between CUDA
    events; GB/s = 2 * n * 4 * iterations / time."""
    import torch

    from roofline_gb300 import gemm
    rank, _, local = dist_env()
    torch.cuda.set_device(local)
    n = 256 << 20
    src = torch.ones(n, dtype=torch.float32, device="cuda")
    dst = torch.empty_like(src)
    iters = max(50, args.steps)
    gbs = gemm.hbm_copy_calibrate(src, dst, iters=iters)
    ok = bool(torch.equal(src, dst))
    if rank == 0:
        print(json.dumps({"metric": "HBM copy bandwidth (2 x n x 4 bytes / t)", "value": gbs,
                          "unit": "GB/s", "n_floats": n, "iterations": iters,
                          "copy_exact": ok}), flush=True)
    return 0 if ok else 1


def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args)
    if args.calibrate_only:
        return run_calibration(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
