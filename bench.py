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


def ncu_traffic(kernel_key: str):
    """DRAM bytes per launch from the committed ncu summary, or None when the
    kernel's source changed after the counters were taken."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        e = d[kernel_key]
        if e.get("source_hash") != source_hash(e["sources"]):
            return None, "stale"
        return float(e["dram_bytes_per_launch"]), e.get("note", "")
    except Exception:
        return None, "absent"



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

def workload_config(w, mode, rotation):
    cfg = {"workload": f"{w.name}: {w.description}", "M": w.M, "N": w.N, "K": w.K,
           "alpha": w.alpha, "beta": w.beta, "layout": "row-major", "mode": mode}
    if rotation is not None:
        cfg["l2"] = rotation
    return cfg


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
    nsets = len(sets)
    rotation = rotation_of(w)[2]

    plan = gemm.plan(w.M, w.N, w.K, lda, ldb, ldc, args.mode, 0, w.beta != 0.0)
    stream = torch.cuda.current_stream()

    def step(i):
        a, b, c = sets[i % nsets]
        gemm.matmul(a, b, c, w.alpha, w.beta, args.mode)

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

    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    start.record(stream)
    for i in range(args.steps):
        step(i)
    end.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    ms_total = start.elapsed_time(end)
    if gemm.check_status() != gemm.OK:
        raise RuntimeError("device status reported a timeout during the timed region")

    # Separate pass for the roofline: the library records events around its
    # main kernel (plain stream order for these calls), one pair per step.
    nk = max(3, min(args.steps, 50))
    ev_b = [torch.cuda.Event(enable_timing=True) for _ in range(nk)]
    ev_a = [torch.cuda.Event(enable_timing=True) for _ in range(nk)]
    for e in ev_b + ev_a:  # torch creates the underlying cudaEvent on first record
        e.record(stream)
    torch.cuda.synchronize()
    for i in range(nk):
        gemm.set_profile_events(ev_b[i], ev_a[i])
        step(i)
    gemm.set_profile_events(None, None)
    torch.cuda.synchronize()
    main_ms = [ev_b[i].elapsed_time(ev_a[i]) for i in range(nk)]

    t_max = max_over_ranks(ms_total, world, dev)
    flops = float(w.flops)
    value = whole_job_tflops(flops, args.steps, world, t_max)
    ms_step = t_max / args.steps

    # roofline of the dominant (main GEMM) kernel
    main_avg = statistics.mean(main_ms)
    roof = roofline_for(plan, w, main_avg, info, peaks, peaks_src)
    roof["kernel_timing"] = f"mean of {nk} launches, CUDA events recorded around the kernel on its stream"
    roof["kernel_ms_best"] = min(main_ms)
    roof["achieved_best"] = roof["achieved"] * main_avg / min(main_ms)

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
        line["e2e"] = e2e(args, w, A, B, C0, sets[0], dev, world)

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


def e2e(args, w, A, B, C0, dset, dev, world):
    """The metric measured through the host-buffer C-ABI call gemm_f32_host:
    A, B (and C when beta != 0) in pinned host memory, copied in, multiplied
    and copied back inside the call (row blocks pipelined over copy and
    compute streams).  Timed on the host around whole blocking calls."""
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
    return {"value": whole_job_tflops(float(w.flops), steps, world, ms), "unit": "TFLOP/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": 4 * w.M * w.N, "steps": steps,
            "ms_per_step": ms / steps,
            "path": "pinned host -> gemm_f32_host (row blocks: H2D copy stream, GEMM stream, "
                    "D2H copy stream) -> pinned host; host wall clock around blocking calls"}


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
    traffic, tnote = ncu_traffic(f"{kname}:{w.name}")
    roof["traffic"] = traffic
    roof["kernel"] = kname
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


def measure(w, mode, sets, steps, warmup=3):
    """(mean step ms, mean main-kernel ms, plan) for `steps` library calls."""
    import torch

    from roofline_gb300 import gemm
    n = len(sets)
    plan = gemm.plan(w.M, w.N, w.K, *w.lds(), mode, 0, w.beta != 0.0)

    def fn(i):
        a, b, c = sets[i % n]
        gemm.matmul(a, b, c, w.alpha, w.beta, mode)
    step_ms = time_steps(fn, steps, warmup)
    s = torch.cuda.current_stream()
    eb = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ea = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for e in eb + ea:
        e.record(s)
    torch.cuda.synchronize()
    for i in range(steps):
        gemm.set_profile_events(eb[i], ea[i])
        fn(i)
    gemm.set_profile_events(None, None)
    torch.cuda.synchronize()
    kernel_ms = statistics.mean(eb[i].elapsed_time(ea[i]) for i in range(steps))
    return step_ms, kernel_ms, plan


def rotation_of(w, min_sets=2):
    """(input sets, bytes per set, description) of the L2 rotation the timed
    loop uses: enough sets to exceed L2 three times (2 to 8)."""
    lda, ldb, ldc = w.lds()
    set_bytes = 4 * (w.M * lda + w.K * ldb + w.M * ldc)
    nsets = max(min_sets, min(8, -(-3 * L2_BYTES // set_bytes)))
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


def extras(args, w, sets, info, peaks, peaks_src):
    """Both modes on the same workload, the other large workloads, the FMA and
    HBM copy roofs, and cuBLAS reference points (timed beside the library,
    never inside it)."""
    import torch

    from roofline_gb300 import gemm
    from workloads import WORKLOADS
    out = {}
    n = len(sets)
    for mode in ["fp32_simt", "tf32x3"]:
        try:
            step_ms, kernel_ms, p = measure(w, mode, sets, 20)
        except gemm.GemmError as e:
            out[mode] = {"unavailable": str(e)}
            continue
        out[mode] = {"tflops": float(w.flops) / (step_ms * 1e-3) / 1e12, "ms": step_ms,
                     "kernel": p["kernel_name"], "kernel_ms": kernel_ms,
                     "roofline_frac": roofline_for(p, w, kernel_ms, info, peaks, peaks_src)["frac"]}
    # the other large workloads: a short timing per mode
    for name, modes in [("sq8192", ["auto", "fp32_simt"]), ("skinny", ["auto"])]:
        if name == w.name:
            continue
        wl = WORKLOADS[name]
        try:
            wsets, _ = device_sets(wl, torch.device("cuda"))
            res = {}
            for mode in modes:
                steps = 5 if (name == "sq8192" and mode == "fp32_simt") else 20
                step_ms, kernel_ms, p = measure(wl, mode, wsets, steps)
                r = roofline_for(p, wl, kernel_ms, info, peaks, peaks_src)
                res[mode] = {"tflops": float(wl.flops) / (step_ms * 1e-3) / 1e12, "ms": step_ms,
                             "kernel": p["kernel_name"], "kernel_ms": kernel_ms,
                             "roofline": {k: r[k] for k in ("bound", "achieved", "peak", "unit",
                                                            "frac")}}
            out[name] = res
            del wsets
            torch.cuda.empty_cache()
        except Exception as e:  # pragma: no cover
            out[name] = {"failed": str(e)}
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
