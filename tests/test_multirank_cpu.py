"""Multi-process paths of bench.py on the CPU (gloo, world size 2).

The GEMM runs as independent replicas, one per GPU, with no collective on
the data path; what spans ranks is host logic: the slowest rank's time sets
the whole-job figure, and in the reference arm rank 0 alone works and
prints.  Both are exercised here with real processes and 127.0.0.1
rendezvous."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        ms = bench.max_over_ranks(10.0 + 5.0 * rank, world, "cpu")
        value = bench.whole_job_tflops(2.0e12, 4, world, ms)
        with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
            json.dump({"ms": ms, "value": value}, f)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_value(tmp_path):
    import torch.multiprocessing as mp
    world, port = 2, _free_port()
    mp.spawn(_rank_main, args=(world, port, str(tmp_path)), nprocs=world, join=True)
    got = [json.load(open(tmp_path / f"r{r}.json")) for r in range(world)]
    for g in got:
        assert g["ms"] == 15.0  # the slowest rank's time, on every rank
        # 2 ranks x 4 steps x 2 TFLOP in 15 ms
        assert g["value"] == pytest.approx(2 * 4 * 2.0e12 / 15e-3 / 1e12)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1, "cpu") == 3.5
    assert bench.whole_job_tflops(1e12, 10, 1, 1000.0) == pytest.approx(10.0)  # 1e13 FLOP in 1 s


def test_reference_arm_under_torchrun_prints_once():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py",
           "--impl", "reference", "--workload", "sq512", "--gpus", "2", "--steps", "1",
           "--warmup", "0"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle"


def test_reference_arm_config_matches_ours():
    # both arms name the same workload configuration
    sys.path.insert(0, ROOT)
    import bench
    from workloads import WORKLOADS
    w = WORKLOADS["sq4096"]
    cfg = bench.workload_config(w, "auto", bench.rotation_of(w)[2])
    assert cfg["M"] == cfg["N"] == cfg["K"] == 4096
    assert cfg["l2"] == "inputs rotated over 3 buffer sets (576 MiB > L2)"
