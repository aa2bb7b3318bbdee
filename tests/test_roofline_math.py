"""Pins the roofline arithmetic to the numbers the course pages print (CPU)."""
import json
import os

import pytest

from roofline_gb300 import roofline as rf

with open(os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                       "page_facts.json")) as _f:
    FACTS = json.load(_f)


def test_fp32_peak_formula():
    f = FACTS["h100_fp32_peak"]
    peak = rf.fp32_peak_flops(f["sm"], f["clock_hz"], f["lanes"])
    assert round(peak / 1e9, -2) == f["peak_gflops_rounded"]
    # forgetting that an FMA is two FLOP halves the figure
    assert round(peak / 2 / 1e9, -1) == f["forgot_fma_factor_gflops_rounded"]


def test_results_table_consistency():
    t = FACTS["results_table_4096"]
    flops = rf.gemm_flops(4096, 4096, 4096)
    naive_ms = t["rows"][0]["ms"]
    for row in t["rows"]:
        g = rf.gflops(flops, row["ms"])
        assert abs(g - row["gflops"]) <= 1.0, row
        assert round(rf.pct_of_peak(row["gflops"], t["peak_gflops"]), 1) == row["pct"]
        assert round(naive_ms / row["ms"], 1) == row["speedup"]


def test_tile_reuse_counts():
    f = FACTS["tile_reuse"]
    T = f["tile"]
    assert 2 * T * T == f["loads"] and T ** 3 == f["fmas"]
    assert f["fmas"] // f["loads"] == f["fma_per_load"]
    assert 2 * f["fmas"] // f["loads"] == f["flop_per_load_rounded"]


def test_copy_bytes_and_band():
    f = FACTS["copy_kernel"]
    assert f["n"] * 4 == f["bytes_per_array"]
    assert rf.copy_bytes(f["n"]) == f["bytes_moved"]
    # a copy taking exactly bytes / (0.9 * 3350 GB/s) sits inside the 85-92 % band
    ms = f["bytes_moved"] / (0.9 * f["hbm_gbs"] * 1e9) * 1e3
    pct = rf.pct_of_peak(rf.gbps(f["bytes_moved"], ms), f["hbm_gbs"])
    assert f["expected_pct_low"] <= pct <= f["expected_pct_high"]


def test_ridge_points():
    f = FACTS["ridge_points"]
    assert round(rf.ridge_point(f["bf16_tflops"] * 1e12, f["hbm_tbs"] * 1e12)) == \
        f["bf16_ridge_rounded"]
    assert round(rf.ridge_point(f["fp8_tflops"] * 1e12, f["hbm_tbs"] * 1e12)) == \
        f["fp8_ridge_rounded"]
    assert rf.intensity(f["scale_flop"], f["scale_bytes"]) == f["scale_ai"]


def test_gemm_bytes():
    assert rf.gemm_bytes(512, 512, 512) == 3 * 512 * 512 * 4
    # ragged shape with beta != 0 reads C as well
    assert rf.gemm_bytes(1023, 1025, 777, True) == 4 * (1023 * 777 + 777 * 1025 + 2 * 1023 * 1025)
    assert rf.gemm_bytes(65536, 64, 4096) == 1_091_567_616


def test_traffic_entries_match_current_sources():
    # every committed ncu traffic figure belongs to the kernel source as it
    # is now (comments aside); a stale entry would make bench.py report null
    import json
    import os
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import bench
    import re
    with open(os.path.join(root, "profiles", "traffic.json")) as f:
        entries = json.load(f)
    # keyed by the exact instantiation and launch shape the bench reports
    # (bench.kernel_instance), so counters of one configuration are never
    # attached to another
    pat = re.compile(r"^(tc_tf32x3_kernel<\d+(,\d+){7}>|simt_packed_kernel<\d+(,\d+){6}>) "
                     r"grid=\d+ split_k=\d+ stream_k=[01] @ \w+$")
    for key, e in entries.items():
        assert pat.match(key), key
        kind = "tc" if key.startswith("tc_") else "simt"
        assert sorted(e["sources"]) == sorted(bench.TRAFFIC_SOURCES[kind]), key
        assert e["source_hash"] == bench.source_hash(e["sources"]), key
        assert e["dram_bytes_per_launch"] > 0


def test_kernel_instance_names_the_configuration():
    import os
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    plan = {"kernel_name": "tc_tf32x3", "bm": 128, "bn": 256, "bk": 16, "stages": 5,
            "a_split_in_kernel": 1, "a_hi_tmem": 1, "b_concat": 0, "grid_ctas": 152,
            "split_k": 1, "stream_k": 1, "vec": 1}
    assert bench.kernel_instance(plan) == \
        "tc_tf32x3_kernel<128,256,16,5,2,0,3,0> grid=152 split_k=1 stream_k=1"
    plan.update(kernel_name="tc_tf32", a_hi_tmem=0)
    assert bench.kernel_instance(plan).startswith("tc_tf32x3_kernel<128,256,16,5,1,0,1,0>")
    plan.update(kernel_name="tc_tf32x3", b_split_in_kernel=1, stream_k=0)
    assert bench.kernel_instance(plan).startswith("tc_tf32x3_kernel<128,256,16,5,1,0,3,2>")
    assert bench.kernel_instance(plan, b_stored_nk=True).startswith(
        "tc_tf32x3_kernel<128,256,16,5,1,0,3,1>")
    plan.update(kernel_name="simt", bm=64, bn=128, bk=16, stages=4, grid_ctas=2048, stream_k=0)
    assert bench.kernel_instance(plan) == \
        "simt_packed_kernel<64,128,16,4,1,0,0> grid=2048 split_k=1 stream_k=0"


def test_source_hash_ignores_comments_only():
    import os
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    a = "int f() {  // one\n  return 1; /* two\n three */\n}\n"
    b = "int f() {\n\n  return 1;   // changed comment\n}\n"
    c = "int f() {\n  return 2;\n}\n"
    assert bench.code_only(a) == bench.code_only(b)
    assert bench.code_only(a) != bench.code_only(c)
