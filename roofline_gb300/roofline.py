"""Roofline arithmetic used to report GEMM and copy results.

Definitions follow the course pages:
  * work of C = A*B: 2 FLOP (one multiply, one add) per k per output, so
    2*M*N*K ("Project - tiled matrix multiply", section "Numerical
    background - the metrics we report");
  * throughput = FLOP / seconds; percent of peak = 100 * achieved / peak
    (same section, and the "report" helper of section "Starter
    scaffolding");
  * FP32 non-tensor peak = SMs x FP32 lanes per SM x 2 (an FMA is two
    FLOP) x clock ("Bandwidths and peak rate - exercises", exercise 1);
  * copy bandwidth = 2 * n * sizeof(float) / seconds (each element read once
    and written once; same page, exercise 2);
  * ridge point = arithmetic peak / memory bandwidth, in FLOP per byte
    (same page, exercise 3).
"""
from __future__ import annotations


def gemm_flops(M: int, N: int, K: int) -> int:
    return 2 * M * N * K


def gemm_bytes(M: int, N: int, K: int, beta_nonzero: bool = False, elem: int = 4) -> int:
    """Algorithmic HBM bytes: read A and B once, write C once, read C if beta != 0."""
    return elem * (M * K + K * N + M * N * (2 if beta_nonzero else 1))


def gflops(flops: float, ms: float) -> float:
    return flops / (ms / 1000.0) / 1e9


def tflops(flops: float, ms: float) -> float:
    return flops / (ms / 1000.0) / 1e12


def pct_of_peak(achieved: float, peak: float) -> float:
    return 100.0 * achieved / peak


def fp32_peak_flops(sm_count: int, clock_hz: float, lanes_per_sm: int = 128) -> float:
    return sm_count * lanes_per_sm * 2.0 * clock_hz


def copy_bytes(n_elems: int, elem: int = 4) -> int:
    return 2 * n_elems * elem


def gbps(nbytes: float, ms: float) -> float:
    return nbytes / (ms / 1000.0) / 1e9


def ridge_point(peak_flops: float, bandwidth_bytes_per_s: float) -> float:
    return peak_flops / bandwidth_bytes_per_s


def intensity(flops: float, nbytes: float) -> float:
    return flops / nbytes
