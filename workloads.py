"""Seeded synthetic inputs for the FP32 GEMM workloads.

This module only draws numbers and describes shapes; it holds none of the
GEMM arithmetic.  Both the CUDA path's tests/bench and the CPU oracle take
their inputs from here, so the two sides always see identical bits.

Generator: SplitMix64 (Steele, Lea, Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014) evaluated counter-style, x_i = mix(seed_key
+ (i+1) * golden_gamma), in numpy uint64 arithmetic (wraps mod 2^64).  It is
platform independent, so the x86 build host and the Arm GPU host produce the
same matrices.

Value distributions follow the workloads of the tiled-matmul course page
("Project - tiled matrix multiply", section "What we build": square FP32
N x N, N = 4096 by default) extended to the five shapes the library is
measured on:

* ``u11``  : uniform on [-1, 1): 2*u - 1 with u a 24-bit dyadic in [0, 1),
             exact in FP32.
* ``int2`` : integers uniform in {-2, ..., 2} (exact in FP32 and TF32).
* ``normal``: N(0, sigma^2) by Box-Muller on two 53-bit uniforms, rounded
             once to FP32.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def splitmix64(seed: int, start: int, count: int, stream: int = 0) -> np.ndarray:
    """Counter-based SplitMix64 outputs for indices [start, start+count)."""
    key = np.uint64((seed * 0x100000001B3 + stream * 0x9E3779B1) & 0xFFFFFFFFFFFFFFFF)
    idx = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix(key + idx * _GAMMA)


def _fill(out_flat: np.ndarray, seed: int, dist: str, sigma: float) -> None:
    n = out_flat.size
    for s in range(0, n, _CHUNK):
        c = min(_CHUNK, n - s)
        if dist == "u11":
            u = (splitmix64(seed, s, c) >> np.uint64(40)).astype(np.float64) * 2.0 ** -24
            out_flat[s:s + c] = (2.0 * u - 1.0).astype(np.float32)
        elif dist == "int2":
            r = (splitmix64(seed, s, c) >> np.uint64(32)) % np.uint64(5)
            out_flat[s:s + c] = r.astype(np.float32) - 2.0
        elif dist == "normal":
            u1 = ((splitmix64(seed, s, c, 1) >> np.uint64(11)).astype(np.float64) + 1.0) * 2.0 ** -53
            u2 = (splitmix64(seed, s, c, 2) >> np.uint64(11)).astype(np.float64) * 2.0 ** -53
            z = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * math.pi * u2)
            out_flat[s:s + c] = (sigma * z).astype(np.float32)
        else:
            raise ValueError(f"unknown distribution {dist!r}")


def matrix(rows: int, cols: int, ld: Optional[int], seed: int, dist: str,
           sigma: float = 1.0, pad_value: float = float("nan")) -> np.ndarray:
    """A rows x cols float32 matrix stored row-major with leading dimension ld.

    Returns the full (rows, ld) backing array; the logical matrix is
    ``arr[:, :cols]``.  Padding columns hold ``pad_value`` (NaN by default) so
    a kernel that reads past the logical width poisons its result.
    """
    ld = cols if ld is None else ld
    assert ld >= cols
    arr = np.empty((rows, ld), dtype=np.float32)
    if ld > cols:
        arr[:, cols:] = pad_value
    logical = np.empty(rows * cols, dtype=np.float32)
    _fill(logical, seed, dist, sigma)
    arr[:, :cols] = logical.reshape(rows, cols)
    return arr


@dataclasses.dataclass(frozen=True)
class Workload:
    """One GEMM problem C <- alpha * A B + beta * C, all row-major FP32."""
    name: str
    M: int
    N: int
    K: int
    alpha: float = 1.0
    beta: float = 0.0
    a_dist: str = "u11"
    b_dist: str = "u11"
    c_dist: str = "u11"
    a_sigma: float = 1.0
    b_sigma: float = 1.0
    seed: int = 1000
    lda: Optional[int] = None
    ldb: Optional[int] = None
    ldc: Optional[int] = None
    sampled: bool = False  # large shapes: the oracle checks sampled entries
    description: str = ""

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K

    def lds(self):
        return (self.lda or self.K, self.ldb or self.N, self.ldc or self.N)

    def make(self):
        """(A, B, C0) as (rows, ld) float32 arrays; C0 is None when beta == 0."""
        lda, ldb, ldc = self.lds()
        A = matrix(self.M, self.K, lda, self.seed, self.a_dist, self.a_sigma)
        B = matrix(self.K, self.N, ldb, self.seed + 50, self.b_dist, self.b_sigma)
        C0 = None
        if self.beta != 0.0:
            C0 = matrix(self.M, self.N, ldc, self.seed + 100, self.c_dist)
        return A, B, C0


WORKLOADS = {
    "sq512": Workload("sq512", 512, 512, 512, seed=1001,
                      description="square 512^3, U[-1,1], alpha=1 beta=0"),
    "sq512_int": Workload("sq512_int", 512, 512, 512, seed=1101, a_dist="int2", b_dist="int2",
                          description="square 512^3, integers in {-2..2} (bit-exact check)"),
    "ragged": Workload("ragged", 1023, 1025, 777, alpha=1.5, beta=0.5, seed=1002,
                       description="ragged M=1023 K=777 N=1025, alpha=1.5 beta=0.5, "
                                   "lda=777 ldb=1025 ldc=1025 (unaligned)"),
    "sq4096": Workload("sq4096", 4096, 4096, 4096, seed=1003, sampled=True,
                       description="square 4096^3, U[-1,1] (137.4 GFLOP)"),
    "sq8192": Workload("sq8192", 8192, 8192, 8192, seed=1004, a_dist="normal", b_dist="normal",
                       a_sigma=1.0, b_sigma=0.02, sampled=True,
                       description="square 8192^3, A~N(0,1), B~N(0,0.02^2)"),
    "skinny": Workload("skinny", 65536, 64, 4096, seed=1005, sampled=True,
                       description="skinny M=65536 K=4096 N=64, U[-1,1] (memory-bound)"),
}


def sample_entries(M: int, N: int, n: int = 4096, seed: int = 1200):
    """n (row, col) output positions: the four corners, the last row and last
    column of the edge tiles, then seeded uniform positions."""
    fixed = [(0, 0), (0, N - 1), (M - 1, 0), (M - 1, N - 1)]
    for t in range(1, 9):
        fixed.append((M - 1, max(0, N - 1 - 37 * t)))
        fixed.append((max(0, M - 1 - 41 * t), N - 1))
    fixed = fixed[:n]
    rest = n - len(fixed)
    r = splitmix64(seed, 0, rest, 3) % np.uint64(M)
    c = splitmix64(seed, 0, rest, 4) % np.uint64(N)
    rows = np.concatenate([np.array([p[0] for p in fixed], dtype=np.int64), r.astype(np.int64)])
    cols = np.concatenate([np.array([p[1] for p in fixed], dtype=np.int64), c.astype(np.int64)])
    return rows, cols
