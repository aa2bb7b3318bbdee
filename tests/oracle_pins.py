"""Checks that pin the CPU oracle to facts outside itself.

Each check returns a list of failure strings (empty = pass) so the same
suite can run against the real oracle and against deliberately broken
copies of its source (see test_oracle.py::test_pins_catch_planted_mistakes).

Sources of truth used here, none of them the oracle's own code:
  * closed forms: A*I = A, I*B = B, all-ones gives K, alpha/beta on
    constants;
  * numpy float32 elementwise products (rank-1, K = 1: one rounding);
  * exact integer arithmetic in Python ints;
  * exact rational arithmetic (fractions.Fraction) rounded once;
  * numpy/BLAS float64 matmul at 512^3 (a different summation order, so
    agreement within one float32 ulp).
"""
from __future__ import annotations

import numpy as np

from oracle import exact
from workloads import matrix


def _padded(arr: np.ndarray, extra: int, fill=np.nan) -> np.ndarray:
    """Copy of a 2-D float32 array with `extra` NaN padding columns; returns a
    view of the logical part whose row stride is the padded width."""
    r, c = arr.shape
    buf = np.full((r, c + extra), fill, dtype=np.float32)
    buf[:, :c] = arr
    return buf[:, :c]


def check_identity(orc):
    fails = []
    A = matrix(7, 5, None, 11, "u11")
    I5 = np.eye(5, dtype=np.float32)
    I7 = np.eye(7, dtype=np.float32)
    if not np.array_equal(orc.gemm(A, I5), A):
        fails.append("A @ I != A")
    if not np.array_equal(orc.gemm(I7, A), A):
        fails.append("I @ A != A")
    return fails


def check_all_ones(orc):
    fails = []
    A = np.ones((6, 9), dtype=np.float32)
    B = np.ones((9, 4), dtype=np.float32)
    if not np.all(orc.gemm(A, B) == 9.0):
        fails.append("ones(6,9) @ ones(9,4) != 9")
    C0 = np.full((6, 4), 2.0, dtype=np.float32)
    got = orc.gemm(A, B, alpha=1.5, beta=0.5, C0=C0)
    if not np.all(got == 1.5 * 9 + 0.5 * 2.0):
        fails.append("alpha*K + beta*C0 on constants")
    got = orc.gemm(A, B, alpha=-2.0, beta=-0.25, C0=C0)
    if not np.all(got == -2.0 * 9 - 0.25 * 2.0):
        fails.append("negative alpha/beta on constants")
    return fails


def check_rank1(orc):
    fails = []
    a = matrix(13, 1, None, 21, "u11")
    b = matrix(1, 17, None, 22, "u11")
    want = np.outer(a[:, 0], b[0, :]).astype(np.float32)  # float32 products, one rounding
    if not np.array_equal(orc.gemm(a, b), want):
        fails.append("K=1 outer product != float32 products")
    return fails


def check_integer_bruteforce(orc):
    fails = []
    shapes = [(1, 1, 1), (2, 3, 4), (5, 7, 3), (8, 1, 8), (3, 8, 1), (7, 6, 5)]
    for t, (M, N, K) in enumerate(shapes):
        A = matrix(M, K, None, 100 + t, "int2")
        B = matrix(K, N, None, 200 + t, "int2")
        Ai = [[int(v) for v in row] for row in A]
        Bi = [[int(v) for v in row] for row in B]
        want = np.array([[sum(Ai[i][k] * Bi[k][j] for k in range(K)) for j in range(N)]
                         for i in range(M)], dtype=np.float32)
        # leading dimensions larger than the width, NaN in the padding
        got = orc.gemm(_padded(A, 3), _padded(B, 2))
        if got.shape != (M, N) or not np.array_equal(got, want):
            fails.append(f"integer brute force {M}x{N}x{K}")
    return fails


def check_rational_bruteforce(orc):
    fails = []
    cases = [(4, 5, 3, 1.0, 0.0), (3, 6, 7, 1.5, 0.5), (6, 2, 8, -0.75, 2.0),
             (1, 9, 5, 3.0, -1.0)]
    for t, (M, N, K, alpha, beta) in enumerate(cases):
        A = matrix(M, K, None, 300 + t, "u11")
        B = matrix(K, N, None, 400 + t, "normal", 0.3)
        C0 = matrix(M, N, None, 500 + t, "u11")
        want, _, bound = exact.gemm_exact(A, B, alpha, beta, C0)
        got, D = orc.gemm(_padded(A, 1), _padded(B, 5), alpha=alpha, beta=beta,
                          C0=_padded(C0, 2), with_bound=True)
        if not np.array_equal(got, want):
            fails.append(f"rational brute force {M}x{N}x{K} a={alpha} b={beta}")
        bd = np.array([[float(x) for x in row] for row in bound])
        if not np.allclose(D, bd, rtol=1e-13, atol=0.0):
            fails.append(f"error bound D {M}x{N}x{K}")
    return fails


def check_beta_zero_ignores_c(orc):
    A = matrix(4, 3, None, 600, "u11")
    B = matrix(3, 5, None, 601, "u11")
    C0 = np.full((4, 5), np.nan, dtype=np.float32)
    got = orc.gemm(A, B, alpha=1.0, beta=0.0, C0=C0)
    return [] if np.all(np.isfinite(got)) else ["beta=0 read C_old (NaN propagated)"]


def check_alpha_zero_ignores_ab(orc):
    """BLAS reading of alpha == 0 (as of beta == 0): A and B are not read, so
    C = float_rn(beta * C_old) exactly (a product of two floats rounds once),
    and beta == 0 gives zeros, even with NaN in A and B."""
    A = np.full((4, 3), np.nan, dtype=np.float32)
    B = np.full((3, 5), np.inf, dtype=np.float32)
    C0 = matrix(4, 5, None, 602, "u11")
    fails = []
    got = orc.gemm(A, B, alpha=0.0, beta=-1.5, C0=C0)
    if not np.array_equal(got, np.float32(-1.5) * C0):
        fails.append("alpha=0 read A or B, or did not give beta*C_old")
    if not np.array_equal(orc.gemm(A, B, alpha=0.0, beta=0.0, C0=C0), np.zeros((4, 5), np.float32)):
        fails.append("alpha=0, beta=0 did not give zeros")
    return fails


def check_numpy_f64_512(orc):
    A = matrix(512, 512, None, 700, "u11")
    B = matrix(512, 512, None, 701, "u11")
    got = orc.gemm(A, B)
    ref = (A.astype(np.float64) @ B.astype(np.float64)).astype(np.float32)
    ulp = np.abs(got.view(np.int32).astype(np.int64) - ref.view(np.int32).astype(np.int64))
    fails = []
    if ulp.max() > 1:
        fails.append(f"oracle vs numpy float64 at 512^3: {ulp.max()} ulp")
    if np.count_nonzero(ulp) > 0.01 * ulp.size:
        fails.append("oracle vs numpy float64: too many 1-ulp differences")
    return fails


def check_entries_match_full(orc):
    A = matrix(37, 29, None, 800, "u11")
    B = matrix(29, 41, None, 801, "u11")
    C0 = matrix(37, 41, None, 802, "u11")
    full, D = orc.gemm(A, B, 1.5, 0.5, C0, with_bound=True)
    rows = np.array([0, 36, 5, 17, 36, 0], dtype=np.int64)
    cols = np.array([0, 40, 7, 3, 0, 40], dtype=np.int64)
    v, d = orc.gemm_entries(A, B, rows, cols, 1.5, 0.5, C0)
    fails = []
    if not np.array_equal(v, full[rows, cols]):
        fails.append("sampled entries != full matrix")
    if not np.array_equal(d, D[rows, cols]):
        fails.append("sampled bounds != full bounds")
    return fails


ALL = [check_identity, check_all_ones, check_rank1, check_integer_bruteforce,
       check_rational_bruteforce, check_beta_zero_ignores_c, check_alpha_zero_ignores_ab,
       check_numpy_f64_512,
       check_entries_match_full]


def run_all(orc):
    fails = []
    for chk in ALL:
        try:
            fails += chk(orc)
        except Exception as e:  # a crash in a broken oracle is a caught mistake
            fails.append(f"{chk.__name__}: {type(e).__name__}: {e}")
    return fails
