"""Exact rational GEMM on tiny inputs -- TEST INFRASTRUCTURE ONLY.

An independent second statement of what the oracle computes, used to pin
it: every product and sum is carried exactly as a ``fractions.Fraction``,
then the result is rounded once to the nearest float32 (ties to even).
Pure Python, so only for shapes of a few hundred entries.
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np


def round_to_f32(x: Fraction) -> np.float32:
    """Correctly rounded (nearest, ties to even) float32 value of x."""
    if x == 0:
        return np.float32(0.0)
    sign = -1 if x < 0 else 1
    a = abs(x)
    # exponent e with 2^23 <= a / 2^e < 2^24 (normal range), clamped for subnormals
    e = a.numerator.bit_length() - a.denominator.bit_length() - 24
    while a / Fraction(2) ** e >= 2 ** 24:
        e += 1
    while a / Fraction(2) ** e < 2 ** 23:
        e -= 1
    e = max(e, -149)
    q = a / Fraction(2) ** e
    m = q.numerator // q.denominator
    rem = q - m
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and m % 2 == 1):
        m += 1
    val = float(m) * 2.0 ** e  # exact: m <= 2^24, power of two scaling
    return np.float32(sign * val)


def gemm_exact(A, B, alpha=1.0, beta=0.0, C0=None, M=None, N=None, K=None):
    """Returns (C_rounded float32 MxN, exact Fraction matrix, bound Fractions)."""
    A = np.asarray(A, dtype=np.float32)
    B = np.asarray(B, dtype=np.float32)
    M = A.shape[0] if M is None else M
    K = A.shape[1] if K is None else K
    N = B.shape[1] if N is None else N
    fa = Fraction(float(np.float32(alpha)))
    fb = Fraction(float(np.float32(beta)))
    out = np.empty((M, N), dtype=np.float32)
    exact = [[None] * N for _ in range(M)]
    bound = [[None] * N for _ in range(M)]
    for i in range(M):
        for j in range(N):
            s = Fraction(0)
            sa = Fraction(0)
            for k in range(K if alpha != 0.0 else 0):  # alpha == 0: A, B not read
                p = Fraction(float(A[i, k])) * Fraction(float(B[k, j]))
                s += p
                sa += abs(p)
            v = fa * s
            d = abs(fa) * sa
            if beta != 0.0:
                c = Fraction(float(np.float32(C0[i, j])))
                v += fb * c
                d += abs(fb) * abs(c)
            exact[i][j] = v
            bound[i][j] = d
            out[i, j] = round_to_f32(v)
    return out, exact, bound
