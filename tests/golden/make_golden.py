"""Writes tiny_gemm.json: small GEMM cases with their exactly rounded results.

Expected values come only from ``oracle.exact`` (exact rational arithmetic,
one rounding to float32).  Run from the repository root:
    python tests/golden/make_golden.py
"""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from oracle import exact  # noqa: E402
from workloads import matrix  # noqa: E402

CASES = [
    dict(M=3, N=4, K=5, alpha=1.0, beta=0.0, dist="u11", seed=9001),
    dict(M=5, N=3, K=7, alpha=1.5, beta=0.5, dist="u11", seed=9002),
    dict(M=4, N=4, K=4, alpha=1.0, beta=0.0, dist="int2", seed=9003),
    dict(M=2, N=6, K=9, alpha=-0.5, beta=2.0, dist="normal", seed=9004),
]


def main():
    out = []
    for c in CASES:
        A = matrix(c["M"], c["K"], None, c["seed"], c["dist"], 0.7)
        B = matrix(c["K"], c["N"], None, c["seed"] + 1, c["dist"], 0.7)
        C0 = matrix(c["M"], c["N"], None, c["seed"] + 2, "u11")
        want, _, _ = exact.gemm_exact(A, B, c["alpha"], c["beta"], C0)
        out.append(dict(c, A=A.tolist(), B=B.tolist(), C0=C0.tolist(),
                        C=[[float(v) for v in row] for row in want]))
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_gemm.json")
    with open(path, "w") as f:
        json.dump({"_about": "tiny GEMMs, expected = exact rational result rounded once "
                             "to float32 (written by make_golden.py via oracle.exact)",
                   "cases": out}, f, indent=1)


if __name__ == "__main__":
    main()
