"""Helpers shared by the GPU parity tests: run a workload through the C ABI
and compare it with the CPU oracle on the same seeded inputs."""
from __future__ import annotations

import functools

import numpy as np

import oracle
from workloads import WORKLOADS, sample_entries

TOL_E1 = 1e-5  # max |C - C_ref| / (|alpha| sum|A||B| + |beta||C_old|), FP32 and 3xTF32 modes


@functools.lru_cache(maxsize=8)
def inputs(name: str):
    return WORKLOADS[name].make()


def run(name: str, mode, A=None, B=None, C0=None, repeat: int = 1):
    """Runs workload `name` through roofline_gb300.gemm.matmul; returns the
    full (M, ldc) C buffer after the last of `repeat` calls."""
    import torch
    from roofline_gb300 import gemm
    w = WORKLOADS[name]
    if A is None:
        A, B, C0 = inputs(name)
    lda, ldb, ldc = w.lds()
    dA = torch.from_numpy(A).cuda()
    dB = torch.from_numpy(B).cuda()
    outs = []
    for _ in range(repeat):
        if C0 is not None:
            dC = torch.from_numpy(C0).cuda()
        else:
            dC = torch.full((w.M, ldc), float("nan"), dtype=torch.float32, device="cuda")
        gemm.matmul(dA[:, :w.K], dB[:, :w.N], dC[:, :w.N], w.alpha, w.beta, mode)
        torch.cuda.synchronize()
        outs.append(dC.cpu().numpy())
    return outs if repeat > 1 else outs[0]


@functools.lru_cache(maxsize=8)
def reference(name: str):
    """(positions or None, C_ref, D) from the oracle for workload `name`."""
    w = WORKLOADS[name]
    A, B, C0 = inputs(name)
    c0 = None if C0 is None else C0[:, :w.N]
    if not w.sampled:
        ref, D = oracle.gemm(A[:, :w.K], B[:, :w.N], w.alpha, w.beta, c0, with_bound=True)
        return None, ref, D
    rows, cols = sample_entries(w.M, w.N)
    ref, D = oracle.gemm_entries(A[:, :w.K], B[:, :w.N], rows, cols, w.alpha, w.beta, c0)
    return (rows, cols), ref, D


def compare(name: str, C_full: np.ndarray):
    """Returns dict(e1, mismatches, e3) of the GPU result against the oracle."""
    w = WORKLOADS[name]
    pos, ref, D = reference(name)
    got = C_full[:, :w.N] if pos is None else C_full[pos[0], pos[1]]
    return dict(e1=oracle.err_normalised(got, ref, D), mismatches=oracle.mismatches(got, ref),
                e3=oracle.err_pages(got, ref))


# 1xTF32 mode: each operand rounded to TF32 (11 significant bits, round to
# nearest, ties away): |x - tf32(x)| <= 2^-11 |x|, so each product a*b moves by
# at most (2 * 2^-11 + 2^-22) |a||b| = (2^-10 + 2^-22) |a||b|.  The K products
# are then summed in FP32 (tensor-core accumulation, order and rounding of the
# partial sums not specified: allow 2^-23 per addition, twice the
# round-to-nearest unit), plus the alpha/beta epilogue (two roundings of
# 2^-24).  So the normalised error is at most
#     2^-10 + 2^-22 + K * 2^-23 + 2^-23.
def tol_tf32(K):
    return 2.0 ** -10 + 2.0 ** -22 + (K + 1) * 2.0 ** -23
