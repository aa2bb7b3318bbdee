"""GPU parity for gemm_f32_op: every storage order and operand op.

The operation is C <- alpha * op(A) op(B) + beta * C of the course page's
cuBLAS stage ("Project - tiled matrix multiply", "Stage 3 - the reference
ceiling: cuBLAS"), with op(X) = X or X^T and row- or column-major storage.
Each case is checked twice: against the oracle on the logical matrices
(within the E1 bound, or bit-exact on integer inputs), and bit for bit
against gemm_f32_ex on the same logical matrices stored plainly, with the
same kernel configuration.
"""
import itertools

import numpy as np
import pytest

import oracle
from tests.gpu_util import TOL_E1
from workloads import matrix

pytestmark = pytest.mark.gpu

ROW, COL, N_, T_ = 0, 1, 0, 1


def _dense(x):
    """A fresh C-ordered copy (canonical strides even for 1 x 1 views)."""
    return np.array(x, dtype=np.float32, order="C", copy=True)


COMBOS = list(itertools.product([ROW, COL], [N_, T_], [N_, T_]))


def stored(layout, op, rows, cols, pad, seed, dist):
    """(buffer, ld, logical op(X) as a rows x cols array) for an operand whose
    op(X) is rows x cols.  The buffer's padding is NaN."""
    sr, sc = (rows, cols) if op == N_ else (cols, rows)
    if layout == ROW:
        ld = sc + pad
        buf = matrix(sr, sc, ld, seed, dist)
        S = buf[:, :sc]
    else:
        ld = sr + pad
        buf = matrix(sc, sr, ld, seed, dist)
        S = buf[:, :sr].T
    X = S if op == N_ else S.T
    return buf, ld, _dense(X)


def c_buffer(layout, M, N, pad, seed, dist):
    if layout == ROW:
        ld = N + pad
        buf = matrix(M, N, ld, seed, dist)
        return buf, ld, _dense(buf[:, :N])
    ld = M + pad
    buf = matrix(N, M, ld, seed, dist)
    return buf, ld, _dense(buf[:, :M].T)


def c_logical(layout, buf, M, N):
    return buf[:, :N] if layout == ROW else buf[:, :M].T


def run_op(layout, op_a, op_b, M, N, K, alpha, beta, dist, mode, pad=3, seed=700):
    import torch
    from roofline_gb300 import gemm
    bA, lda, A = stored(layout, op_a, M, K, pad, seed, dist)
    bB, ldb, B = stored(layout, op_b, K, N, pad, seed + 1, dist)
    bC, ldc, C0 = c_buffer(layout, M, N, pad, seed + 2, dist)
    dA, dB, dC = (torch.from_numpy(x).cuda() for x in (bA, bB, bC))
    rc = gemm.gemm_f32_op(layout, op_a, op_b, M, N, K, alpha, dA.data_ptr(), lda, dB.data_ptr(),
                          ldb, beta, dC.data_ptr(), ldc, mode, None, 0,
                          torch.cuda.current_stream().cuda_stream)
    assert rc == gemm.OK, gemm.strerror(rc)
    torch.cuda.synchronize()
    out = dC.cpu().numpy()
    if pad:  # padding of C is never written
        pad_part = out[:, N:] if layout == ROW else out[:, M:]
        assert np.all(np.isnan(pad_part))
    return A, B, C0, _dense(c_logical(layout, out, M, N))


def run_plain(A, B, C0, alpha, beta, mode, transpose_problem=False):
    """gemm_f32_ex on plainly stored logical matrices (or, for a column-major
    call, on the transposed problem C^T = B^T A^T that it runs)."""
    import torch
    from roofline_gb300 import gemm
    if transpose_problem:
        A, B, C0 = _dense(B.T), _dense(A.T), _dense(C0.T)
    dA, dB, dC = (torch.from_numpy(x).cuda() for x in (A, B, C0))
    gemm.matmul(dA, dB, dC, alpha, beta, mode)
    torch.cuda.synchronize()
    out = dC.cpu().numpy()
    return out.T if transpose_problem else out


SHAPES = [(200, 330, 77), (129, 64, 257), (1, 300, 65), (300, 5, 1000)]


@pytest.mark.parametrize("layout,op_a,op_b", COMBOS)
@pytest.mark.parametrize("mode", ["fp32_simt", "tf32x3", "auto"])
@pytest.mark.parametrize("shape", SHAPES)
def test_op_matches_oracle(layout, op_a, op_b, mode, shape):
    M, N, K = shape
    A, B, C0, got = run_op(layout, op_a, op_b, M, N, K, 1.25, -0.5, "u11", mode)
    ref, D = oracle.gemm(A, B, 1.25, -0.5, C0, with_bound=True)
    assert oracle.err_normalised(got, ref, D) <= TOL_E1


@pytest.mark.parametrize("layout,op_a,op_b", COMBOS)
@pytest.mark.parametrize("mode", ["fp32_simt", "tf32x3"])
def test_op_integer_inputs_bit_exact(layout, op_a, op_b, mode):
    # integer entries in {-2..2}: every partial sum is exact in FP32 (and in
    # the hi part of the TF32 split), so the result equals the oracle exactly
    M, N, K = 257, 190, 300
    A, B, C0, got = run_op(layout, op_a, op_b, M, N, K, 1.0, 0.0, "int2", mode)
    ref = oracle.gemm(A, B, 1.0, 0.0, None)
    assert oracle.mismatches(got, ref) == 0


@pytest.mark.parametrize("layout,op_a,op_b", COMBOS)
def test_op_tf32_mode(layout, op_a, op_b):
    M, N, K = 300, 260, 200
    A, B, C0, got = run_op(layout, op_a, op_b, M, N, K, 1.0, 0.0, "u11", "tf32")
    ref, D = oracle.gemm(A, B, 1.0, 0.0, None, with_bound=True)
    # one TF32 product per term: each operand keeps 11 significant bits, so
    # E1 stays below 2^-10 plus the FP32 accumulation error; 2e-3 bounds both
    assert oracle.err_normalised(got, ref, D) <= 2e-3


# configurations forced on both calls, so both run the same kernel with the
# pre-split A that a transposed A needs
SAME_CFG = {"fp32_simt": None, "tf32x3": "256,16,4,0,0", "tf32": "256,16,8,0,0"}


@pytest.mark.parametrize("layout,op_a,op_b", COMBOS)
@pytest.mark.parametrize("mode", list(SAME_CFG))
def test_op_bitwise_equals_plain_storage(layout, op_a, op_b, mode, monkeypatch):
    if SAME_CFG[mode]:
        monkeypatch.setenv("GEMM_TC_CONFIG", SAME_CFG[mode])
    M, N, K = 333, 270, 161
    A, B, C0, got = run_op(layout, op_a, op_b, M, N, K, 0.75, 0.5, "u11", mode)
    want = run_plain(A, B, C0, 0.75, 0.5, mode, transpose_problem=(layout == COL))
    assert np.array_equal(_dense(got).view(np.uint32),
                          _dense(want).view(np.uint32))


def test_matmul_takes_transposed_views():
    import torch
    from roofline_gb300 import gemm
    M, N, K = 190, 250, 130
    At = torch.from_numpy(matrix(K, M, M, 11, "u11")).cuda()   # A^T stored row-major
    Bt = torch.from_numpy(matrix(N, K, K, 12, "u11")).cuda()   # B^T stored row-major
    C = gemm.matmul(At.t(), Bt.t(), mode="fp32_simt")
    torch.cuda.synchronize()
    A = _dense(At.cpu().numpy().T)
    B = _dense(Bt.cpu().numpy().T)
    ref, D = oracle.gemm(A, B, 1.0, 0.0, None, with_bound=True)
    assert oracle.err_normalised(C.cpu().numpy(), ref, D) <= TOL_E1


@pytest.mark.parametrize("mode", ["fp32_simt", "tf32x3"])
def test_op_large_transposed_sampled(mode):
    # a 4096^3 problem with both operands transposed, checked on sampled entries
    import torch
    from roofline_gb300 import gemm
    from workloads import sample_entries
    M = N = K = 4096
    At = matrix(K, M, M, 21, "u11")
    Bt = matrix(N, K, K, 22, "u11")
    dAt, dBt = torch.from_numpy(At).cuda(), torch.from_numpy(Bt).cuda()
    C = gemm.matmul(dAt.t(), dBt.t(), mode=mode)
    torch.cuda.synchronize()
    rows, cols = sample_entries(M, N, n=2048)
    A = _dense(At.T)
    B = _dense(Bt.T)
    ref, D = oracle.gemm_entries(A, B, rows, cols, 1.0, 0.0, None)
    got = C.cpu().numpy()[rows, cols]
    assert oracle.err_normalised(got, ref, D) <= TOL_E1


# built (BK, stages) of the CUDA-core kernel
SIMT_BUILT = ["16,4", "32,2"]


@pytest.mark.parametrize("cfg", SIMT_BUILT)
@pytest.mark.parametrize("op_a,op_b", [(N_, N_), (T_, N_), (N_, T_), (T_, T_)])
@pytest.mark.parametrize("shape", [(333, 270, 161), (64, 128, 32), (1, 1, 1), (200, 131, 1003)])
def test_simt_every_built_configuration(cfg, op_a, op_b, shape, monkeypatch):
    from roofline_gb300 import gemm
    monkeypatch.setenv("GEMM_SIMT_CONFIG", cfg)
    M, N, K = shape
    p = gemm.plan_op(ROW, op_a, op_b, M, N, K, mode="fp32_simt")
    assert "%d,%d" % (p["bk"], p["stages"]) == cfg
    A, B, C0, got = run_op(ROW, op_a, op_b, M, N, K, 1.25, 0.5, "u11", "fp32_simt")
    ref, D = oracle.gemm(A, B, 1.25, 0.5, C0, with_bound=True)
    assert oracle.err_normalised(got, ref, D) <= TOL_E1
    A, B, C0, got = run_op(ROW, op_a, op_b, M, N, K, 1.0, 0.0, "int2", "fp32_simt")
    assert oracle.mismatches(got, oracle.gemm(A, B, 1.0, 0.0, None)) == 0


@pytest.mark.parametrize("group", ["1", "3", "8", "40"])
@pytest.mark.parametrize("op_b", [N_, T_])
def test_simt_tile_orders(group, op_b, monkeypatch):
    # the tile order is a bijection of the grid for any group size, ragged
    # row-tile counts included (1000 rows = 15.6 row-tiles)
    monkeypatch.setenv("GEMM_SIMT_GROUP", group)
    M, N, K = 1000, 1100, 96
    A, B, C0, got = run_op(ROW, N_, op_b, M, N, K, 1.0, 0.0, "int2", "fp32_simt")
    assert oracle.mismatches(got, oracle.gemm(A, B, 1.0, 0.0, None)) == 0


# Tensor-core configurations built with B split on chip, for B stored N x K
# (bm, bn, bk, stages, a_split, b_concat): read as stored, B_hi is the landed
# tile itself and B_lo = B - tf32_trunc(B) is written beside it on chip.
TC_BSPLIT = ["128,256,16,5,2,0", "128,128,32,4,2,1", "128,64,32,6,1,1", "128,64,32,4,0,1"]


@pytest.mark.parametrize("cfg", TC_BSPLIT)
@pytest.mark.parametrize("shape", [(333, 270, 164), (129, 64, 777), (1, 300, 68), (300, 5, 1000)])
def test_tc_b_split_on_chip_every_configuration(cfg, shape, monkeypatch):
    from roofline_gb300 import gemm
    M, N, K = shape
    # A split on chip needs A stored M x K; the pre-split-A configuration
    # takes a transposed A too
    op_a = N_ if cfg.split(",")[4] != "0" else T_
    pad = (-K) % 4  # ld = K + pad: rows of B (N x K) start on 16-byte boundaries
    ldb = K + pad
    lda = K + pad if op_a == N_ else M + pad
    monkeypatch.setenv("GEMM_TC_CONFIG", cfg + ",1")
    p = gemm.plan_op(ROW, op_a, T_, M, N, K, lda=lda, ldb=ldb, ldc=N + pad, mode="tf32x3")
    assert p["b_split_in_kernel"] == 1
    assert "%d,%d,%d,%d" % (p["bm"], p["bn"], p["bk"], p["stages"]) == cfg.rsplit(",", 2)[0]
    A, B, C0, got = run_op(ROW, op_a, T_, M, N, K, 1.25, -0.5, "u11", "tf32x3", pad=pad)
    ref, D = oracle.gemm(A, B, 1.25, -0.5, C0, with_bound=True)
    assert oracle.err_normalised(got, ref, D) <= TOL_E1
    # the same bits as this configuration with B split by the pass (both
    # take B_hi = tf32_trunc(B) and issue the same MMAs in the same order)
    monkeypatch.setenv("GEMM_TC_CONFIG", cfg + ",0")
    _, _, _, got0 = run_op(ROW, op_a, T_, M, N, K, 1.25, -0.5, "u11", "tf32x3", pad=pad)
    assert np.array_equal(_dense(got).view(np.uint32), _dense(got0).view(np.uint32))
    monkeypatch.setenv("GEMM_TC_CONFIG", cfg + ",1")
    A, B, C0, got = run_op(ROW, op_a, T_, M, N, K, 1.0, 0.0, "int2", "tf32x3", pad=pad)
    assert oracle.mismatches(got, oracle.gemm(A, B, 1.0, 0.0, None)) == 0


def test_tc_b_split_on_chip_planner_sampled():
    # 2048^3 with B stored N x K: the planner's one-wave choice splits both
    # operands on chip, one launch; sampled entries against the oracle
    import torch
    from roofline_gb300 import gemm
    from workloads import sample_entries
    M = N = K = 2048
    A = matrix(M, K, K, 31, "u11")
    Bt = matrix(N, K, K, 32, "u11")
    p = gemm.plan_op(ROW, N_, T_, M, N, K, mode="auto")
    assert (p["kernel_name"], p["a_split_in_kernel"], p["b_split_in_kernel"], p["launches"]) == \
        ("tc_tf32x3", 1, 1, 1)
    C = gemm.matmul(torch.from_numpy(A).cuda(), torch.from_numpy(Bt).cuda().t(), mode="auto")
    torch.cuda.synchronize()
    rows, cols = sample_entries(M, N, n=2048)
    ref, D = oracle.gemm_entries(A, _dense(Bt.T), rows, cols, 1.0, 0.0, None)
    assert oracle.err_normalised(C.cpu().numpy()[rows, cols], ref, D) <= TOL_E1
