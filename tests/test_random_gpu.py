"""Seeded random parity sweep: shapes, padded leading dimensions, base
offsets, alpha/beta, storage order of each operand, mode and the stream-K
switch drawn from a fixed-seed generator, each case checked against the oracle (normalised error
for the FP32 and 3xTF32 modes, the TF32 bound for 1xTF32) with C's padding
columns left untouched."""
import numpy as np
import pytest

import oracle
from tests.gpu_util import TOL_E1, tol_tf32
from workloads import matrix

N_CASES = 64


def _dense(x):
    """A fresh C-ordered copy with unit element stride on every axis (numpy
    keeps odd strides on length-1 axes of a transposed view)."""
    return np.array(x, dtype=np.float32, order="C", copy=True)


def _case(i):
    rng = np.random.default_rng(20260 + i)
    dims = [int(x) for x in rng.integers(1, 640, size=3)]
    if rng.random() < 0.25:  # one dimension large enough for several waves of tiles
        dims[int(rng.integers(0, 3))] = int(rng.integers(640, 2100))
    M, N, K = dims
    pads = [int(x) for x in rng.integers(0, 6, size=3)]
    alpha = float(rng.choice([1.0, -1.5, 0.75]))
    beta = float(rng.choice([0.0, 0.5, -1.0]))
    mode = str(rng.choice(["fp32_simt", "tf32x3", "tf32", "auto"]))
    ta, tb = bool(rng.random() < 0.3), bool(rng.random() < 0.3)
    streamk = str(rng.choice(["", "0", "1"]))
    return M, N, K, pads, alpha, beta, mode, ta, tb, streamk


@pytest.mark.gpu
@pytest.mark.parametrize("i", range(N_CASES))
def test_random_case(i, monkeypatch):
    import torch
    from roofline_gb300 import gemm
    M, N, K, pads, alpha, beta, mode, ta, tb, streamk = _case(i)
    if streamk:
        monkeypatch.setenv("GEMM_TC_STREAMK", streamk)
    seed = 31000 + 10 * i
    # A stored M x K, or K x M (then used through its transposed view)
    if ta:
        At = matrix(K, M, M + pads[0], seed, "u11")
        A = _dense(At[:, :M].T)
        dAs = torch.from_numpy(At).cuda()
        dA = dAs[:, :M].t()
    else:
        As = matrix(M, K, K + pads[0], seed, "u11")
        A = As[:, :K]
        dA = torch.from_numpy(As).cuda()[:, :K]
    if tb:
        Bt = matrix(N, K, K + pads[1], seed + 1, "u11")
        B = _dense(Bt[:, :K].T)
        dB = torch.from_numpy(Bt).cuda()[:, :K].t()
    else:
        Bs = matrix(K, N, N + pads[1], seed + 1, "u11")
        B = Bs[:, :N]
        dB = torch.from_numpy(Bs).cuda()[:, :N]
    Cs = matrix(M, N, N + pads[2], seed + 2, "u11")
    dCs = torch.from_numpy(Cs).cuda()
    # each operand at a random float offset inside a larger buffer, so base
    # addresses are 4-byte aligned only (no TMA on the operand itself)
    offs = [int(x) for x in np.random.default_rng(999 + i).integers(0, 4, size=3)]

    def shift(t, off):
        buf = torch.empty(t.numel() + 8, dtype=torch.float32, device="cuda")
        buf[off:off + t.numel()] = t.reshape(-1)
        return buf[off:off + t.numel()].view(t.shape)
    dA = shift(dAs, offs[0])[:, :M].t() if ta else shift(torch.from_numpy(As).cuda(), offs[0])[:, :K]
    dB = (shift(torch.from_numpy(Bt).cuda(), offs[1])[:, :K].t() if tb
          else shift(torch.from_numpy(Bs).cuda(), offs[1])[:, :N])
    dCs = shift(dCs, offs[2])
    gemm.matmul(dA, dB, dCs[:, :N], alpha, beta, mode)
    torch.cuda.synchronize()
    out = dCs.cpu().numpy()
    if pads[2]:
        assert np.all(np.isnan(out[:, N:])), "padding columns of C were written"
    ref, D = oracle.gemm(_dense(A), _dense(B), alpha, beta, _dense(Cs[:, :N]), with_bound=True)
    tol = tol_tf32(K) if mode == "tf32" else TOL_E1
    e1 = oracle.err_normalised(out[:, :N], ref, D)
    assert e1 <= tol, (M, N, K, pads, alpha, beta, mode, ta, tb, streamk, e1)
    assert gemm.check_status() == gemm.OK


def test_cases_cover_every_mode_and_layout():
    """The drawn cases include every mode, both storage orders of each
    operand, beta == 0 and beta != 0, and shapes past a wave of tiles."""
    cases = [_case(i) for i in range(N_CASES)]
    assert {c[6] for c in cases} == {"fp32_simt", "tf32x3", "tf32", "auto"}
    assert {c[7] for c in cases} == {False, True} and {c[8] for c in cases} == {False, True}
    assert {c[5] == 0.0 for c in cases} == {False, True}
    assert any(max(c[0], c[1], c[2]) >= 640 for c in cases)


@pytest.mark.gpu
@pytest.mark.parametrize("shape", [(1, 99, 449), (77, 1, 300), (1, 1, 513), (200, 150, 1),
                                   (1, 300, 1)], ids=lambda v: "x".join(map(str, v)))
@pytest.mark.parametrize("ta", [False, True])
@pytest.mark.parametrize("tb", [False, True])
@pytest.mark.parametrize("mode", ["fp32_simt", "tf32x3", "auto"])
def test_single_row_or_column_operands(shape, ta, tb, mode):
    """Operands with one row or one column, stored either way: torch reports
    arbitrary strides along a length-1 dimension, which the binding must not
    take for a leading dimension (a 1 x 449 transposed view has row stride 1)."""
    import torch
    from roofline_gb300 import gemm
    M, N, K = shape
    A = matrix(K, M, None, 61, "u11") if ta else matrix(M, K, None, 61, "u11")
    B = matrix(N, K, None, 62, "u11") if tb else matrix(K, N, None, 62, "u11")
    dA = torch.from_numpy(A).cuda()
    dB = torch.from_numpy(B).cuda()
    dA, dB = (dA.t() if ta else dA), (dB.t() if tb else dB)
    C = gemm.matmul(dA, dB, mode=mode)
    torch.cuda.synchronize()
    ref, D = oracle.gemm(_dense(A.T if ta else A), _dense(B.T if tb else B), with_bound=True)
    assert oracle.err_normalised(C.cpu().numpy(), ref, D) <= TOL_E1

