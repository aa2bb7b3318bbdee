"""GPU parity for gemm_f32_host: host buffers in, host buffer out, the
product pipelined in row blocks (copies of later blocks overlapping the GEMM
of the current one).  Checked against the oracle on the same seeded inputs,
and bit for bit against the device-pointer call when both run one block
with the same plan."""
import numpy as np
import pytest

import oracle
from tests.gpu_util import TOL_E1
from workloads import matrix, sample_entries

pytestmark = pytest.mark.gpu


def host_tensor(arr, pinned):
    import torch
    t = torch.from_numpy(arr)
    return t.pin_memory() if pinned else t.clone()


def run_host(M, N, K, alpha, beta, mode, blocks, pad=(0, 0, 0), dist="u11", pinned=True,
             seed=900):
    import torch
    from roofline_gb300 import gemm
    a = matrix(M, K, K + pad[0], seed, dist)
    b = matrix(K, N, N + pad[1], seed + 1, dist)
    c = matrix(M, N, N + pad[2], seed + 2, dist)
    hA, hB, hC = host_tensor(a, pinned), host_tensor(b, pinned), host_tensor(c, pinned)
    rc = gemm.gemm_f32_host(M, N, K, alpha, hA.data_ptr(), K + pad[0], hB.data_ptr(), N + pad[1],
                            beta, hC.data_ptr(), N + pad[2], gemm.MODES[mode], blocks)
    assert rc == gemm.OK, gemm.strerror(rc)
    out = hC.numpy()
    if pad[2]:
        assert np.all(np.isnan(out[:, N:]))  # padding of C untouched
    return a[:, :K], b[:, :N], c[:, :N], out[:, :N].copy()


CASES = [
    # (M, N, K, blocks)
    (1000, 300, 257, 3),    # ragged last block
    (777, 513, 129, 0),
    (513, 64, 1000, 5),
    (128, 200, 64, 1),
    (1, 7, 3, 0),
    (300, 1, 65, 4),
]


@pytest.mark.parametrize("case", CASES)
@pytest.mark.parametrize("mode", ["fp32_simt", "tf32x3", "tf32", "auto"])
@pytest.mark.parametrize("beta", [0.0, -0.75])
def test_host_matches_oracle(case, mode, beta):
    M, N, K, blocks = case
    A, B, C0, got = run_host(M, N, K, 1.5, beta, mode, blocks, pad=(3, 1, 2))
    ref, D = oracle.gemm(A, B, 1.5, beta, C0 if beta else None, with_bound=True)
    tol = 2e-3 if mode == "tf32" else TOL_E1
    assert oracle.err_normalised(got, ref, D) <= tol


@pytest.mark.parametrize("mode", ["fp32_simt", "tf32x3"])
@pytest.mark.parametrize("blocks", [1, 4, 7])
def test_host_integer_bit_exact(mode, blocks):
    A, B, C0, got = run_host(1100, 260, 300, 1.0, 0.0, mode, blocks, dist="int2")
    assert oracle.mismatches(got, oracle.gemm(A, B, 1.0, 0.0, None)) == 0


GRID_CASES = [
    # (M, N, K, row blocks, column blocks): A row blocks and B column blocks
    # arrive alternately; ragged last blocks both ways
    (1000, 700, 257, 3, 3),
    (777, 1300, 129, 2, 5),
    (300, 2000, 96, 1, 4),   # one row block: each B column block is one GEMM
    (1100, 513, 300, 4, 2),
]


@pytest.mark.parametrize("case", GRID_CASES)
@pytest.mark.parametrize("mode", ["fp32_simt", "tf32x3", "auto"])
@pytest.mark.parametrize("beta", [0.0, 0.5])
def test_host_grid_of_blocks(case, mode, beta, monkeypatch):
    M, N, K, nb, nc = case
    monkeypatch.setenv("GEMM_HOST_COL_BLOCKS", str(nc))
    A, B, C0, got = run_host(M, N, K, -1.25, beta, mode, nb, pad=(1, 3, 2))
    ref, D = oracle.gemm(A, B, -1.25, beta, C0 if beta else None, with_bound=True)
    assert oracle.err_normalised(got, ref, D) <= TOL_E1
    # integer inputs: exact whatever the blocking
    A, B, C0, got = run_host(M, N, K, 1.0, 1.0, mode, nb, dist="int2", seed=77)
    assert oracle.mismatches(got, oracle.gemm(A, B, 1.0, 1.0, C0)) == 0


STREAM_CASES = [
    # (M, N, K, rows per block or None for the library's choice): blocks == 0
    # with K % 4 == 0 and a tensor-core plan that splits A on chip, so with
    # GEMM_HOST_STREAM=1 the call takes the streaming form (one GEMM launch
    # consuming row blocks of A as they land, C copied back block by block as
    # the GEMM publishes it)
    (2048, 2048, 2048, None),
    (1500, 1024, 1024, 384),   # ragged last row block
    (1100, 1300, 512, 128),    # many small blocks, ragged edges
    (4096, 64, 2048, None),    # narrow: the skinny shape's plan
]


@pytest.mark.parametrize("case", STREAM_CASES)
@pytest.mark.parametrize("mode", ["tf32x3", "auto"])
@pytest.mark.parametrize("beta", [0.0, -0.75])
def test_host_streaming_matches_oracle(case, mode, beta, monkeypatch):
    M, N, K, rows = case
    monkeypatch.setenv("GEMM_HOST_STREAM", "1")
    if rows:
        monkeypatch.setenv("GEMM_HOST_STREAM_ROWS", str(rows))
    A, B, C0, got = run_host(M, N, K, 1.5, beta, mode, 0, pad=(3, 1, 2), seed=M + N)
    if M * N * K > 2 ** 30:
        rows_, cols_ = sample_entries(M, N, n=8192, seed=11)
        ref, D = oracle.gemm_entries(A, B, rows_, cols_, 1.5, beta, C0 if beta else None)
        assert oracle.err_normalised(got[rows_, cols_], ref, D) <= TOL_E1
    else:
        ref, D = oracle.gemm(A, B, 1.5, beta, C0 if beta else None, with_bound=True)
        assert oracle.err_normalised(got, ref, D) <= TOL_E1


def test_host_streaming_tf32_mode(monkeypatch):
    """1xTF32 through the streaming form (the narrow tile splits A on chip):
    within the mode's bound."""
    from tests.gpu_util import tol_tf32
    monkeypatch.setenv("GEMM_HOST_STREAM", "1")
    M, N, K = 2048, 64, 1024
    A, B, C0, got = run_host(M, N, K, 1.0, 0.5, "tf32", 0, pad=(0, 0, 0), seed=71)
    ref, D = oracle.gemm(A, B, 1.0, 0.5, C0, with_bound=True)
    assert oracle.err_normalised(got, ref, D) <= tol_tf32(K)


@pytest.mark.parametrize("stream", ["1", "0"])
def test_host_streaming_integer_bit_exact_and_repeatable(stream, monkeypatch):
    """Integer inputs are exact in either form (streaming on, or the blocked
    form with GEMM_HOST_STREAM=0); repeated streaming calls reuse the flags
    (a new value each call) and stay exact."""
    monkeypatch.setenv("GEMM_HOST_STREAM", stream)
    monkeypatch.setenv("GEMM_HOST_STREAM_ROWS", "256")
    for rep in range(3):
        A, B, C0, got = run_host(1280, 1536, 1024, 1.0, 1.0, "tf32x3", 0, dist="int2",
                                 seed=300 + rep)
        assert oracle.mismatches(got, oracle.gemm(A, B, 1.0, 1.0, C0)) == 0, rep


def test_host_auto_grid_2048():
    """2048 x 2048 x 1024 (8.6 GFLOP): the library's blocking is 2 x 2."""
    import torch
    from roofline_gb300 import gemm
    M, N, K = 2048, 2048, 1024
    a = matrix(M, K, None, 5, "u11")
    b = matrix(K, N, None, 6, "u11")
    c = matrix(M, N, None, 7, "u11")
    hC = torch.from_numpy(c.copy()).pin_memory()
    gemm.matmul_host(torch.from_numpy(a).pin_memory(), torch.from_numpy(b).pin_memory(), hC,
                     0.75, -0.5, blocks=0)
    rows, cols = sample_entries(M, N, n=20000, seed=3)
    ref, D = oracle.gemm_entries(a, b, rows, cols, 0.75, -0.5, c)
    assert oracle.err_normalised(hC.numpy()[rows, cols], ref, D) <= TOL_E1


def test_host_pageable_buffers():
    A, B, C0, got = run_host(700, 400, 300, 1.0, 0.5, "auto", 3, pinned=False)
    ref, D = oracle.gemm(A, B, 1.0, 0.5, C0, with_bound=True)
    assert oracle.err_normalised(got, ref, D) <= TOL_E1


def test_host_k_zero_scales_c():
    # lda >= max(K, 1) = 1, as in BLAS
    A, B, C0, got = run_host(300, 200, 0, 1.0, 2.0, "auto", 2, pad=(1, 0, 0))
    assert np.array_equal(got, np.float32(2.0) * C0)


@pytest.mark.parametrize("mode", ["fp32_simt", "tf32x3"])
def test_host_one_block_equals_device_call(mode):
    import torch
    from roofline_gb300 import gemm
    M, N, K = 640, 384, 320
    A, B, C0, got = run_host(M, N, K, 0.5, 0.25, mode, 1)
    dC = torch.from_numpy(C0.copy()).cuda()
    gemm.matmul(torch.from_numpy(A.copy()).cuda(), torch.from_numpy(B.copy()).cuda(), dC, 0.5,
                0.25, mode)
    torch.cuda.synchronize()
    assert np.array_equal(got.view(np.uint32), dC.cpu().numpy().view(np.uint32))


@pytest.mark.parametrize("blocks", [0, 8])
def test_host_square_4096_sampled(blocks):
    import torch
    from roofline_gb300 import gemm
    from workloads import WORKLOADS
    w = WORKLOADS["sq4096"]
    a, b, _ = w.make()
    hA = torch.from_numpy(a).pin_memory()
    hB = torch.from_numpy(b).pin_memory()
    hC = gemm.matmul_host(hA[:, :w.K], hB[:, :w.N], blocks=blocks)
    rows, cols = sample_entries(w.M, w.N)
    ref, D = oracle.gemm_entries(a[:, :w.K], b[:, :w.N], rows, cols, 1.0, 0.0, None)
    assert oracle.err_normalised(hC.numpy()[rows, cols], ref, D) <= TOL_E1


def test_host_calls_from_two_threads():
    # calls on one device are serialised by the library; results stay exact
    import threading

    import torch
    from roofline_gb300 import gemm
    M, N, K = 700, 520, 300
    jobs = []
    for seed in (1, 2):
        a = matrix(M, K, None, 100 * seed, "int2")
        b = matrix(K, N, None, 100 * seed + 1, "int2")
        jobs.append((torch.from_numpy(a).pin_memory(), torch.from_numpy(b).pin_memory(),
                     oracle.gemm(a, b, 1.0, 0.0, None)))
    out = [None, None]
    errs = []

    def work(i):
        try:
            for _ in range(5):
                out[i] = gemm.matmul_host(jobs[i][0], jobs[i][1], mode="auto", blocks=3).numpy()
        except Exception as e:  # pragma: no cover - reported below
            errs.append(e)

    ts = [threading.Thread(target=work, args=(i,)) for i in range(2)]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    assert not errs, errs
    for i in range(2):
        assert oracle.mismatches(out[i], jobs[i][2]) == 0


@pytest.mark.parametrize("shape,blocks", [((4097, 1024, 1600), 0), ((1700, 2048, 1152), 4)])
def test_host_blocks_mixing_on_chip_and_pass_b_splits(shape, blocks):
    """Row blocks whose GEMMs split B differently in one column block: the
    full blocks are small products that split B on chip (no planes in the
    workspace) and the short last block splits B with the pass, so it must
    not take the column's planes as already written.  (4097 x 1024 x 1600:
    the library's blocking, 3 x 1152 rows + 641; 1700 x 2048 x 1152 in 4
    blocks: 3 x 512 + 164.)"""
    import torch
    from roofline_gb300 import gemm
    M, N, K = shape
    rows = -(-M // (blocks if blocks else 4)) if blocks else 1152
    rows = -(-rows // 128) * 128
    first = gemm.plan(rows, N, K, K, N, N, mode="tf32x3")
    last = gemm.plan(M - (-(-M // rows) - 1) * rows, N, K, K, N, N, mode="tf32x3")
    assert first["b_split_in_kernel"] == 1 and last["b_split_in_kernel"] == 0
    a = matrix(M, K, None, 15, "u11")
    b = matrix(K, N, None, 16, "u11")
    c = matrix(M, N, None, 17, "u11")
    hC = torch.from_numpy(c.copy()).pin_memory()
    gemm.matmul_host(torch.from_numpy(a).pin_memory(), torch.from_numpy(b).pin_memory(), hC,
                     0.75, -0.5, mode="tf32x3", blocks=blocks)
    rows_s, cols_s = sample_entries(M, N, n=8192, seed=5)
    # every row of the last block is checked as well
    tail = np.arange(M - 164 if blocks else M - 641, M)
    rows_s = np.concatenate([rows_s, tail])
    cols_s = np.concatenate([cols_s, (tail * 7) % N])
    ref, D = oracle.gemm_entries(a, b, rows_s, cols_s, 0.75, -0.5, c)
    assert oracle.err_normalised(hC.numpy()[rows_s, cols_s], ref, D) <= TOL_E1
