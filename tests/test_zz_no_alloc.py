"""gemm_f32_splitk_noalloc: the split-K GEMM for callers that cannot allocate
device memory (a fixed memory budget, or no room for cudaMalloc's device-wide
synchronisation in a hot loop).  Its partial sums live in the library's
static device array instead of a cudaMalloc'd workspace.

Checked through the C ABI against the oracle and against the ordinary entry
point (gemm_f32_ex, FP32_SIMT) on the same inputs, twice, with a call on
other inputs in between, because every call reuses the same array and must
not depend on what an earlier call left in it.  This file sorts last so that
a run stopping at the first failure has already run everything else; it
also passes on its own in a fresh process."""
import numpy as np
import pytest

import oracle
from workloads import matrix, sample_entries

pytestmark = pytest.mark.gpu

TOL_E1 = 1e-5


@pytest.fixture(scope="module")
def lib():
    from roofline_gb300 import build, gemm
    build.build()
    return gemm


def _stream():
    import torch
    return torch.cuda.current_stream().cuda_stream


def _existing(gemm, dA, dB, dC0, M, N, K, alpha, beta):
    C = dC0.clone()
    rc = gemm.gemm_f32_ex(M, N, K, alpha, dA.data_ptr(), K, dB.data_ptr(), N, beta,
                          C.data_ptr(), N, gemm.MODE_FP32_SIMT, None, 0, _stream())
    assert rc == gemm.OK
    return C


def _noalloc(gemm, dA, dB, dC0, M, N, K, alpha, beta, split):
    C = dC0.clone()
    rc = gemm.gemm_f32_splitk_noalloc(M, N, K, alpha, dA.data_ptr(), K, dB.data_ptr(), N,
                                      beta, C.data_ptr(), N, split, _stream())
    assert rc == gemm.OK, gemm.strerror(rc)
    return C


def _inputs(M, N, K, seed, dist="u11"):
    import torch
    A = matrix(M, K, None, seed, dist)
    B = matrix(K, N, None, seed + 1, dist)
    C0 = matrix(M, N, None, seed + 2, dist)
    return (A, B, C0), tuple(torch.from_numpy(x).cuda() for x in (A, B, C0))


@pytest.mark.parametrize("shape,split", [((512, 512, 512), 0), ((512, 512, 512), 8),
                                         ((300, 200, 1000), 3), ((1023, 1025, 777), 1),
                                         ((64, 48, 40000), 256)])
def test_noalloc_matches_oracle_and_existing_entry_point_twice(lib, shape, split):
    import torch
    gemm = lib
    M, N, K = shape
    (A, B, C0), (dA, dB, dC0) = _inputs(M, N, K, 31 + M)
    ref, D = oracle.gemm(A, B, 1.5, 0.5, C0, with_bound=True)
    want = _existing(gemm, dA, dB, dC0, M, N, K, 1.5, 0.5)
    torch.cuda.synchronize()
    want = want.cpu().numpy()
    assert oracle.err_normalised(want, ref, D) <= TOL_E1
    # another product in between leaves other partial sums in the array
    _, (oA, oB, oC) = _inputs(M, N, K, 977 + N)
    for i in range(2):
        got = _noalloc(gemm, dA, dB, dC0, M, N, K, 1.5, 0.5, split)
        torch.cuda.synchronize()
        got = got.cpu().numpy()
        assert oracle.err_normalised(got, ref, D) <= TOL_E1, i
        assert oracle.err_normalised(got, want, D) <= TOL_E1, i
        if i == 0:
            _noalloc(gemm, oA, oB, oC, M, N, K, -2.0, 1.0, split)


@pytest.mark.parametrize("split", [2, 7, 0])
def test_noalloc_integer_inputs_bit_exact(lib, split):
    # integer-valued inputs in {-2..2}: every partial sum is an integer below
    # 2^24, so each slice and their sum are exact, whatever the slice count
    import torch
    gemm = lib
    M, N, K = 384, 320, 2048
    (A, B, _), (dA, dB, _) = _inputs(M, N, K, 4242, "int2")
    ref = oracle.gemm(A, B)
    zero = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    _, (oA, oB, oC) = _inputs(M, N, K, 5151, "int2")
    for i in range(2):
        got = _noalloc(gemm, dA, dB, zero, M, N, K, 1.0, 0.0, split)
        torch.cuda.synchronize()
        assert oracle.mismatches(got.cpu().numpy(), ref) == 0, i
        if i == 0:
            _noalloc(gemm, oA, oB, oC, M, N, K, 1.0, 1.0, split)


def test_noalloc_fits_the_planner_split_to_the_array(lib):
    # split_k = 0 on a shape whose planner slice count (7 for the CUDA cores)
    # would need 28 MiB of partial sums: the call takes as many slices as the
    # 8 MiB array holds (2) instead of failing
    import torch
    gemm = lib
    M, N, K = 1024, 1024, 16384
    p = gemm.plan(M, N, K, mode="fp32_simt")
    assert p["split_k"] * M * N * 4 > gemm.NOALLOC_SCRATCH_BYTES
    (A, B, _), (dA, dB, _) = _inputs(M, N, K, 6161)
    zero = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    got = _noalloc(gemm, dA, dB, zero, M, N, K, 1.0, 0.0, 0)
    torch.cuda.synchronize()
    rows, cols = sample_entries(M, N, n=4096, seed=17)
    ref, D = oracle.gemm_entries(A, B, rows, cols)
    assert oracle.err_normalised(got.cpu().numpy()[rows, cols], ref, D) <= TOL_E1


def test_noalloc_allocates_no_device_memory(lib):
    # with the library's own workspace released, a split-K call changes the
    # device's free memory by nothing (a first call loads the kernels and
    # looks up the array's address; the calls measured come after it)
    import torch
    gemm = lib
    M, N, K = 512, 512, 4096
    (_, _, _), (dA, dB, dC0) = _inputs(M, N, K, 7171)
    gemm.shutdown()
    _noalloc(gemm, dA, dB, dC0, M, N, K, 1.0, 0.5, 8)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    C = dC0.clone()
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        rc = gemm.gemm_f32_splitk_noalloc(M, N, K, 1.0, dA.data_ptr(), K, dB.data_ptr(), N, 0.5,
                                          C.data_ptr(), N, 8, _stream())
        assert rc == gemm.OK
    torch.cuda.synchronize()
    free2, _ = torch.cuda.mem_get_info()
    assert free2 == free1, (free0, free1, free2)


def test_noalloc_rejects_scratch_beyond_its_maximum(lib):
    import torch
    gemm = lib
    M = N = 512
    K = 4096
    dA = torch.zeros((M, K), device="cuda")
    dB = torch.zeros((K, N), device="cuda")
    C = torch.full((M, N), 7.0, device="cuda")
    split = 16  # 16 * 512 * 512 * 4 bytes = 16 MiB of partial sums
    assert split * M * N * 4 > gemm.NOALLOC_SCRATCH_BYTES
    rc = gemm.gemm_f32_splitk_noalloc(M, N, K, 1.0, dA.data_ptr(), K, dB.data_ptr(), N, 0.0,
                                      C.data_ptr(), N, split, _stream())
    assert rc == gemm.ERR_WORKSPACE_TOO_SMALL
    for bad in (-1, gemm.NOALLOC_MAX_SPLIT + 1):
        rc = gemm.gemm_f32_splitk_noalloc(M, N, K, 1.0, dA.data_ptr(), K, dB.data_ptr(), N, 0.0,
                                          C.data_ptr(), N, bad, _stream())
        assert rc == gemm.ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert torch.all(C == 7.0)  # nothing was launched
