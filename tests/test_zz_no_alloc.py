"""gemm_f32_splitk_noalloc: the split-K GEMM for callers that cannot allocate
device memory (a fixed memory budget, or no room for cudaMalloc's device-wide
synchronisation in a hot loop).  Its partial sums live in the library's
static device array instead of a cudaMalloc'd workspace.

Checked through the C ABI against the ordinary entry point (gemm_f32_ex,
FP32_SIMT) on the same inputs, twice in a row, because every call reuses the
same array and must not depend on what an earlier call left in it.  This
file sorts last so that a run stopping at the first failure has already run
everything else; it also passes on its own in a fresh process."""
import numpy as np
import pytest

import oracle
from workloads import matrix

pytestmark = pytest.mark.gpu

TOL_E1 = 1e-5


@pytest.fixture(scope="module")
def lib():
    from roofline_gb300 import build, gemm
    build.build()
    return gemm


def _existing(gemm, dA, dB, dC0, M, N, K, alpha, beta):
    import torch
    C = dC0.clone()
    rc = gemm.gemm_f32_ex(M, N, K, alpha, dA.data_ptr(), K, dB.data_ptr(), N, beta,
                          C.data_ptr(), N, gemm.MODE_FP32_SIMT, None, 0,
                          torch.cuda.current_stream().cuda_stream)
    assert rc == gemm.OK
    return C


def _noalloc(gemm, dA, dB, dC0, M, N, K, alpha, beta, split):
    import torch
    C = dC0.clone()
    rc = gemm.gemm_f32_splitk_noalloc(M, N, K, alpha, dA.data_ptr(), K, dB.data_ptr(), N,
                                      beta, C.data_ptr(), N, split,
                                      torch.cuda.current_stream().cuda_stream)
    assert rc == gemm.OK, gemm.strerror(rc)
    return C


@pytest.mark.parametrize("shape,split", [((512, 512, 512), 0), ((512, 512, 512), 8),
                                         ((300, 200, 1000), 3), ((1023, 1025, 777), 1)])
def test_noalloc_matches_existing_entry_point_twice(lib, shape, split):
    import torch
    gemm = lib
    M, N, K = shape
    A = matrix(M, K, None, 31 + M, "u11")
    B = matrix(K, N, None, 32 + N, "u11")
    C0 = matrix(M, N, None, 33 + K, "u11")
    dA, dB, dC0 = (torch.from_numpy(x).cuda() for x in (A, B, C0))
    _, D = oracle.gemm(A, B, 1.5, 0.5, C0, with_bound=True)
    want = _existing(gemm, dA, dB, dC0, M, N, K, 1.5, 0.5)
    torch.cuda.synchronize()
    want = want.cpu().numpy()
    for _ in range(2):
        got = _noalloc(gemm, dA, dB, dC0, M, N, K, 1.5, 0.5, split)
        torch.cuda.synchronize()
        got = got.cpu().numpy()
        assert oracle.err_normalised(got, want, D) <= TOL_E1


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
                                      C.data_ptr(), N, split,
                                      torch.cuda.current_stream().cuda_stream)
    assert rc == gemm.ERR_WORKSPACE_TOO_SMALL
    torch.cuda.synchronize()
    assert torch.all(C == 7.0)  # nothing was launched
