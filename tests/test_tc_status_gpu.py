"""The tensor-core kernel's bounded waits: a stalled pipeline must end with
GEMM_ERR_DEVICE_TIMEOUT in the device status word, not a hang, and leave the
context usable.  The stall is made on purpose with a test hook that keeps
the producer from issuing any copy, so the waits run out on barriers that
nothing will ever complete (no copy or MMA is in flight when they give up)."""
import os

import numpy as np
import pytest

import oracle
from workloads import matrix

pytestmark = pytest.mark.gpu


def test_stalled_pipeline_reports_timeout_and_context_survives():
    import torch
    from roofline_gb300 import gemm
    A = torch.from_numpy(matrix(256, 300, None, 1, "u11")).cuda()
    B = torch.from_numpy(matrix(300, 384, None, 2, "u11")).cuda()
    C = torch.zeros((256, 384), device="cuda")
    assert gemm.check_status() == gemm.OK
    os.environ["GEMM_DEBUG_STALL_PRODUCER"] = "1"
    os.environ["GEMM_DEBUG_WAIT_LIMIT_NS"] = "2000000"  # 2 ms
    try:
        gemm.matmul(A, B, C, mode="tf32x3")
        st = gemm.check_status()
    finally:
        del os.environ["GEMM_DEBUG_STALL_PRODUCER"]
        del os.environ["GEMM_DEBUG_WAIT_LIMIT_NS"]
    assert st == gemm.ERR_DEVICE_TIMEOUT
    assert gemm.check_status() == gemm.OK  # read-and-clear
    # the context still works and the next call is correct
    gemm.matmul(A, B, C, mode="tf32x3")
    torch.cuda.synchronize()
    ref, D = oracle.gemm(A.cpu().numpy(), B.cpu().numpy(), with_bound=True)
    assert oracle.err_normalised(C.cpu().numpy(), ref, D) <= 1e-5
    assert gemm.check_status() == gemm.OK


def test_streaming_host_call_with_a_block_that_never_lands():
    """gemm_f32_host in its streaming form waits, tile by tile, for flags the
    copy stream sets as A's row blocks land.  With a test hook one block's
    flag is never set: the tiles of that block wait until the (shortened)
    wait limit, the GEMM gives up, releases the copies back that wait on it,
    and the call returns GEMM_ERR_DEVICE_TIMEOUT instead of hanging; the next
    call is correct."""
    import torch
    from roofline_gb300 import gemm
    M, N, K = 1280, 1536, 1024  # 240 tiles of 128 x 64: A split on chip, so it streams
    a = matrix(M, K, None, 11, "int2")
    b = matrix(K, N, None, 12, "int2")
    hA = torch.from_numpy(a).pin_memory()
    hB = torch.from_numpy(b).pin_memory()
    hC = torch.zeros((M, N), dtype=torch.float32).pin_memory()
    env = {"GEMM_HOST_STREAM": "1", "GEMM_HOST_STREAM_ROWS": "256",
           "GEMM_DEBUG_STREAM_SKIP_BLOCK": "2", "GEMM_DEBUG_WAIT_LIMIT_NS": "50000000"}
    os.environ.update(env)
    try:
        rc = gemm.gemm_f32_host(M, N, K, 1.0, hA.data_ptr(), K, hB.data_ptr(), N, 0.0,
                                hC.data_ptr(), N, gemm.MODES["tf32x3"], 0)
    finally:
        for k in env:
            del os.environ[k]
    assert rc == gemm.ERR_DEVICE_TIMEOUT, gemm.strerror(rc)
    assert gemm.check_status() == gemm.OK  # the call read and cleared the word
    os.environ["GEMM_HOST_STREAM"] = "1"
    try:
        rc = gemm.gemm_f32_host(M, N, K, 1.0, hA.data_ptr(), K, hB.data_ptr(), N, 0.0,
                                hC.data_ptr(), N, gemm.MODES["tf32x3"], 0)
    finally:
        del os.environ["GEMM_HOST_STREAM"]
    assert rc == gemm.OK, gemm.strerror(rc)
    assert oracle.mismatches(hC.numpy(), oracle.gemm(a, b)) == 0
