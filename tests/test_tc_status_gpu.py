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
