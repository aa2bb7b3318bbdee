"""Host-side checks of gemm_f32_host (no GPU needed): argument validation
and the no-device path."""
import pytest

from roofline_gb300 import build, gemm


@pytest.fixture(scope="module")
def lib():
    build.build()
    return gemm.load()


@pytest.mark.parametrize("args", [
    dict(M=-1), dict(N=-2), dict(K=-3),
    dict(lda=3), dict(ldb=5), dict(ldc=5),
    dict(blocks=-1), dict(blocks=gemm.HOST_MAX_BLOCKS + 1),
    dict(mode=99),
])
def test_invalid_arguments(lib, args):
    a = dict(M=8, N=6, K=4, lda=4, ldb=6, ldc=6, blocks=0, mode=gemm.MODE_AUTO)
    a.update(args)
    rc = gemm.gemm_f32_host(a["M"], a["N"], a["K"], 1.0, 256, a["lda"], 256, a["ldb"], 0.0, 256,
                            a["ldc"], a["mode"], a["blocks"])
    assert rc == gemm.ERR_INVALID_ARG


def test_null_pointers(lib):
    assert gemm.gemm_f32_host(8, 6, 4, 1.0, None, 4, 256, 6, 0.0, 256, 6, 0, 0) == \
        gemm.ERR_INVALID_ARG
    assert gemm.gemm_f32_host(8, 6, 4, 1.0, 256, 4, None, 6, 0.0, 256, 6, 0, 0) == \
        gemm.ERR_INVALID_ARG
    assert gemm.gemm_f32_host(8, 6, 4, 1.0, 256, 4, 256, 6, 0.0, None, 6, 0, 0) == \
        gemm.ERR_INVALID_ARG


def test_empty_and_no_device(lib):
    import torch
    assert gemm.gemm_f32_host(0, 6, 4, 1.0, None, 4, None, 6, 0.0, None, 6, 0, 0) == gemm.OK
    assert gemm.gemm_f32_host(8, 0, 4, 1.0, None, 4, None, 1, 0.0, None, 1, 0, 0) == gemm.OK
    if not torch.cuda.is_available():
        assert gemm.gemm_f32_host(8, 6, 4, 1.0, 256, 4, 256, 6, 0.0, 256, 6, 0, 3) == \
            gemm.ERR_NO_DEVICE


def test_matmul_host_rejects_device_or_strided_tensors(lib):
    import torch
    A = torch.zeros(4, 8)
    with pytest.raises(ValueError):
        gemm.matmul_host(A.t(), torch.zeros(4, 3))   # unit row stride
    with pytest.raises(ValueError):
        gemm.matmul_host(torch.zeros(4, 8, dtype=torch.float64), torch.zeros(8, 3))
    with pytest.raises(ValueError):
        gemm.matmul_host(A, torch.zeros(7, 3))       # inner dimensions differ
