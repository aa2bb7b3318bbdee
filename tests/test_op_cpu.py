"""Host-side checks of gemm_f32_op / gemm_f32_op_plan (no GPU needed): the
storage-order and op arguments, leading-dimension rules, and the row-major
problem each call is planned as."""
import itertools

import pytest

from roofline_gb300 import build, gemm

ROW, COL, N_, T_ = gemm.ROW_MAJOR, gemm.COL_MAJOR, gemm.OP_N, gemm.OP_T


@pytest.fixture(scope="module")
def lib():
    build.build()
    return gemm.load()


def test_bad_layout_or_op_rejected(lib):
    for layout, op_a, op_b in [(2, 0, 0), (-1, 0, 0), (0, 2, 0), (0, 0, -1), (1, 3, 1)]:
        rc = gemm.gemm_f32_op(layout, op_a, op_b, 4, 4, 4, 1.0, 256, 4, 256, 4, 0.0, 256, 4,
                              0, None, 0, 0)
        assert rc == gemm.ERR_INVALID_ARG
        with pytest.raises(gemm.GemmError):
            gemm.plan_op(layout, op_a, op_b, 4, 4, 4, 4, 4, 4)


# (layout, op_a, op_b, M, N, K) -> smallest legal (lda, ldb, ldc)
LD_CASES = [
    ((ROW, N_, N_, 8, 6, 4), (4, 6, 6)),
    ((ROW, T_, N_, 8, 6, 4), (8, 6, 6)),
    ((ROW, N_, T_, 8, 6, 4), (4, 4, 6)),
    ((ROW, T_, T_, 8, 6, 4), (8, 4, 6)),
    ((COL, N_, N_, 8, 6, 4), (8, 4, 8)),
    ((COL, T_, N_, 8, 6, 4), (4, 4, 8)),
    ((COL, N_, T_, 8, 6, 4), (8, 6, 8)),
    ((COL, T_, T_, 8, 6, 4), (4, 6, 8)),
]


@pytest.mark.parametrize("case,lds", LD_CASES)
def test_leading_dimension_rules(lib, case, lds):
    layout, op_a, op_b, M, N, K = case
    assert gemm.stored_shape(layout, op_a, M, K)[1] == lds[0]
    assert gemm.stored_shape(layout, op_b, K, N)[1] == lds[1]
    assert gemm.stored_shape(layout, N_, M, N)[1] == lds[2]
    gemm.plan_op(layout, op_a, op_b, M, N, K, *lds, mode="fp32_simt")
    for i in range(3):
        bad = list(lds)
        bad[i] -= 1
        with pytest.raises(gemm.GemmError) as e:
            gemm.plan_op(layout, op_a, op_b, M, N, K, *bad, mode="fp32_simt")
        assert e.value.code == gemm.ERR_INVALID_ARG
        rc = gemm.gemm_f32_op(layout, op_a, op_b, M, N, K, 1.0, 256, bad[0], 256, bad[1], 0.0,
                              256, bad[2], 1, None, 0, 0)
        assert rc == gemm.ERR_INVALID_ARG


@pytest.mark.parametrize("mode", ["fp32_simt", "tf32x3", "tf32", "auto"])
@pytest.mark.parametrize("shape", [(4096, 4096, 4096), (1023, 515, 777), (65536, 64, 4096)])
def test_plain_row_major_plans_equal_gemm_f32_plan(lib, mode, shape):
    M, N, K = shape
    assert gemm.plan_op(ROW, N_, N_, M, N, K, mode=mode) == gemm.plan(M, N, K, mode=mode)


@pytest.mark.parametrize("mode", ["fp32_simt", "tf32x3", "auto"])
@pytest.mark.parametrize("shape", [(4096, 2048, 1024), (1023, 515, 777), (64, 65536, 4096)])
def test_column_major_is_the_transposed_row_major_problem(lib, mode, shape):
    M, N, K = shape
    # column-major A*B = row-major (B^T A^T)^T: an N x M problem
    assert gemm.plan_op(COL, N_, N_, M, N, K, mode=mode) == \
        gemm.plan(N, M, K, K, M, M, mode=mode)


def test_transposed_a_uses_the_pre_split(lib):
    p = gemm.plan_op(ROW, T_, N_, 4096, 4096, 4096, mode="tf32x3")
    assert p["kernel_name"] == "tc_tf32x3" and p["a_split_in_kernel"] == 0
    assert p["launches"] == 2 + p["stream_k"]
    assert p["b_split_in_kernel"] == 0  # B stored K x N: the transposing pass
    # B stored N x K at this size (stream-K): still one split pass for B, A
    # split on chip
    q = gemm.plan_op(ROW, N_, T_, 4096, 4096, 4096, mode="tf32x3")
    assert q["a_split_in_kernel"] == 1 and q["b_split_in_kernel"] == 0
    assert q["launches"] == 2 + q["stream_k"]
    # the tensor-core workspace then also holds A_hi / A_lo
    assert p["workspace_bytes"] >= q["workspace_bytes"] + 2 * 4096 * 4096 * 4


@pytest.mark.parametrize("mode", ["naive", "coalesced", "tiled16", "tiled32"])
def test_teaching_kernels_take_plain_operands_only(lib, mode):
    assert gemm.plan_op(ROW, N_, N_, 64, 64, 64, mode=mode)["kernel"] > 0
    for layout, op_a, op_b in itertools.product([ROW, COL], [N_, T_], [N_, T_]):
        if layout == ROW and op_a == N_ and op_b == N_:
            continue
        plain_colmajor = layout == COL and op_a == N_ and op_b == N_
        if plain_colmajor:
            # column-major with no ops is a plain row-major problem again
            assert gemm.plan_op(layout, op_a, op_b, 64, 64, 64, mode=mode)["kernel"] > 0
            continue
        with pytest.raises(gemm.GemmError) as e:
            gemm.plan_op(layout, op_a, op_b, 64, 64, 64, mode=mode)
        assert e.value.code == gemm.ERR_UNSUPPORTED


def test_empty_and_no_device(lib):
    import torch
    assert gemm.gemm_f32_op(COL, T_, T_, 0, 5, 5, 1.0, None, 5, None, 5, 0.0, None, 1, 0,
                            None, 0, 0) == gemm.OK
    if not torch.cuda.is_available():
        rc = gemm.gemm_f32_op(COL, T_, N_, 4, 4, 4, 1.0, 256, 4, 256, 4, 0.0, 256, 4, 1,
                              None, 0, 0)
        assert rc == gemm.ERR_NO_DEVICE


class _View:
    """Shape and strides of a 2-D float32 CUDA tensor, for the binding's
    operand classification (no device needed)."""

    def __init__(self, shape, strides):
        import torch
        self.shape, self._strides = shape, strides
        self.is_cuda, self.dtype = True, torch.float32

    def stride(self, i):
        return self._strides[i]

    def dim(self):
        return 2


@pytest.mark.parametrize("shape,strides,want", [
    ((5, 7), (7, 1), (gemm.OP_N, 7)),       # row-major rows of 7
    ((5, 7), (9, 1), (gemm.OP_N, 9)),       # row slice of a wider buffer
    ((7, 5), (1, 7), (gemm.OP_T, 7)),       # transposed view X.t()
    ((1, 449), (1, 1), (gemm.OP_N, 449)),   # one row: its row stride is never used
    ((1, 449), (3, 1), (gemm.OP_N, 449)),
    ((449, 1), (1, 1), (gemm.OP_N, 1)),     # one column
    ((449, 1), (1, 3), (gemm.OP_N, 1)),
    ((1, 1), (1, 1), (gemm.OP_N, 1)),
])
def test_operand_leading_dimension(shape, strides, want):
    assert gemm._operand(_View(shape, strides), "X") == want



def test_b_stored_n_by_k_split_on_chip_for_one_wave(lib):
    # B stored N x K is split on chip when the tiles fit one wave without
    # stream-K (measured on GB300: 1200 x 640 x 336 13.0 -> 10.5 us, 2048^3
    # 68.5 -> 65.8 us); longer runs of full tiles keep the pass (8192^3)
    for shape in [(2048, 2048, 2048), (1200, 640, 336)]:
        q = gemm.plan_op(ROW, N_, T_, *shape, mode="tf32x3")
        assert (q["a_split_in_kernel"], q["b_split_in_kernel"], q["launches"]) == (1, 1, 1)
        assert q["workspace_bytes"] == 0
    assert gemm.plan_op(ROW, N_, T_, 8192, 8192, 8192, mode="tf32x3")["b_split_in_kernel"] == 0
    # small products: A split on chip too, so the call is one launch
    for shape in [(512, 512, 512), (1024, 1024, 1024)]:
        q = gemm.plan_op(ROW, N_, T_, *shape, mode="tf32x3")
        assert (q["bn"], q["stages"], q["a_split_in_kernel"], q["b_split_in_kernel"],
                q["launches"]) == (64, 6, 1, 1, 1)
    # B stored K x N always goes through the transposing pass
    assert gemm.plan_op(ROW, N_, N_, 2048, 2048, 2048, mode="tf32x3")["b_split_in_kernel"] == 0
    # ldb not a multiple of 4: no TMA of B as stored
    assert gemm.plan_op(ROW, N_, T_, 2048, 2048, 2047, mode="tf32x3")["b_split_in_kernel"] == 0


def test_b_split_plan_invariants_random(lib):
    # Over random shapes, leading dimensions, storage orders and alignments,
    # a plan that splits B on chip only does so where the kernel can: B read
    # by TMA (ldb a multiple of 4, 16-byte aligned pointers), B stored N x K
    # or the 64 x 32 small-product tiles with A split on chip as well, one
    # wave of whole tiles (no stream-K); such a plan keeps no B planes, and
    # with A also split on chip it is one launch.
    import random
    rng = random.Random(2024)
    seen = {0: 0, 1: 0}
    for _ in range(600):
        M, N, K = (rng.choice([rng.randint(128, 4096), rng.randint(128, 1200),
                               rng.randint(128, 700)]) for _ in range(3))
        op_b = rng.choice([N_, T_])
        ldb_min = K if op_b == T_ else N
        ldb = ldb_min + rng.choice([0, 0, 1, 3, 4])
        lda = K + rng.choice([0, 0, 1, 4])
        align = rng.choice([0, 0, 0, 4])
        mode = rng.choice(["tf32x3", "tf32x3", "tf32", "auto"])
        p = gemm.plan_op(ROW, N_, op_b, M, N, K, lda=lda, ldb=ldb, mode=mode, align_hint=align)
        if p["kernel_name"] not in ("tc_tf32x3", "tc_tf32"):
            continue
        seen[p["b_split_in_kernel"]] += 1
        if not p["b_split_in_kernel"]:
            continue
        assert ldb % 4 == 0 and align % 16 == 0
        assert p["kernel_name"] == "tc_tf32x3"
        assert op_b == T_ or (p["bn"], p["bk"], p["a_split_in_kernel"]) == (64, 32, 1)
        assert p["stream_k"] == 0 and p["grid_ctas"] <= 152 * p["ctas_per_sm"]
        if p["a_split_in_kernel"]:
            assert p["launches"] == 1 and p["workspace_bytes"] == 0
        else:
            assert p["launches"] == 2
            assert p["workspace_bytes"] < 2 * N * (-(-K // 32) * 32) * 4 + 2 * M * (-(-K // 32) * 32) * 4
    # both forms occur in the sample
    assert seen[0] > 50 and seen[1] > 10, seen
