"""GPU parity: the CUDA path through the C ABI against the CPU oracle."""
import ctypes
import functools

import numpy as np
import pytest

import oracle
from tests import gpu_util
from tests.gpu_util import TOL_E1, tol_tf32
from workloads import WORKLOADS, matrix

pytestmark = pytest.mark.gpu

SMALL = ["sq512", "sq512_int", "ragged"]
LARGE = ["sq4096", "sq8192", "skinny"]
LADDER = ["naive", "coalesced", "tiled16", "tiled32"]


def _check(name, mode):
    C = gpu_util.run(name, mode)
    r = gpu_util.compare(name, C)
    w = WORKLOADS[name]
    if w.a_dist == "int2":
        assert r["mismatches"] == 0, r
    else:
        assert r["e1"] <= TOL_E1, r
    # leading-dimension padding of C is never written
    lda, ldb, ldc = w.lds()
    if ldc > w.N:
        assert np.all(np.isnan(C[:, w.N:]))
    return r


@pytest.mark.parametrize("name", SMALL)
@pytest.mark.parametrize("mode", ["fp32_simt", "tf32x3", "auto"] + LADDER)
def test_small_configs(name, mode):
    _check(name, mode)


@pytest.mark.parametrize("name", LARGE)
@pytest.mark.parametrize("mode", ["fp32_simt", "tf32x3", "auto"])
def test_large_configs_sampled(name, mode):
    _check(name, mode)


def test_int_config_bit_exact_and_deterministic():
    outs = gpu_util.run("sq512_int", "fp32_simt", repeat=3)
    for o in outs[1:]:
        assert np.array_equal(o.view(np.uint32), outs[0].view(np.uint32))
    assert gpu_util.compare("sq512_int", outs[0])["mismatches"] == 0


@pytest.mark.parametrize("mode", ["fp32_simt", "tf32x3", "auto"])
def test_real_config_deterministic(mode):
    outs = gpu_util.run("ragged", mode, repeat=2)
    assert np.array_equal(outs[0].view(np.uint32), outs[1].view(np.uint32))


EDGE_SHAPES = [(1, 1, 1), (2, 3, 5), (17, 31, 33), (33, 17, 1), (127, 129, 64),
               (129, 127, 255), (64, 64, 7), (1, 300, 257), (300, 1, 129), (255, 257, 1000),
               (513, 65, 129), (1000, 3, 77)]


def _run_shape(M, N, K, mode, alpha, beta, pad=(0, 0, 0), offset=0, seed=0, dist="u11",
               sampled=False):
    """Runs one GEMM with guard bands checked; returns (C, C_ref, D), or with
    ``sampled`` ({"C": C, "inputs": (A, B, C_old)}, None, None) for the
    caller to check sampled entries."""
    import torch
    from roofline_gb300 import gemm
    lda, ldb, ldc = K + pad[0], N + pad[1], N + pad[2]
    A = matrix(M, K, lda, 7000 + seed, dist)
    B = matrix(K, N, ldb, 7100 + seed, dist)
    C0 = matrix(M, N, ldc, 7200 + seed, "u11")
    # device buffers with an `offset`-float shift (misaligned when offset % 4 != 0)
    # and a guard band of sentinel rows around C
    sentinel = 12345.0

    def dev(arr):
        flat = torch.full((arr.size + offset + 64,), sentinel, dtype=torch.float32, device="cuda")
        flat[offset:offset + arr.size] = torch.from_numpy(arr.reshape(-1)).cuda()
        return flat, flat[offset:offset + arr.size].view(arr.shape)

    fA, dA = dev(A)
    fB, dB = dev(B)
    cbuf = np.full((M + 2, ldc), sentinel, dtype=np.float32)
    cbuf[1:M + 1] = C0
    fC, dC = dev(cbuf)
    gemm.matmul(dA[:, :K], dB[:, :N], dC[1:M + 1, :N], alpha, beta, mode)
    torch.cuda.synchronize()
    out = fC.cpu().numpy()
    full = out[offset:offset + cbuf.size].reshape(cbuf.shape)
    # guard bands: rows above/below, padding columns, and the tail of the buffer
    assert np.all(full[0] == sentinel) and np.all(full[M + 1] == sentinel)
    if ldc > N:
        assert np.all(np.isnan(full[1:M + 1, N:]) | (full[1:M + 1, N:] == sentinel))
        assert np.array_equal(np.isnan(full[1:M + 1, N:]), np.isnan(C0[:, N:]))
    assert np.all(out[offset + cbuf.size:] == sentinel)
    assert np.all(out[:offset] == sentinel)
    if sampled:
        return {"C": full[1:M + 1, :N], "inputs": (A[:, :K], B[:, :N], C0[:, :N])}, None, None
    ref, D = oracle.gemm(A[:, :K], B[:, :N], alpha, beta, C0[:, :N], with_bound=True)
    return full[1:M + 1, :N], ref, D


@pytest.mark.parametrize("shape", EDGE_SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("mode", ["fp32_simt", "tf32x3", "tiled32", "auto"])
def test_edge_shapes(shape, mode):
    M, N, K = shape
    got, ref, D = _run_shape(M, N, K, mode, 1.25, -0.5, pad=(3, 1, 2), offset=1, seed=M + N + K)
    assert oracle.err_normalised(got, ref, D) <= TOL_E1


@pytest.mark.parametrize("shape", [(64, 64, 64), (130, 260, 100), (256, 512, 1024),
                                   (384, 48, 520), (1000, 64, 96)])
@pytest.mark.parametrize("offset", [0, 1, 2])
@pytest.mark.parametrize("mode", ["fp32_simt", "tf32x3"])
def test_alignment_paths_integer_exact(shape, offset, mode):
    M, N, K = shape
    got, ref, D = _run_shape(M, N, K, mode, 1.0, 0.0, pad=(0, 0, 0), offset=offset,
                             seed=offset, dist="int2")
    assert oracle.mismatches(got, ref) == 0


@pytest.mark.parametrize("shape", [(1000, 64, 96), (513, 33, 1000), (256, 64, 4096),
                                   (129, 17, 40)])
def test_tf32x3_split_in_kernel(shape):
    """N <= 64 with an aligned A takes the path that splits A inside the GEMM."""
    from roofline_gb300 import gemm
    M, N, K = shape
    p = gemm.plan(M, N, K, K, N, N, mode="tf32x3")
    assert p["a_split_in_kernel"] == (1 if K % 4 == 0 else 0)
    got, ref, D = _run_shape(M, N, K, "tf32x3", 0.75, 0.25, pad=(0, 0, 0), offset=0, seed=K)
    assert oracle.err_normalised(got, ref, D) <= TOL_E1


def test_beta_zero_does_not_read_c():
    import torch
    from roofline_gb300 import gemm
    A = torch.from_numpy(matrix(96, 80, None, 1, "u11")).cuda()
    B = torch.from_numpy(matrix(80, 72, None, 2, "u11")).cuda()
    for mode in ["fp32_simt", "tf32x3", "auto", "tiled16"]:
        C = torch.full((96, 72), float("nan"), device="cuda")
        gemm.matmul(A, B, C, 1.0, 0.0, mode)
        torch.cuda.synchronize()
        assert torch.isfinite(C).all()


def test_k_zero_scales_c():
    import torch
    from roofline_gb300 import gemm
    C0 = torch.from_numpy(matrix(33, 45, None, 3, "u11")).cuda()
    A = torch.empty((33, 0), device="cuda")
    B = torch.empty((0, 45), device="cuda")
    C = C0.clone()
    gemm.matmul(A, B, C, 2.0, 0.5, "auto")
    torch.cuda.synchronize()
    assert torch.equal(C, C0 * 0.5)
    C = C0.clone()
    gemm.matmul(A, B, C, 2.0, 0.0, "auto")
    torch.cuda.synchronize()
    assert torch.equal(C, torch.zeros_like(C))


def test_workspace_paths():
    import torch
    from roofline_gb300 import gemm
    p = gemm.plan(512, 512, 512, mode="fp32_simt")
    assert p["split_k"] > 1 and p["workspace_bytes"] > 0
    A, B, _ = gpu_util.inputs("sq512")
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    small = torch.empty(p["workspace_bytes"] // 2, dtype=torch.uint8, device="cuda")
    C = torch.empty((512, 512), device="cuda")
    with pytest.raises(gemm.GemmError) as ei:
        gemm.matmul(dA, dB, C, mode="fp32_simt", workspace=small)
    assert ei.value.code == gemm.ERR_WORKSPACE_TOO_SMALL
    ws = torch.empty(p["workspace_bytes"], dtype=torch.uint8, device="cuda")
    gemm.matmul(dA, dB, C, mode="fp32_simt", workspace=ws)
    torch.cuda.synchronize()
    r = gpu_util.compare("sq512", C.cpu().numpy())
    assert r["e1"] <= TOL_E1


def test_device_info_from_device():
    from roofline_gb300 import gemm
    d = gemm.device_info(0)
    assert d["from_device"] == 1 and d["sm_count"] > 100 and d["cc_major"] == 10
    assert d["fp32_peak_tflops"] > 50


def test_copy_kernel_exact():
    import torch
    from roofline_gb300 import gemm
    n = 1_000_003
    src = torch.randn(n + 8, device="cuda")
    for off in [0, 1, 3]:
        dst = torch.zeros(n + 8, device="cuda")
        gemm.hbm_copy(src[off:off + n], dst[off:off + n])
        torch.cuda.synchronize()
        assert torch.equal(dst[off:off + n], src[off:off + n])
        assert torch.all(dst[:off] == 0) and torch.all(dst[off + n:] == 0)


def test_copy_calibration_runs():
    import torch
    from roofline_gb300 import gemm
    n = 64 << 20
    src = torch.ones(n, device="cuda")
    dst = torch.empty(n, device="cuda")
    gbs = gemm.hbm_copy_calibrate(src, dst, iters=5)
    assert 500.0 < gbs < 20000.0
    assert torch.equal(dst, src)


def test_status_clear_after_normal_runs():
    from roofline_gb300 import gemm
    assert gemm.check_status() == gemm.OK


# The planner's own choice for representative shapes:
# (M, N, K, lda) -> (bn, bk, stages, A split in kernel, concatenated B)
TC_PLANS = [
    ((1000, 64, 96, 96), (128, 64, 32, 6, 1, 1, 0)),       # narrow, few tiles: 6 stages, 1 CTA/SM
    ((9000, 64, 96, 96), (128, 64, 32, 3, 1, 1, 0)),       # narrow, more tiles: 3 stages, 2 CTAs/SM
    ((512, 512, 512, 512), (128, 64, 32, 6, 1, 1, 1)),     # small product: a CTA per 128 x 64 tile,
                                                           # A and B split on chip, one launch
    ((512, 512, 1024, 1024), (128, 128, 32, 4, 1, 1, 0)),   # few tiles, longer K: stream-K
    ((2432, 8192, 128, 128), (128, 256, 16, 5, 1, 0, 0)),
    ((1023, 1025, 777, 777), (128, 64, 32, 4, 0, 1, 0)),    # small product, A and B pre-split
    ((1200, 640, 336, 336), (128, 64, 32, 6, 1, 1, 1)),    # shallow small product: one launch
    ((600, 600, 3000, 3001), (128, 128, 16, 6, 0, 1, 0)),   # A pre-split, under half a wave: 6 stages
    ((5000, 250, 777, 777), (128, 128, 16, 3, 0, 1, 0)),    # A pre-split, more tiles: 3 stages, 2 CTAs/SM
    ((2432, 8192, 129, 129), (128, 256, 16, 4, 0, 0, 0)),
    ((5120, 8192, 64, 64), (128, 256, 16, 5, 1, 0, 0)),   # many tiles, aligned A: split on chip
    ((5120, 8192, 65, 65), (256, 256, 16, 3, 0, 0, 0)),   # many tiles, A pre-split: 256 x 256
]


@pytest.mark.parametrize("shape,cfg", TC_PLANS, ids=lambda v: "x".join(map(str, v)))
def test_tf32x3_planner_choices(shape, cfg):
    import torch
    from roofline_gb300 import gemm
    from workloads import sample_entries
    M, N, K, lda = shape
    p = gemm.plan(M, N, K, lda, N, N, mode="tf32x3")
    assert (p["bm"], p["bn"], p["bk"], p["stages"], p["a_split_in_kernel"], p["b_concat"],
            p["b_split_in_kernel"]) == cfg
    assert p["ctas_per_sm"] >= 1
    A = matrix(M, K, lda, 4000 + K, "u11")
    B = matrix(K, N, None, 4100 + K, "u11")
    C0 = matrix(M, N, None, 4200 + K, "u11")
    dA, dB, dC = (torch.from_numpy(x).cuda() for x in (A, B, C0))
    gemm.matmul(dA[:, :K], dB, dC, 0.5, -1.5, "tf32x3")
    torch.cuda.synchronize()
    got = dC.cpu().numpy()
    rows, cols = sample_entries(M, N, 2048, seed=K)
    ref, D = oracle.gemm_entries(A[:, :K], B, rows, cols, 0.5, -1.5, C0)
    assert oracle.err_normalised(got[rows, cols], ref, D) <= TOL_E1


# Every tensor-core configuration the library is built with, forced through
# the GEMM_TC_CONFIG knob, on one ragged shape (full check).
TC_BUILT = ["256,16,5,1,0", "128,32,4,1,1", "64,32,6,1,1", "64,32,3,1,1", "64,32,2,1,0",
            "64,16,4,1,0", "256,16,4,0,0", "128,16,3,0,1", "128,16,6,0,1", "256,256,16,3,0,0",
            "256,16,5,2,0", "128,32,4,2,1", "64,16,6,0,1", "64,32,4,0,1"]


def _cfg(cfg):
    """(bm, bn, bk, stages, a_split_in_kernel, b_concat) of a GEMM_TC_CONFIG string."""
    v = list(map(int, cfg.split(",")))
    return tuple(v) if len(v) == 6 else (128, *v)


@pytest.mark.parametrize("cfg", TC_BUILT)
def test_tf32x3_every_built_configuration(cfg, monkeypatch):
    from roofline_gb300 import gemm
    bm, bn, bk, st, ak, cc = _cfg(cfg)
    monkeypatch.setenv("GEMM_TC_CONFIG", cfg)
    M, N, K = 777, 200, 300
    pad = (0 if ak else 1, 0, 0)
    p = gemm.plan(M, N, K, K + pad[0], N, N, mode="tf32x3")
    assert (p["bm"], p["bn"], p["bk"], p["stages"], p["a_split_in_kernel"], p["b_concat"]) == \
        (bm, bn, bk, st, min(ak, 1), cc)
    assert p["a_hi_tmem"] == (1 if ak == 2 else 0)
    got, ref, D = _run_shape(M, N, K, "tf32x3", 1.5, 0.5, pad=pad, offset=0, seed=st + bn)
    assert oracle.err_normalised(got, ref, D) <= TOL_E1


@pytest.mark.parametrize("split", [1, 2, 3, 7, 16])
def test_simt_forced_splits(split, monkeypatch):
    from roofline_gb300 import gemm
    monkeypatch.setenv("GEMM_SIMT_SPLIT", str(split))
    M, N, K = 300, 260, 1000
    p = gemm.plan(M, N, K, K + 1, N, N + 2, mode="fp32_simt")
    assert p["split_k"] == min(split, -(-K // (-(-(-(-K // split)) // 16) * 16)))
    got, ref, D = _run_shape(M, N, K, "fp32_simt", 0.75, 1.25, pad=(1, 0, 2), offset=1,
                             seed=split)
    assert oracle.err_normalised(got, ref, D) <= TOL_E1


@pytest.mark.parametrize("shape", [(1000, 64, 96), (777, 200, 300), (300, 520, 64), (2100, 900, 1000),
                                   (129, 300, 4000)])
@pytest.mark.parametrize("streamk", ["0", "1"])
def test_tf32x3_stream_k(shape, streamk, monkeypatch):
    """Persistent stream-K scheduling (tiles split between CTAs, summed by the
    fix-up kernel) against one CTA per tile, with aligned and unaligned A."""
    from roofline_gb300 import gemm
    monkeypatch.setenv("GEMM_TC_STREAMK", streamk)
    M, N, K = shape
    for pad in (0, 1):
        p = gemm.plan(M, N, K, K + pad, N, N, mode="tf32x3")
        if streamk == "0":
            assert p["stream_k"] == 0
        else:
            assert p["stream_k"] == 1 and p["grid_ctas"] >= 2
        got, ref, D = _run_shape(M, N, K, "tf32x3", -1.25, 0.5, pad=(pad, 0, 0), offset=0,
                                 seed=M + pad)
        assert oracle.err_normalised(got, ref, D) <= TOL_E1


@pytest.mark.parametrize("cfg", ["64,32,4,0,1", "64,16,6,0,1"])
@pytest.mark.parametrize("streamk", ["0", "1"])
@pytest.mark.parametrize("shape,pad", [((300, 200, 1000), (1, 0, 1)), ((777, 130, 64), (0, 0, 0)),
                                       ((129, 1025, 777), (1, 1, 3))])
def test_old_c_through_tensor_memory(cfg, streamk, shape, pad, monkeypatch):
    """Pre-split 128 x 64 tiles copy C's old values into tensor memory while
    the MMAs run and fold beta * C in at the epilogue; tiles shared out
    stream-K take C through the fix-up instead.  Both against the oracle with
    beta != 0, unaligned and aligned ldc, ragged edges; beta == 0 must leave
    C unread (NaN in C stays out of the result)."""
    from roofline_gb300 import gemm
    monkeypatch.setenv("GEMM_TC_CONFIG", cfg)
    monkeypatch.setenv("GEMM_TC_STREAMK", streamk)
    M, N, K = shape
    p = gemm.plan(M, N, K, K + pad[0], N + pad[1], N + pad[2], mode="tf32x3")
    assert (p["bm"], p["bn"], p["a_split_in_kernel"], p["b_concat"]) == (128, 64, 0, 1)
    for alpha, beta in ((1.5, -0.75), (-1.0, 2.0)):
        got, ref, D = _run_shape(M, N, K, "tf32x3", alpha, beta, pad=pad, offset=0,
                                 seed=M + N + int(streamk))
        assert oracle.err_normalised(got, ref, D) <= TOL_E1
    import torch
    A = torch.from_numpy(matrix(M, K, None, 5, "u11")).cuda()
    B = torch.from_numpy(matrix(K, N, None, 6, "u11")).cuda()
    C = torch.full((M, N), float("nan"), device="cuda")
    gemm.matmul(A, B, C, 1.0, 0.0, "tf32x3")
    torch.cuda.synchronize()
    assert torch.isfinite(C).all()


def test_tf32x3_stream_k_deterministic():
    outs = gpu_util.run("ragged", "tf32x3", repeat=3)
    for o in outs[1:]:
        assert np.array_equal(o.view(np.uint32), outs[0].view(np.uint32))


@pytest.mark.parametrize("cfg", [None, "256,256,16,3,0,0"])
@pytest.mark.parametrize("shape", [(129, 300, 4000), (2100, 900, 1000)])
def test_stream_k_parts_summed_in_cta_order(cfg, shape, monkeypatch):
    """Tiles shared by many CTAs (up to ~40 parts a tile for 129 x 300 x 4000):
    the fix-up sums a tile's parts in CTA order, so repeated calls agree to
    the bit; integer inputs are exact."""
    import torch
    from roofline_gb300 import gemm
    from workloads import matrix
    monkeypatch.setenv("GEMM_TC_STREAMK", "1")
    if cfg:
        monkeypatch.setenv("GEMM_TC_CONFIG", cfg)
    M, N, K = shape
    pad = 1 if cfg else 0  # the 256-row configuration takes a pre-split A
    p = gemm.plan(M, N, K, K + pad, N, N, mode="tf32x3")
    assert p["stream_k"] == 1 and p["grid_ctas"] >= 2
    for dist, seed in (("u11", 5), ("int2", 6)):
        A = matrix(M, K, K + pad, seed, dist)
        B = matrix(K, N, None, seed + 1, dist)
        C0 = matrix(M, N, None, seed + 2, dist)
        dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
        outs = []
        for _ in range(4):
            dC = torch.from_numpy(C0).cuda()
            gemm.matmul(dA[:, :K], dB, dC, 1.0, 1.0 if dist == "int2" else 0.5, "tf32x3")
            outs.append(dC.cpu().numpy())
        for o in outs[1:]:
            assert np.array_equal(o.view(np.uint32), outs[0].view(np.uint32))
        if dist == "int2":
            assert oracle.mismatches(outs[0], oracle.gemm(A[:, :K], B, 1.0, 1.0, C0)) == 0
        else:
            ref, D = oracle.gemm(A[:, :K], B, 1.0, 0.5, C0, with_bound=True)
            assert oracle.err_normalised(outs[0], ref, D) <= TOL_E1
    assert gemm.check_status() == gemm.OK


def test_fma_peak_probe():
    from roofline_gb300 import gemm
    d = gemm.device_info(0)
    for packed in (False, True):
        tf = gemm.fp32_fma_peak(1 << 14, packed)
        # the probe cannot beat the derived peak by more than clock noise
        assert 0.2 * d["fp32_peak_tflops"] < tf < 1.05 * d["fp32_peak_tflops"], (packed, tf)


def _fma_chain_expected(iters, packed):
    """What the FMA probe's sink must hold for each of its 256 threads, from
    the chains the probe runs ("Bandwidths and peak rate - exercises",
    exercise 5: acc = acc * x + y, several independent chains per thread,
    result written out): every fmaf taken exactly in rationals and rounded
    once to float32 (an FMA rounds once), then the per-thread sum in float32
    in the kernel's order.  x, y and the starting values are the probe's."""
    from fractions import Fraction

    from oracle.exact import round_to_f32
    x, y = np.float32(0.999999), np.float32(1e-6)
    fx, fy = Fraction(float(x)), Fraction(float(y))
    chains = 8

    @functools.lru_cache(maxsize=None)
    def chain(v0):
        a = np.float32(v0)
        for _ in range(iters):
            a = round_to_f32(Fraction(float(a)) * fx + fy)
        return a

    out = np.empty(256, dtype=np.float32)
    for t in range(256):
        s = np.float32(0.0)
        for c in range(chains):
            if packed:  # lanes start at (t, c); s += lane0 + lane1
                s = np.float32(s + np.float32(chain(t) + chain(c)))
            else:  # chain c starts at t + c
                s = np.float32(s + chain(t + c))
        out[t] = s
    return out


@pytest.mark.parametrize("packed", [False, True])
def test_fma_peak_probe_does_the_counted_work(packed):
    # The probe reports FLOP = threads x iterations x chains x 2 (x2 packed);
    # its sink must hold exactly the value those chains define, so a probe
    # that skipped or shortened its loop (and so overstated its FLOP/s)
    # fails here.  Bit for bit: each fmaf is rounded once, as IEEE requires.
    import torch

    from roofline_gb300 import gemm
    iters = 64
    lib = gemm.load()
    n = lib.fp32_fma_peak_sink_floats()
    sink = torch.full((n,), float("nan"), dtype=torch.float32, device="cuda")
    out = ctypes.c_double(0.0)
    rc = lib.fp32_fma_peak(iters, 1 if packed else 0, sink.data_ptr(),
                           torch.cuda.current_stream().cuda_stream, ctypes.byref(out))
    assert rc == gemm.OK
    torch.cuda.synchronize()
    got = sink.cpu().numpy().reshape(-1, 256)
    want = _fma_chain_expected(iters, packed)
    assert got.shape[0] == lib.fp32_fma_peak_sink_floats() // 256
    assert np.array_equal(got, np.broadcast_to(want, got.shape))
    # a chain that ran fewer iterations would hold another value
    assert not np.array_equal(want, _fma_chain_expected(iters - 1, packed))




TF32_BUILT = ["256,16,8,1,0", "64,32,4,1,0", "256,16,8,0,0", "256,256,16,6,0,0",
              "256,256,32,3,0,0"]


@pytest.mark.parametrize("cfg", TF32_BUILT)
@pytest.mark.parametrize("streamk", ["0", "1"])
def test_tf32_mode_every_configuration(cfg, streamk, monkeypatch):
    from roofline_gb300 import gemm
    bm, bn, bk, st, ak, cc = _cfg(cfg)
    monkeypatch.setenv("GEMM_TC_CONFIG", cfg)
    monkeypatch.setenv("GEMM_TC_STREAMK", streamk)
    M, N, K = 777, 200, 300
    pad = (0 if ak else 1, 0, 0)
    p = gemm.plan(M, N, K, K + pad[0], N, N, mode="tf32")
    assert p["kernel_name"] == "tc_tf32"
    assert (p["bm"], p["bn"], p["bk"], p["stages"], p["a_split_in_kernel"]) == (bm, bn, bk, st, ak)
    got, ref, D = _run_shape(M, N, K, "tf32", 1.5, 0.5, pad=pad, offset=0, seed=st + bn)
    e1 = oracle.err_normalised(got, ref, D)
    assert e1 <= tol_tf32(K), e1
    # integer inputs are exact in TF32: bit-exact
    got, ref, D = _run_shape(M, N, K, "tf32", 1.0, 0.0, pad=pad, offset=0, seed=7, dist="int2")
    assert oracle.mismatches(got, ref) == 0


@pytest.mark.parametrize("name", ["sq512_int", "ragged", "sq4096", "skinny"])
def test_tf32_mode_workloads(name):
    C = gpu_util.run(name, "tf32")
    r = gpu_util.compare(name, C)
    if WORKLOADS[name].a_dist == "int2":
        assert r["mismatches"] == 0, r
    else:
        assert r["e1"] <= tol_tf32(WORKLOADS[name].K), r


def _waves(tiles, num_kb, G):
    """Whole-tile waves and stream-K tiles of the tensor-core work split."""
    waves, rest = tiles // G, tiles % G
    while rest > 0 and waves > 0 and (rest * num_kb < 4 * G or G > 250 * rest):
        waves, rest = waves - 1, rest + G
    return waves, rest


@pytest.mark.parametrize("order", ["0", "1", "g3", "g5", None])
@pytest.mark.parametrize("mode,cfg", [("tf32x3", None), ("tf32x3", "256,256,16,3,0,0"),
                                      ("tf32", "256,16,8,0,0"), ("tf32", "256,256,16,6,0,0")])
def test_tc_whole_waves_then_stream_k(mode, cfg, order, monkeypatch):
    # 168 tiles x 64 K blocks (2688 or 5376 rows, 2048 columns, K = 1024): one
    # wave of whole tiles, then a stream-K remainder whose partial tiles the
    # fix-up sums
    from roofline_gb300 import gemm
    from workloads import sample_entries
    if cfg:
        monkeypatch.setenv("GEMM_TC_CONFIG", cfg)
    monkeypatch.setenv("GEMM_TC_STREAMK", "1")
    # tiles numbered along rows (0), down columns (1), in bands of 3 or 5
    # column-tiles, or in the planner's bands (None)
    if order in ("0", "1"):
        monkeypatch.setenv("GEMM_TC_ORDER", order)
    elif order is not None:
        monkeypatch.setenv("GEMM_TC_GROUP", order[1:])
    M, N, K = 2688 * (2 if cfg and cfg.startswith("256,256") else 1), 2048, 1024
    p = gemm.plan(M, N, K, K, N, N, mode=mode)
    tiles = -(-M // p["bm"]) * -(-N // p["bn"])
    waves, rest = _waves(tiles, -(-K // p["bk"]), p["grid_ctas"])
    assert p["stream_k"] == 1 and waves >= 1 and rest > 0, (p, waves, rest)
    got_full, _, _ = _run_shape(M, N, K, mode, 0.75, 0.25, seed=31, sampled=True)
    A, B, C0 = got_full["inputs"]
    rows, cols = sample_entries(M, N, n=30000, seed=77)
    ref, D = oracle.gemm_entries(A, B, rows, cols, 0.75, 0.25, C0)
    tol = tol_tf32(K) if mode == "tf32" else TOL_E1
    assert oracle.err_normalised(got_full["C"][rows, cols], ref, D) <= tol


@pytest.mark.parametrize("mode,shape", [("fp32_simt", (512, 512, 512)), ("tf32x3", (1000, 520, 300)),
                                        ("tf32x3", (4096, 4096, 512)), ("tf32", (1024, 1024, 256))])
def test_calls_capture_into_a_cuda_graph(mode, shape):
    # with a caller workspace (no allocation inside the call) a GEMM can be
    # captured in a CUDA graph and replayed; every replay recomputes C
    import torch
    from roofline_gb300 import gemm
    M, N, K = shape
    A = torch.from_numpy(matrix(M, K, None, 61, "int2")).cuda()
    B = torch.from_numpy(matrix(K, N, None, 62, "int2")).cuda()
    C = torch.full((M, N), float("nan"), device="cuda")
    p = gemm.plan(M, N, K, mode=mode)
    ws = torch.empty(max(p["workspace_bytes"], 256), dtype=torch.uint8, device="cuda")
    gemm.matmul(A, B, C, mode=mode, workspace=ws)  # warm-up outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.graph(g, stream=s):
        gemm.matmul(A, B, C, mode=mode, workspace=ws)
    ref = oracle.gemm(A.cpu().numpy(), B.cpu().numpy(), 1.0, 0.0, None)
    for _ in range(3):
        C.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert oracle.mismatches(C.cpu().numpy(), ref) == 0


@functools.lru_cache(maxsize=1)
def _extreme_inputs(M, N, K):
    A = matrix(M, K, None, 91, "int2")
    B = matrix(K, N, None, 92, "int2")
    if K > (1 << 20):
        # keep |partial sums| below 2^24: entries in {-1, 0, 1}
        A = np.clip(A, -1, 1)
        B = np.clip(B, -1, 1)
    return A, B


EXTREME = [
    (1, 1, 1 << 22),          # one dot product of 4M terms (split K)
    (1 << 20, 1, 16),         # a million rows, one column
    (2, 1 << 20, 8),          # two rows, a million columns
    (128, 128, (65535 * 32) - 32),  # the longest K the tensor-core split passes take
]


@pytest.mark.parametrize("mode", ["auto", "fp32_simt", "tf32x3"])
@pytest.mark.parametrize("shape", EXTREME, ids=lambda s: "x".join(map(str, s)))
def test_extreme_shapes_sampled(shape, mode):
    # extreme aspect ratios and the longest K, integer inputs so every
    # sampled entry must equal the oracle exactly (|partial sums| < 2^24)
    import torch
    from roofline_gb300 import gemm
    from workloads import sample_entries
    M, N, K = shape
    try:
        gemm.plan(M, N, K, mode=mode)
    except gemm.GemmError as e:
        assert e.code == gemm.ERR_UNSUPPORTED
        pytest.skip("K beyond what the tensor-core split passes take")
    A, B = _extreme_inputs(M, N, K)
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    C = gemm.matmul(dA, dB, mode=mode)
    torch.cuda.synchronize()
    rows, cols = sample_entries(M, N, n=min(2048, M * N), seed=5)
    ref, _ = oracle.gemm_entries(A, B, rows, cols, 1.0, 0.0, None)
    got = C.cpu().numpy()[rows, cols]
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("mode", ["fp32_simt", "tf32x3", "tf32", "auto", "tiled16"])
@pytest.mark.parametrize("beta", [0.0, -1.5])
def test_alpha_zero_reads_neither_a_nor_b(mode, beta):
    """BLAS semantics of alpha == 0: A and B are not read (NaN and Inf there
    do not reach C) and C <- beta * C, bit for bit with the oracle."""
    import torch
    from roofline_gb300 import gemm
    M, N, K = 300, 200, 129
    A = np.full((M, K), np.nan, dtype=np.float32)
    B = np.full((K, N), np.inf, dtype=np.float32)
    C0 = matrix(M, N, None, 77, "u11")
    want = oracle.gemm(A, B, 0.0, beta, C0)
    dC = torch.from_numpy(C0.copy()).cuda()
    gemm.matmul(torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda(), dC, 0.0, beta, mode)
    torch.cuda.synchronize()
    assert np.array_equal(dC.cpu().numpy(), want)
    # host buffers, and the no-allocation split-K entry point
    hC = torch.from_numpy(C0.copy())
    gemm.matmul_host(torch.from_numpy(A), torch.from_numpy(B), hC, 0.0, beta, mode)
    assert np.array_equal(hC.numpy(), want)
    dC = torch.from_numpy(C0.copy()).cuda()
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    rc = gemm.gemm_f32_splitk_noalloc(M, N, K, 0.0, dA.data_ptr(), K, dB.data_ptr(), N, beta,
                                      dC.data_ptr(), N)
    torch.cuda.synchronize()
    assert rc == gemm.OK and np.array_equal(dC.cpu().numpy(), want)


@pytest.mark.parametrize("mode", ["fp32_simt", "tf32x3", "tf32", "auto"])
def test_non_finite_inputs(mode):
    """A NaN in A makes its row of C NaN in every mode.  An Inf in A gives the
    oracle's +-Inf row on the CUDA cores; the TF32 split modes give NaN there
    (tf32(Inf) = Inf, and the Inf meets a zero part of the other operand in a
    cross product, Inf * 0 = NaN).  Every other row stays within tolerance."""
    import torch
    from roofline_gb300 import gemm
    M, N, K = 260, 300, 200
    A = matrix(M, K, None, 81, "u11")
    B = matrix(K, N, None, 82, "u11")
    A[3, 17] = np.nan
    A[200, 5] = np.inf
    C = gemm.matmul(torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda(), mode=mode)
    torch.cuda.synchronize()
    got = C.cpu().numpy()
    ref = oracle.gemm(A, B)
    assert np.all(np.isnan(got[3]))
    if mode == "fp32_simt":
        assert np.array_equal(got[200], ref[200])  # +-Inf, signs from B
    else:
        assert np.all(~np.isfinite(got[200]))
    rest = np.ones(M, bool)
    rest[[3, 200]] = False
    Af = A[rest]
    ref_r, D = oracle.gemm(Af, B, with_bound=True)
    tol = 2e-3 if mode == "tf32" else TOL_E1
    assert oracle.err_normalised(got[rest], ref_r, D) <= tol


@pytest.mark.parametrize("mode,shape", [("tf32x3", (1000, 900, 700)), ("fp32_simt", (300, 260, 2000)),
                                        ("auto", (1023, 1025, 777))])
def test_concurrent_streams_with_own_workspaces(mode, shape):
    """Calls running at the same time on two streams, each with its own
    workspace (split planes, stream-K partial tiles, split-K slices), do not
    disturb each other: integer inputs give exact results on both."""
    import torch
    from roofline_gb300 import gemm
    M, N, K = shape
    p = gemm.plan(M, N, K, mode=mode)
    jobs = []
    for seed in (11, 12):
        A = matrix(M, K, None, seed, "int2")
        B = matrix(K, N, None, seed + 100, "int2")
        ws = torch.empty(max(p["workspace_bytes"], 256), dtype=torch.uint8, device="cuda")
        jobs.append((torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda(), ws,
                     oracle.gemm(A, B), torch.cuda.Stream()))
    torch.cuda.synchronize()
    outs = [[], []]
    for rep in range(6):
        for i, (dA, dB, ws, _, st) in enumerate(jobs):
            with torch.cuda.stream(st):
                C = torch.empty(M, N, device="cuda")
                gemm.matmul(dA, dB, C, 1.0, 0.0, mode, stream=st, workspace=ws)
                outs[i].append(C)
    torch.cuda.synchronize()
    for i in range(2):
        for C in outs[i]:
            assert oracle.mismatches(C.cpu().numpy(), jobs[i][3]) == 0
    assert gemm.check_status() == gemm.OK



@pytest.mark.parametrize("mode,shape", [("fp32_simt", (512, 512, 4096)),
                                        ("tf32x3", (1024, 1024, 1024)),
                                        ("tf32x3", (2688, 2048, 1024))])
def test_profile_stamps_time_the_main_kernel(mode, shape):
    # gemm_set_profile_stamps: the main kernel folds its CTAs' start and end
    # times into the caller's pair; one pair per call, results unchanged
    import torch

    from roofline_gb300 import gemm
    M, N, K = shape
    A = torch.from_numpy(matrix(M, K, None, 5, "u11")).cuda()
    B = torch.from_numpy(matrix(K, N, None, 6, "u11")).cuda()
    plain = gemm.matmul(A, B, mode=mode)
    st = torch.empty((3, 2), dtype=torch.int64, device="cuda")
    st[:, 0] = -1
    st[:, 1] = 0
    outs = []
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(2):
        gemm.set_profile_stamps(st[i])
        outs.append(gemm.matmul(A, B, mode=mode))
    gemm.set_profile_stamps(None)
    e1.record()
    torch.cuda.synchronize()
    v = st.cpu().numpy().view(np.uint64)
    for i in range(2):
        assert 0 < v[i, 1] - v[i, 0] < 10**9, v[i]
        assert torch.equal(outs[i], plain)
    assert v[1, 0] >= v[0, 0]                      # the second call started later
    assert v[2, 0] == np.uint64(2**64 - 1) and v[2, 1] == 0  # an unset pair is untouched
    total_ns = e0.elapsed_time(e1) * 1e6
    assert (v[0, 1] - v[0, 0]) + (v[1, 1] - v[1, 0]) <= total_ns * 1.05 + 2000


@pytest.mark.parametrize("group", ["1", "2", "3", "7", "100"])
@pytest.mark.parametrize("streamk", ["0", "1"])
def test_tc_tile_bands_cover_every_tile_once(group, streamk, monkeypatch):
    # the banded tile order is a bijection of the tile grid for any band width,
    # a narrower last band included (1300 columns = 5.1 column tiles of 256,
    # 1000 rows = 7.8 row tiles of 128): integer inputs, every entry exact,
    # guard bands untouched
    monkeypatch.setenv("GEMM_TC_GROUP", group)
    monkeypatch.setenv("GEMM_TC_STREAMK", streamk)
    monkeypatch.setenv("GEMM_TC_CONFIG", "256,16,5,2,0")
    got, ref, _ = _run_shape(1000, 1300, 200, "tf32x3", 1.0, 0.0, seed=int(group), dist="int2")
    assert oracle.mismatches(got, ref) == 0


@pytest.mark.parametrize("cfg", ["64,32,3,1,1", "64,32,6,1,1"])
@pytest.mark.parametrize("streamk", ["0", "1"])
@pytest.mark.parametrize("M,N", [(4173, 64), (2000, 50)])
def test_narrow_b_tiles(cfg, streamk, M, N, monkeypatch):
    # narrow B (N <= 64), A split on chip, with and without stream-K, a
    # ragged last row tile
    monkeypatch.setenv("GEMM_TC_CONFIG", cfg)
    monkeypatch.setenv("GEMM_TC_STREAMK", streamk)
    K = 1024
    got, ref, D = _run_shape(M, N, K, "tf32x3", 1.0, 0.0, seed=M + N, dist="int2")
    assert oracle.mismatches(got, ref) == 0
    got, ref, D = _run_shape(M, N, K, "tf32x3", 0.5, 2.0, seed=M - N)
    assert oracle.err_normalised(got, ref, D) <= TOL_E1


# Small-product tiles with B stored K x N read as stored, transposed and
# split on chip (B_hi the raw values, B_lo beside them; no pass for B),
# forced through the knob's b_split field: against the oracle, exactly on
# integer inputs, and bit for bit against the same tiles with B split by the
# pass (both take B_hi = tf32_trunc(B) and issue the same MMAs).
TC_BSPLIT_KN = ["128,64,32,6,1,1", "128,64,32,4,0,1"]


@pytest.mark.parametrize("cfg", TC_BSPLIT_KN)
@pytest.mark.parametrize("shape", [(333, 272, 164), (129, 64, 777), (1, 300, 68), (300, 8, 1000),
                                   (777, 200, 300)])
def test_tc_b_transposed_on_chip(cfg, shape, monkeypatch):
    from roofline_gb300 import gemm
    M, N, K = shape
    ak = int(cfg.split(",")[4])
    pad = ((-K) % 4, (-N) % 4, (-N) % 4)  # every row on a 16-byte boundary
    monkeypatch.setenv("GEMM_TC_CONFIG", cfg + ",1")
    p = gemm.plan(M, N, K, K + pad[0], N + pad[1], N + pad[2], mode="tf32x3")
    assert (p["bn"], p["bk"], p["a_split_in_kernel"], p["b_split_in_kernel"]) == (64, 32, ak, 1)
    assert p["launches"] == (1 if ak else 2) + p["stream_k"]
    got, ref, D = _run_shape(M, N, K, "tf32x3", 1.5, 0.5, pad=pad, seed=K)
    assert oracle.err_normalised(got, ref, D) <= TOL_E1
    monkeypatch.setenv("GEMM_TC_CONFIG", cfg + ",0")
    got0, _, _ = _run_shape(M, N, K, "tf32x3", 1.5, 0.5, pad=pad, seed=K)
    assert np.array_equal(np.ascontiguousarray(got).view(np.uint32),
                          np.ascontiguousarray(got0).view(np.uint32))
    monkeypatch.setenv("GEMM_TC_CONFIG", cfg + ",1")
    got, ref, D = _run_shape(M, N, K, "tf32x3", 1.0, 0.0, pad=pad, seed=K, dist="int2")
    assert oracle.mismatches(got, ref) == 0


def test_tc_b_split_knob_refuses_unbuilt_forms(monkeypatch):
    # B stored K x N is transposed on chip only in 64 x 32 tiles: asking for
    # it with 128 x 256 tiles leaves the planner's choice in place
    from roofline_gb300 import gemm
    monkeypatch.setenv("GEMM_TC_CONFIG", "128,256,16,5,2,0,1")
    p = gemm.plan(2048, 2048, 2048, mode="tf32x3")
    assert not (p["bn"] == 256 and p["b_split_in_kernel"] == 1)
