"""Host-side checks of the C ABI: the library loads, exports every symbol the
header declares, and rejects bad arguments before touching a GPU."""
import os
import re

import pytest

from roofline_gb300 import build, gemm

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return gemm.load()


def _declared_symbols():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            with open(os.path.join(ROOT, "include", fn)) as f:
                src = f.read()
            names |= set(re.findall(r"GEMM_API\s+[\w\s\*]+?\b(\w+)\s*\(", src))
    return names


def test_exports_every_declared_symbol(lib):
    declared = _declared_symbols()
    assert declared, "no declarations found"
    assert declared == set(gemm.EXPORTED), declared ^ set(gemm.EXPORTED)
    for name in declared:
        assert hasattr(lib, name), name


def test_abi_version_and_strerror(lib):
    assert gemm.abi_version() == gemm.ABI_VERSION == 2
    for code in [0, -1, -2, -3, -4, -5, -6, 12345]:
        assert isinstance(gemm.strerror(code), str) and gemm.strerror(code)
    assert "invalid" in gemm.strerror(gemm.ERR_INVALID_ARG)


def test_device_info_defaults(lib):
    d = gemm.device_info(-1)
    assert d["from_device"] == 0 and d["sm_count"] > 0
    # peak = SMs x 128 lanes x 2 x clock
    assert d["fp32_peak_tflops"] == pytest.approx(d["sm_count"] * 128 * 2 * d["clock_khz"] * 1e3 / 1e12)


BAD = [
    dict(M=-1, N=4, K=4, lda=4, ldb=4, ldc=4),
    dict(M=4, N=-1, K=4, lda=4, ldb=4, ldc=4),
    dict(M=4, N=4, K=-1, lda=4, ldb=4, ldc=4),
    dict(M=4, N=4, K=8, lda=7, ldb=4, ldc=4),   # lda < K
    dict(M=4, N=8, K=4, lda=4, ldb=7, ldc=8),   # ldb < N
    dict(M=4, N=8, K=4, lda=4, ldb=8, ldc=7),   # ldc < N
]


@pytest.mark.parametrize("a", BAD)
def test_invalid_shapes_rejected(lib, a):
    rc = gemm.gemm_f32(a["M"], a["N"], a["K"], 16, a["lda"], 16, a["ldb"], 16, a["ldc"], 0, 0)
    assert rc == gemm.ERR_INVALID_ARG
    with pytest.raises(gemm.GemmError):
        gemm.plan(a["M"], a["N"], a["K"], a["lda"], a["ldb"], a["ldc"])


def test_null_pointers_and_mode_rejected(lib):
    assert gemm.gemm_f32(4, 4, 4, None, 4, 16, 4, 16, 4, 0, 0) == gemm.ERR_INVALID_ARG
    assert gemm.gemm_f32(4, 4, 4, 16, 4, None, 4, 16, 4, 0, 0) == gemm.ERR_INVALID_ARG
    assert gemm.gemm_f32(4, 4, 4, 16, 4, 16, 4, None, 4, 0, 0) == gemm.ERR_INVALID_ARG
    assert gemm.gemm_f32(4, 4, 4, 16, 4, 16, 4, 16, 4, 99, 0) == gemm.ERR_INVALID_ARG
    assert gemm.gemm_f32_ex(4, 4, 4, 1.0, 16, 4, 16, 4, 0.0, 16, 4, 0, 17, 1 << 20, 0) == \
        gemm.ERR_INVALID_ARG  # workspace not 256-byte aligned
    assert gemm.hbm_copy_calibrate.__doc__ is None or True
    assert lib.hbm_copy_calibrate(None, None, 16, 1, None, None) == gemm.ERR_INVALID_ARG


def test_noalloc_argument_errors(lib):
    # gemm_f32_splitk_noalloc rejects bad arguments before touching a device
    f = gemm.gemm_f32_splitk_noalloc
    ok = dict(M=4, N=4, K=4, alpha=1.0, A=256, lda=4, B=256, ldb=4, beta=0.0, C=256, ldc=4)

    def call(split=0, **kw):
        a = dict(ok, **kw)
        return f(a["M"], a["N"], a["K"], a["alpha"], a["A"], a["lda"], a["B"], a["ldb"],
                 a["beta"], a["C"], a["ldc"], split, 0)
    assert call(split=-1) == gemm.ERR_INVALID_ARG
    assert call(split=gemm.NOALLOC_MAX_SPLIT + 1) == gemm.ERR_INVALID_ARG
    assert call(M=-1) == gemm.ERR_INVALID_ARG
    assert call(K=-1) == gemm.ERR_INVALID_ARG
    assert call(lda=3) == gemm.ERR_INVALID_ARG   # lda < K
    assert call(ldb=3) == gemm.ERR_INVALID_ARG   # ldb < N
    assert call(ldc=3) == gemm.ERR_INVALID_ARG   # ldc < N
    assert call(C=None) == gemm.ERR_INVALID_ARG
    assert call(A=None) == gemm.ERR_INVALID_ARG
    assert call(M=0, A=None, B=None, C=None) == gemm.OK  # empty: nothing to do


def test_profile_stamps_argument_check(lib):
    assert lib.gemm_set_profile_stamps(4) == gemm.ERR_INVALID_ARG  # not 8-byte aligned
    assert lib.gemm_set_profile_stamps(None) == gemm.OK


def test_empty_products_are_noops_without_a_device(lib):
    # M == 0 or N == 0: nothing to do, no device needed, NULL pointers allowed
    assert gemm.gemm_f32(0, 5, 5, None, 5, None, 5, None, 5, 0, 0) == gemm.OK
    assert gemm.gemm_f32(5, 0, 5, None, 5, None, 1, None, 1, 0, 0) == gemm.OK


def test_plans_for_the_workloads(lib):
    p = gemm.plan(512, 512, 512, mode="fp32_simt")
    assert p["kernel_name"] == "simt" and p["vec"] == 1
    assert p["flops"] == 2 * 512 ** 3 and p["bytes"] == 3 * 512 * 512 * 4
    if p["split_k"] > 1:
        assert p["workspace_bytes"] == p["split_k"] * 512 * 512 * 4
    r = gemm.plan(1023, 1025, 777, 777, 1025, 1025, mode="fp32_simt", beta_nonzero=True)
    assert r["vec"] == 0  # lda = 777 is not a multiple of 4 floats
    assert r["bytes"] == 4 * (1023 * 777 + 777 * 1025 + 2 * 1023 * 1025)
    q = gemm.plan(4096, 4096, 4096, mode="fp32_simt")
    assert q["bm"] == 64 and q["bn"] == 128 and q["split_k"] == 1 and q["bound_name"] == "fp32"
    s = gemm.plan(65536, 64, 4096, mode="fp32_simt")
    assert s["intensity"] == pytest.approx(2 * 65536 * 64 * 4096 / 1_091_567_616)
    mis = gemm.plan(512, 512, 512, mode="fp32_simt", align_hint=4)
    assert mis["vec"] == 0
    z = gemm.plan(8, 8, 0)
    assert z["kernel_name"] == "scale"
    n = gemm.plan(0, 8, 8)
    assert n["kernel_name"] == "none"
    for m, name in [("naive", "naive"), ("coalesced", "coalesced"), ("tiled16", "tiled"),
                    ("tiled32", "tiled")]:
        assert gemm.plan(64, 64, 64, mode=m)["kernel_name"] == name


def test_valid_call_without_device_reports_no_device(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is visible")
    rc = gemm.gemm_f32(4, 4, 4, 256, 4, 256, 4, 256, 4, 1, 0)
    assert rc == gemm.ERR_NO_DEVICE


def test_simt_split_choice(lib):
    # small shapes slice K so every SM gets work; big ones do not
    assert gemm.plan(512, 512, 512, mode="fp32_simt")["split_k"] > 1
    assert gemm.plan(8192, 8192, 8192, mode="fp32_simt")["split_k"] == 1
    for shape in [(512, 512, 512), (1023, 1025, 777), (300, 200, 1000), (64, 64, 64)]:
        p = gemm.plan(*shape, mode="fp32_simt")
        M, N, K = shape
        kps = -(-K // p["split_k"])
        assert p["split_k"] == 1 or kps >= 16
        assert p["workspace_bytes"] == (p["split_k"] * M * N * 4 if p["split_k"] > 1 else 0)
        assert p["grid_ctas"] == -(-M // 64) * -(-N // 128) * p["split_k"]


def test_tc_plans_on_cpu(lib):
    p = gemm.plan(4096, 4096, 4096, mode="tf32x3")
    assert p["kernel_name"] == "tc_tf32x3" and p["bn"] == 256 and p["a_split_in_kernel"] == 1
    # B_hi and B_lo, plus two partial 128 x 256 tiles per stream-K CTA
    extra = p["grid_ctas"] * 2 * 128 * 256 * 4 if p["stream_k"] else 0
    assert p["workspace_bytes"] == 2 * 4096 * 4096 * 4 + extra
    s = gemm.plan(65536, 64, 4096, mode="tf32x3")
    assert s["bn"] == 64 and s["ctas_per_sm"] == 2 and s["bound_name"] == "hbm"
    r = gemm.plan(1023, 1025, 777, 777, 1025, 1025, mode="tf32x3")
    assert r["a_split_in_kernel"] == 0 and r["launches"] == 2 + r["stream_k"]
    assert gemm.plan(4096, 4096, 4096)["kernel_name"] == "tc_tf32x3"  # auto
    big = gemm.plan(8192, 8192, 8192, mode="tf32x3")  # A split on chip, A_hi and A_lo in TMEM
    assert (big["bm"], big["bn"], big["a_split_in_kernel"], big["a_hi_tmem"]) == (128, 256, 1, 1)
    # A pre-split anyway (leading dimension not a multiple of 4) and many tiles: 256 x 256
    big2 = gemm.plan(8192, 8192, 8191, 8191, 8192, 8192, mode="tf32x3")
    assert (big2["bm"], big2["bn"], big2["a_split_in_kernel"]) == (256, 256, 0)
    assert gemm.plan(384, 384, 1024)["kernel_name"] == "simt"  # auto: few tiles, long K


def test_stream_k_plan_bounds(lib):
    # each CTA owns at least 4 K blocks and a tile is split among at most 64 CTAs
    for shape in [(128, 128, 65536), (65536, 64, 4096), (4096, 4096, 4096), (256, 256, 256)]:
        p = gemm.plan(*shape, mode="tf32x3")
        if not p["stream_k"]:
            continue
        M, N, K = shape
        tiles = -(-M // 128) * -(-N // p["bn"])
        total = tiles * -(-K // p["bk"])
        assert 2 <= p["grid_ctas"] <= total // 4
        assert p["grid_ctas"] <= 64 * tiles
    # one tile with a very long K still spreads over 64 CTAs
    p = gemm.plan(128, 128, 16384, mode="tf32x3")
    assert p["stream_k"] == 1 and p["grid_ctas"] == 64


def test_auto_choice(lib):
    """AUTO takes the tensor cores once a problem amortises the split pass
    (about 2e8 multiply-adds), with K >= 128, M >= 128 and a C larger than
    256 x 256 (or K > 16384)."""
    tc = [(1023, 1025, 777, 777, 1025, 1025), (640, 640, 640), (1024, 1024, 1024),
          (2048, 2048, 512), (4096, 64, 4096), (512, 512, 1024), (128, 2048, 1024),
          (128, 1024, 8192), (256, 256, 65536),
          # small products that fit one wave of 128 x 64 tiles (13.7 against
          # 14.4 us at 512^3; 10.6 / 14.4 at 768 x 768 x 256)
          (512, 512, 512), (768, 768, 256), (512, 2048, 128), (576, 576, 576)]
    simt = [(4096, 4096, 64), (8192, 8192, 32), (384, 384, 1024),
            (64, 4096, 4096), (300, 300, 2000), (128, 128, 16384),
            (256, 256, 4096), (128, 512, 8192)]
    for shape in tc:
        assert gemm.plan(*shape)["kernel_name"] == "tc_tf32x3", shape
    for shape in simt:
        assert gemm.plan(*shape)["kernel_name"] == "simt", shape


def test_tf32_mode_plans(lib):
    p = gemm.plan(4096, 4096, 4096, mode="tf32")
    assert p["kernel_name"] == "tc_tf32" and p["bound_name"] == "tf32"
    # square: A pre-split too; A_hi and B_hi only (no lo parts), plus stream-K partials
    assert p["a_split_in_kernel"] == 0 and p["launches"] == 2 + p["stream_k"]
    extra = p["grid_ctas"] * 2 * p["bm"] * p["bn"] * 4 if p["stream_k"] else 0
    assert p["workspace_bytes"] == 2 * 4096 * 4096 * 4 + extra
    assert (p["bm"], p["bn"], p["bk"]) == (256, 256, 16)  # wide: 256 x 256 tiles
    big = gemm.plan(8192, 8192, 8192, mode="tf32")
    assert (big["bm"], big["bn"], big["bk"], big["stages"]) == (256, 256, 32, 3)  # long K
    s = gemm.plan(65536, 64, 4096, mode="tf32")
    assert s["bound_name"] == "hbm" and s["ctas_per_sm"] == 2 and s["a_split_in_kernel"] == 1
    assert gemm.plan(64, 64, 64, mode="tf32")["mode"] == gemm.MODE_TF32


def test_tensor_core_shape_limits(lib):
    # TMA tile coordinates are 32-bit and the split passes tile K on a grid's
    # y dimension: such shapes are refused in tensor-core modes, and AUTO
    # keeps them on the CUDA cores
    n_big = 1 << 31
    for mode in ("tf32x3", "tf32"):
        with pytest.raises(gemm.GemmError) as e:
            gemm.plan(1, n_big, 8, 8, n_big, n_big, mode=mode)
        assert e.value.code == gemm.ERR_UNSUPPORTED
        with pytest.raises(gemm.GemmError) as e:
            gemm.plan(128, 128, 65535 * 32 + 1, mode=mode)
        assert e.value.code == gemm.ERR_UNSUPPORTED
    assert gemm.plan(1, n_big, 8, 8, n_big, n_big)["kernel_name"] == "simt"
    assert gemm.plan(4096, 4096, 65535 * 32 + 1)["kernel_name"] == "simt"


def test_stream_k_choice(lib):
    # stream-K for HBM-bound shapes, for tiles filling at most half the SMs,
    # and where the time model says spreading K over the SMs beats the
    # partial tiles and the fix-up (the measured GB300 choices)
    assert gemm.plan(4096, 4096, 4096, mode="tf32x3")["stream_k"] == 1
    assert gemm.plan(2560, 2560, 4096, mode="tf32x3")["stream_k"] == 1
    # unaligned A with 128 x 64 tiles filling one wave: one CTA per tile, no
    # fix-up (1023 x 1025 x 777, lda 777: 35.0 against 37.6 us stream-K)
    r = gemm.plan(1023, 1025, 777, 777, 1025, 1025, mode="tf32x3")
    assert (r["bn"], r["stream_k"], r["grid_ctas"]) == (64, 0, 136)
    # a wave of 128 x 64 tiles with a moderate K: one CTA per tile
    assert gemm.plan(1024, 1024, 1024, mode="tf32x3")["stream_k"] == 0
    assert gemm.plan(1024, 1024, 4096, mode="tf32x3")["stream_k"] == 1
    # 1xTF32 2048^3: 64 tiles of 256 x 256 are under half a wave, so 128 x 256
    # tiles, one CTA each (48.6 us against 60.1 us stream-K on 256 x 256)
    p = gemm.plan(2048, 2048, 2048, mode="tf32")
    assert (p["bm"], p["bn"], p["stream_k"]) == (128, 256, 0)
    for shape in [(1536, 1536, 1536), (2048, 2048, 512), (2048, 2048, 2048),
                  (3000, 3000, 3000, 3003, 3000, 3000)]:
        assert gemm.plan(*shape, mode="tf32x3")["stream_k"] == 0, shape
    p = gemm.plan(2048, 4096, 4096, mode="tf32x3")
    assert (p["bn"], p["stream_k"], p["grid_ctas"]) == (256, 1, 152)
    # under one wave (128 tiles on 152 SMs): one CTA per tile
    q = gemm.plan(1024, 4096, 4096, mode="tf32x3")
    assert (q["bn"], q["stream_k"], q["grid_ctas"]) == (256, 0, 128)
    # few tiles for the SMs and a long K (512 x 512 x 1024): split K across them
    assert gemm.plan(512, 512, 1024, mode="tf32x3")["stream_k"] == 1
    assert gemm.plan(65536, 64, 4096, mode="tf32x3")["stream_k"] == 1
    assert gemm.plan(4096, 4096, 4096, mode="tf32")["stream_k"] == 0
    # whole waves only: no stream-K
    q = gemm.plan(152 * 128, 256, 4096, mode="tf32x3")
    assert q["stream_k"] == 0


def test_wide_tiles_from_half_a_wave(lib):
    # 128 x 256 tiles once there are at least 76 of them (half of 152 SMs)
    assert gemm.plan(1024, 4096, 4096, mode="tf32x3")["bn"] == 256
    assert gemm.plan(512, 512, 1024, mode="tf32x3")["bn"] == 128


# Planner decisions checked against exhaustive GB300 sweeps (every built
# configuration with and without stream-K; CUDA-core split counts forced one
# by one): (bm, bn, bk, stages, A split on chip, stream-K, split-K, B split
# on chip).
MEASURED_CHOICES = [
    ((4096, 4096, 4096), "tf32x3", (128, 256, 16, 5, 1, 1, 1, 0)),   # 460 vs 513 us without stream-K
    ((8192, 8192, 8192), "tf32x3", (128, 256, 16, 5, 1, 0, 1, 0)),
    ((1024, 1024, 16384), "tf32x3", (128, 256, 16, 5, 1, 1, 1, 0)),  # 154 vs 208 us for 128 x 128
    ((1024, 4096, 4096), "tf32x3", (128, 256, 16, 5, 1, 0, 1, 0)),   # 143 vs 169 us stream-K
    ((2560, 2560, 1024), "tf32x3", (128, 256, 16, 5, 1, 1, 1, 0)),   # 66 vs 73 us
    ((1536, 1536, 1536), "tf32x3", (128, 128, 32, 4, 1, 0, 1, 0)),
    ((8192, 384, 8192), "tf32x3", (128, 128, 32, 4, 1, 1, 1, 0)),    # 184 vs 206 us for 128 x 256
    ((1023, 1025, 777, 777, 1025, 1025), "tf32x3", (128, 64, 32, 4, 0, 0, 1, 0)),  # 35.0 vs 37.6 us
    ((512, 512, 512), "tf32x3", (128, 64, 32, 6, 1, 0, 1, 1)),    # 13.1 vs 14.0 us pre-split
    ((1024, 1024, 1024), "tf32x3", (128, 64, 32, 6, 1, 0, 1, 1)), # 21.0 vs 23.9 us pre-split
    ((1000, 1000, 1001, 1001, 1000, 1000), "tf32x3", (128, 64, 32, 4, 0, 0, 1, 0)),  # 30.5 vs 37.0 us
    ((1200, 640, 333, 333, 640, 640), "tf32x3", (128, 64, 32, 4, 0, 0, 1, 0)),  # 16.9 vs 20.9 us
    ((1200, 640, 336), "tf32x3", (128, 64, 32, 6, 1, 0, 1, 1)),   # 11.0 vs 13.3 us B pre-split
    ((768, 768, 768), "tf32x3", (128, 64, 32, 6, 1, 0, 1, 1)),    # 16.9 vs 18.9 us B pre-split
    ((1024, 64, 8192), "tf32x3", (128, 64, 32, 6, 1, 1, 1, 0)),      # 29.7 vs 38.2 us
    ((65536, 64, 4096), "tf32x3", (128, 64, 32, 3, 1, 1, 1, 0)),     # 204 vs 271 us for 6 stages
    ((4096, 4096, 4096), "tf32", (256, 256, 16, 6, 0, 0, 1, 0)),     # 212 vs 217 us for BK 32
    ((8192, 8192, 8192), "tf32", (256, 256, 32, 3, 0, 1, 1, 0)),     # 1337 vs 1468 us for BK 16
    ((2048, 2048, 2048), "tf32", (128, 256, 16, 8, 0, 0, 1, 0)),     # 48.6 vs 60.1 us for 256 x 256
    ((1024, 1024, 1024), "tf32", (128, 256, 16, 8, 0, 0, 1, 0)),     # 25.6 vs 27.1 us stream-K
    ((32, 32, 65536), "fp32_simt", (64, 128, 16, 4, 0, 0, 142, 0)),  # ~39 us vs 238 us at 16 slices
    ((128, 128, 16384), "fp32_simt", (64, 128, 16, 4, 0, 0, 69, 0)),
    ((512, 512, 512), "fp32_simt", (64, 128, 16, 4, 0, 0, 8, 0)),
]


@pytest.mark.parametrize("shape,mode,want", MEASURED_CHOICES,
                         ids=lambda v: "x".join(map(str, v)) if isinstance(v, tuple) else str(v))
def test_measured_planner_choices(lib, shape, mode, want):
    p = gemm.plan(*shape, mode=mode)
    got = (p["bm"], p["bn"], p["bk"], p["stages"], p["a_split_in_kernel"], p["stream_k"],
           p["split_k"], p["b_split_in_kernel"])
    assert got == want

