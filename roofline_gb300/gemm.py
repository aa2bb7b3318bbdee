"""ctypes binding of libgb300gemm.so (include/gb300_gemm.h).

Argument marshalling only: every GEMM, split and copy runs in the library's
CUDA kernels.  The library must have been built (``roofline_gb300.build``);
loading fails loudly otherwise -- there is no CPU fallback.

Tensors passed to the tensor-level helpers are torch CUDA tensors (PyTorch
serves as the device allocator and stream provider); the raw-pointer
functions take integer device addresses and a cudaStream_t handle.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

MODE_AUTO = 0
MODE_FP32_SIMT = 1
MODE_TF32X3 = 2
MODE_TF32 = 3
MODE_NAIVE = 10
MODE_COALESCED = 11
MODE_TILED16 = 12
MODE_TILED32 = 13
MODES = {"auto": MODE_AUTO, "fp32_simt": MODE_FP32_SIMT, "tf32x3": MODE_TF32X3, "tf32": MODE_TF32,
         "naive": MODE_NAIVE, "coalesced": MODE_COALESCED, "tiled16": MODE_TILED16,
         "tiled32": MODE_TILED32}

# storage order and operand ops of gemm_f32_op
ABI_VERSION = 2  # GEMM_ABI_VERSION of include/gb300_gemm.h
ROW_MAJOR = 0
COL_MAJOR = 1
OP_N = 0
OP_T = 1

OK = 0
ERR_INVALID_ARG = -1
ERR_UNSUPPORTED = -2
ERR_CUDA = -3
ERR_DEVICE_TIMEOUT = -4
ERR_WORKSPACE_TOO_SMALL = -5
ERR_NO_DEVICE = -6

KERNELS = {0: "none", 1: "scale", 2: "naive", 3: "coalesced", 4: "tiled", 5: "simt",
           6: "tc_tf32x3", 7: "tc_tf32"}
BOUNDS = {0: "none", 1: "fp32", 2: "tf32x3", 3: "hbm", 4: "tf32"}

# Every symbol include/gb300_gemm.h declares.
EXPORTED = ["gemm_f32", "gemm_f32_ex", "gemm_f32_plan", "gemm_f32_op", "gemm_f32_op_plan",
            "gemm_f32_host", "hbm_copy_f32", "hbm_copy_calibrate",
            "gemm_device_info", "gemm_strerror", "gemm_check_status", "gemm_shutdown",
            "gemm_abi_version", "gemm_set_profile_events", "gemm_set_profile_stamps",
            "gemm_f32_splitk_noalloc",
            "fp32_fma_peak", "fp32_fma_peak_sink_floats"]

# most row blocks gemm_f32_host pipelines
HOST_MAX_BLOCKS = 64

# size of the static scratch array behind gemm_f32_splitk_noalloc, and the
# most K slices it takes (GEMM_NOALLOC_SCRATCH_BYTES, GEMM_NOALLOC_MAX_SPLIT;
# a CPU test compiles the header and compares)
NOALLOC_SCRATCH_BYTES = 8 << 20
NOALLOC_MAX_SPLIT = 256


class GemmPlan(ctypes.Structure):
    _fields_ = [("mode", ctypes.c_int32), ("kernel", ctypes.c_int32),
                ("bm", ctypes.c_int32), ("bn", ctypes.c_int32), ("bk", ctypes.c_int32),
                ("stages", ctypes.c_int32), ("split_k", ctypes.c_int32),
                ("vec", ctypes.c_int32), ("a_split_in_kernel", ctypes.c_int32),
                ("bound", ctypes.c_int32), ("threads", ctypes.c_int32),
                ("launches", ctypes.c_int32), ("grid_ctas", ctypes.c_int64),
                ("workspace_bytes", ctypes.c_uint64), ("flops", ctypes.c_double),
                ("bytes", ctypes.c_double), ("intensity", ctypes.c_double),
                ("b_concat", ctypes.c_int32), ("ctas_per_sm", ctypes.c_int32),
                ("stream_k", ctypes.c_int32), ("a_hi_tmem", ctypes.c_int32),
                ("b_split_in_kernel", ctypes.c_int32)]

    def as_dict(self):
        d = {name: getattr(self, name) for name, _ in self._fields_}
        d["kernel_name"] = KERNELS.get(self.kernel, "?")
        d["bound_name"] = BOUNDS.get(self.bound, "?")
        return d


class DeviceInfo(ctypes.Structure):
    _fields_ = [("device", ctypes.c_int32), ("sm_count", ctypes.c_int32),
                ("cc_major", ctypes.c_int32), ("cc_minor", ctypes.c_int32),
                ("clock_khz", ctypes.c_int32), ("mem_clock_khz", ctypes.c_int32),
                ("mem_bus_width_bits", ctypes.c_int32), ("fp32_lanes_per_sm", ctypes.c_int32),
                ("regs_per_sm", ctypes.c_int32), ("smem_per_sm", ctypes.c_int32),
                ("smem_per_block_optin", ctypes.c_int32), ("from_device", ctypes.c_int32),
                ("l2_bytes", ctypes.c_int64), ("hbm_bytes", ctypes.c_int64),
                ("fp32_peak_tflops", ctypes.c_double), ("name", ctypes.c_char * 128)]

    def as_dict(self):
        d = {name: getattr(self, name) for name, _ in self._fields_}
        d["name"] = self.name.decode(errors="replace")
        return d


class GemmError(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        self.code = code
        super().__init__(f"{what}: {strerror(code)} ({code})" if what else strerror(code))


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB


def load(path: str | None = None):
    """Load the library (once).  Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or _build.LIB
        if not os.path.exists(p):
            raise RuntimeError(f"{p} is missing: build it with `python -m roofline_gb300.build` "
                               "(the GEMM library has no CPU fallback)")
        lib = ctypes.CDLL(p)
        i64, f32, vp, i32 = ctypes.c_int64, ctypes.c_float, ctypes.c_void_p, ctypes.c_int
        lib.gemm_f32.argtypes = [i64, i64, i64, vp, i64, vp, i64, vp, i64, i32, vp]
        lib.gemm_f32.restype = i32
        lib.gemm_f32_ex.argtypes = [i64, i64, i64, f32, vp, i64, vp, i64, f32, vp, i64, i32,
                                    vp, ctypes.c_size_t, vp]
        lib.gemm_f32_ex.restype = i32
        lib.gemm_f32_plan.argtypes = [i64, i64, i64, i64, i64, i64, i32, ctypes.c_size_t, i32,
                                      ctypes.POINTER(GemmPlan)]
        lib.gemm_f32_plan.restype = i32
        lib.gemm_f32_op.argtypes = [i32, i32, i32, i64, i64, i64, f32, vp, i64, vp, i64, f32,
                                    vp, i64, i32, vp, ctypes.c_size_t, vp]
        lib.gemm_f32_op.restype = i32
        lib.gemm_f32_op_plan.argtypes = [i32, i32, i32, i64, i64, i64, i64, i64, i64, i32,
                                         ctypes.c_size_t, i32, ctypes.POINTER(GemmPlan)]
        lib.gemm_f32_op_plan.restype = i32
        lib.gemm_f32_host.argtypes = [i64, i64, i64, f32, vp, i64, vp, i64, f32, vp, i64, i32,
                                      i32]
        lib.gemm_f32_host.restype = i32
        lib.hbm_copy_f32.argtypes = [vp, vp, ctypes.c_size_t, vp]
        lib.hbm_copy_f32.restype = i32
        lib.hbm_copy_calibrate.argtypes = [vp, vp, ctypes.c_size_t, i32, vp,
                                           ctypes.POINTER(ctypes.c_double)]
        lib.hbm_copy_calibrate.restype = i32
        lib.gemm_device_info.argtypes = [i32, ctypes.POINTER(DeviceInfo)]
        lib.gemm_device_info.restype = i32
        lib.gemm_strerror.argtypes = [i32]
        lib.gemm_strerror.restype = ctypes.c_char_p
        lib.gemm_check_status.argtypes = [vp]
        lib.gemm_check_status.restype = i32
        lib.gemm_shutdown.argtypes = []
        lib.gemm_shutdown.restype = None
        lib.gemm_abi_version.argtypes = []
        lib.gemm_abi_version.restype = i32
        lib.gemm_set_profile_events.argtypes = [vp, vp]
        lib.gemm_set_profile_events.restype = i32
        lib.gemm_set_profile_stamps.argtypes = [vp]
        lib.gemm_set_profile_stamps.restype = i32
        lib.gemm_f32_splitk_noalloc.argtypes = [i64, i64, i64, f32, vp, i64, vp, i64, f32, vp,
                                                i64, i32, vp]
        lib.gemm_f32_splitk_noalloc.restype = i32
        lib.fp32_fma_peak.argtypes = [i64, i32, vp, vp, ctypes.POINTER(ctypes.c_double)]
        lib.fp32_fma_peak.restype = i32
        lib.fp32_fma_peak_sink_floats.argtypes = []
        lib.fp32_fma_peak_sink_floats.restype = i64
        # the structures above mirror this version of the header
        if lib.gemm_abi_version() != ABI_VERSION:
            raise RuntimeError(f"{p} reports ABI version {lib.gemm_abi_version()}, this binding "
                               f"is written for {ABI_VERSION}: rebuild the library")
        if path is None:
            _lib = lib
        return lib


def strerror(code: int) -> str:
    return load().gemm_strerror(int(code)).decode()


def _mode(mode) -> int:
    return MODES[mode] if isinstance(mode, str) else int(mode)


# ------------------------------------------------------------ raw pointers

def gemm_f32(M, N, K, A, lda, B, ldb, C, ldc, mode=MODE_AUTO, stream=0) -> int:
    return load().gemm_f32(M, N, K, A, lda, B, ldb, C, ldc, _mode(mode), stream)


def gemm_f32_ex(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, mode=MODE_AUTO,
                workspace=None, ws_bytes=0, stream=0) -> int:
    return load().gemm_f32_ex(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, _mode(mode),
                              workspace, ws_bytes, stream)


def gemm_f32_op(layout, op_a, op_b, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc,
                mode=MODE_AUTO, workspace=None, ws_bytes=0, stream=0) -> int:
    return load().gemm_f32_op(layout, op_a, op_b, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc,
                              _mode(mode), workspace, ws_bytes, stream)


def gemm_f32_host(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, mode=MODE_AUTO,
                  blocks=0) -> int:
    """Host-memory GEMM (raw host addresses); blocking; returns the status."""
    return load().gemm_f32_host(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, _mode(mode),
                                blocks)


def gemm_f32_splitk_noalloc(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, split_k=0,
                            stream=0) -> int:
    """Split-K CUDA-core GEMM whose scratch is the library's static device
    array: no device allocation happens in the call (for callers that cannot
    allocate).  Raw device pointers; returns the status code."""
    return load().gemm_f32_splitk_noalloc(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc,
                                          split_k, stream)


def plan(M, N, K, lda=None, ldb=None, ldc=None, mode=MODE_AUTO, align_hint=0,
         beta_nonzero=False) -> dict:
    out = GemmPlan()
    rc = load().gemm_f32_plan(M, N, K, max(K, 1) if lda is None else lda,
                              max(N, 1) if ldb is None else ldb,
                              max(N, 1) if ldc is None else ldc, _mode(mode), align_hint,
                              1 if beta_nonzero else 0, ctypes.byref(out))
    if rc != OK:
        raise GemmError(rc, "gemm_f32_plan")
    return out.as_dict()


def stored_shape(layout, op, rows, cols):
    """(rows, cols) of the matrix as stored for a logical rows x cols
    operand op(X), and the smallest legal leading dimension."""
    r, c = (rows, cols) if op == OP_N else (cols, rows)
    return (r, c), max(c if layout == ROW_MAJOR else r, 1)


def plan_op(layout, op_a, op_b, M, N, K, lda=None, ldb=None, ldc=None, mode=MODE_AUTO,
            align_hint=0, beta_nonzero=False) -> dict:
    """gemm_f32_op_plan: the row-major problem a gemm_f32_op call runs."""
    out = GemmPlan()
    lda = stored_shape(layout, op_a, M, K)[1] if lda is None else lda
    ldb = stored_shape(layout, op_b, K, N)[1] if ldb is None else ldb
    ldc = stored_shape(layout, OP_N, M, N)[1] if ldc is None else ldc
    rc = load().gemm_f32_op_plan(layout, op_a, op_b, M, N, K, lda, ldb, ldc, _mode(mode),
                                 align_hint, 1 if beta_nonzero else 0, ctypes.byref(out))
    if rc != OK:
        raise GemmError(rc, "gemm_f32_op_plan")
    return out.as_dict()


def device_info(dev: int = 0) -> dict:
    out = DeviceInfo()
    rc = load().gemm_device_info(dev, ctypes.byref(out))
    if rc != OK:
        raise GemmError(rc, "gemm_device_info")
    return out.as_dict()


def check_status(stream=0) -> int:
    return load().gemm_check_status(stream)


def shutdown() -> None:
    load().gemm_shutdown()


def abi_version() -> int:
    return load().gemm_abi_version()


def set_profile_events(before=None, after=None) -> None:
    """Record torch.cuda.Event `before`/`after` around the main kernel of the
    following calls made from this thread (None, None to stop)."""
    b = None if before is None else before.cuda_event
    a = None if after is None else after.cuda_event
    if (before is not None and not b) or (after is not None and not a):
        raise ValueError("record the events once before passing them (torch creates them lazily)")
    rc = load().gemm_set_profile_events(b, a)
    if rc != OK:
        raise GemmError(rc, "gemm_set_profile_events")


def set_profile_stamps(stamps=None) -> None:
    """Main-kernel stamps of the following calls from this thread go to the
    device int64 pair `stamps` (a tensor of 2 or more int64 starting at that
    pair, or a device address); None stops.  The caller fills [~0, 0]
    first; afterwards stamps[1] - stamps[0] is the kernel's duration in ns."""
    if stamps is None:
        ptr = None
    elif isinstance(stamps, int):
        ptr = stamps
    else:
        if not stamps.is_cuda or stamps.dtype.itemsize != 8:
            raise ValueError("stamps must be a CUDA tensor of 8-byte integers")
        ptr = stamps.data_ptr()
    rc = load().gemm_set_profile_stamps(ptr)
    if rc != OK:
        raise GemmError(rc, "gemm_set_profile_stamps")


# ------------------------------------------------------------ torch tensors

def _stream_handle(stream):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _operand(t, name):
    """(op, ld) of a 2-D float32 CUDA tensor used as a GEMM operand: a
    row-major view (unit column stride) is op N with ld = row stride; a
    transposed view of a row-major buffer (unit row stride, e.g. ``X.t()``)
    is op T with ld = column stride."""
    import torch
    if not (t.is_cuda and t.dtype == torch.float32 and t.dim() == 2):
        raise ValueError(f"{name} must be a 2-D float32 CUDA tensor")
    # A stride along a dimension of length 1 is never used (torch may report
    # any value there), so the leading dimension is then at least the row
    # length of the stored matrix.
    if t.stride(1) == 1 or t.shape[1] <= 1:
        ld = t.stride(0) if t.shape[0] > 1 else max(t.stride(0), t.shape[1])
        return OP_N, max(ld, 1)
    if t.stride(0) == 1 or t.shape[0] <= 1:
        ld = t.stride(1) if t.shape[1] > 1 else max(t.stride(1), t.shape[0])
        return OP_T, max(ld, 1)
    raise ValueError(f"{name} must have a unit row or column stride")


def matmul(A, B, C=None, alpha=1.0, beta=0.0, mode=MODE_AUTO, stream=None,
           workspace=None):
    """C <- alpha * A @ B + beta * C for float32 CUDA tensors.

    A (M x K) and B (K x N) may be row slices of larger buffers (row stride =
    leading dimension) or transposed views of row-major buffers (``X.t()``,
    run as op T without a copy).  C is row-major, allocated when None (then
    beta must be 0).  ``workspace``: optional uint8/float CUDA tensor used as
    caller-owned scratch; without one the library's per-device buffer is
    used, which calls running at the same time on different streams must not
    share.  Returns C.
    """
    import torch
    M, K = A.shape
    K2, N = B.shape
    if K2 != K:
        raise ValueError(f"inner dimensions differ: {K} vs {K2}")
    if C is None:
        if beta != 0.0:
            raise ValueError("beta != 0 needs C")
        C = torch.empty((M, N), dtype=torch.float32, device=A.device)
    op_a, lda = _operand(A, "A")
    op_b, ldb = _operand(B, "B")
    op_c, ldc = _operand(C, "C")
    if op_c != OP_N:
        raise ValueError("C must be a 2-D float32 CUDA tensor with unit column stride")
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    if op_a == OP_N and op_b == OP_N:
        rc = load().gemm_f32_ex(M, N, K, float(alpha), A.data_ptr(), lda, B.data_ptr(), ldb,
                                float(beta), C.data_ptr(), ldc, _mode(mode), ws_ptr, ws_bytes,
                                _stream_handle(stream))
        what = "gemm_f32_ex"
    else:
        rc = load().gemm_f32_op(ROW_MAJOR, op_a, op_b, M, N, K, float(alpha), A.data_ptr(), lda,
                                B.data_ptr(), ldb, float(beta), C.data_ptr(), ldc, _mode(mode),
                                ws_ptr, ws_bytes, _stream_handle(stream))
        what = "gemm_f32_op"
    if rc != OK:
        raise GemmError(rc, what)
    return C


def _host_matrix(t, name):
    import torch
    if not (t.device.type == "cpu" and t.dtype == torch.float32 and t.dim() == 2 and
            (t.stride(1) == 1 or t.shape[1] <= 1)):
        raise ValueError(f"{name} must be a 2-D float32 CPU tensor with unit column stride")
    # the row stride of a one-row matrix is never used (torch may report any value)
    ld = t.stride(0) if t.shape[0] > 1 else max(t.stride(0), t.shape[1])
    return max(ld, 1)


def matmul_host(A, B, C=None, alpha=1.0, beta=0.0, mode=MODE_AUTO, blocks=0):
    """C <- alpha * A @ B + beta * C for row-major float32 CPU tensors (pin
    them with ``.pin_memory()`` so the copies overlap the GEMM).  The library
    moves the data to the GPU and back in blocks (row blocks of A and C,
    column blocks of B and C) and runs the GEMMs there as the blocks arrive;
    the call returns when C holds the result.  Returns C."""
    import torch
    M, K = A.shape
    K2, N = B.shape
    if K2 != K:
        raise ValueError(f"inner dimensions differ: {K} vs {K2}")
    if C is None:
        if beta != 0.0:
            raise ValueError("beta != 0 needs C")
        C = torch.empty((M, N), dtype=torch.float32, pin_memory=A.is_pinned())
    lda, ldb, ldc = _host_matrix(A, "A"), _host_matrix(B, "B"), _host_matrix(C, "C")
    rc = load().gemm_f32_host(M, N, K, float(alpha), A.data_ptr(), lda, B.data_ptr(), ldb,
                              float(beta), C.data_ptr(), ldc, _mode(mode), int(blocks))
    if rc != OK:
        raise GemmError(rc, "gemm_f32_host")
    return C


def hbm_copy(src, dst, stream=None) -> None:
    n = src.numel()
    if dst.numel() < n:
        raise ValueError("dst smaller than src")
    rc = load().hbm_copy_f32(src.data_ptr(), dst.data_ptr(), n, _stream_handle(stream))
    if rc != OK:
        raise GemmError(rc, "hbm_copy_f32")


def hbm_copy_calibrate(src, dst, iters=50, stream=None) -> float:
    out = ctypes.c_double(0.0)
    rc = load().hbm_copy_calibrate(src.data_ptr(), dst.data_ptr(), src.numel(), iters,
                                   _stream_handle(stream), ctypes.byref(out))
    if rc != OK:
        raise GemmError(rc, "hbm_copy_calibrate")
    return out.value


def fp32_fma_peak(iters=1 << 16, packed=True, stream=None) -> float:
    """Measured FP32 FMA throughput of the CUDA cores, TFLOP/s."""
    import torch
    sink = torch.empty(load().fp32_fma_peak_sink_floats(), dtype=torch.float32, device="cuda")
    out = ctypes.c_double(0.0)
    rc = load().fp32_fma_peak(int(iters), 1 if packed else 0, sink.data_ptr(),
                              _stream_handle(stream), ctypes.byref(out))
    if rc != OK:
        raise GemmError(rc, "fp32_fma_peak")
    return out.value
