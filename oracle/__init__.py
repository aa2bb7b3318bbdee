"""CPU oracle for the FP32 GEMM library -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline /
reference legs of ``bench.py`` may import this package.  The product path
(``roofline_gb300``) never imports it, and it imports nothing from there.

The arithmetic lives in ``gemm_oracle.c`` (fp64 accumulation in ascending k,
one final rounding to float; the CPU reference of the tiled-matmul course
page, section "Starter scaffolding", generalised to M, N, K, leading
dimensions and alpha/beta).  This module builds that file with gcc, loads it
with ctypes and adds the error metrics.

Pins: the oracle is checked in ``tests/test_oracle.py`` against the FLOP
count the page prints, closed forms (identity, all-ones, rank-1), exact
rational brute force on tiny shapes, numpy float64 matmul and the golden
fixtures under ``tests/golden``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gemm_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libgemm_oracle.so")
_lock = threading.Lock()

_f32p = ctypes.POINTER(ctypes.c_float)
_f64p = ctypes.POINTER(ctypes.c_double)
_i64p = ctypes.POINTER(ctypes.c_int64)


def compile_source(src: str, out: str) -> str:
    """Compile one oracle source file to a shared library with gcc."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
           "-fPIC", "-shared", "-std=c99", src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile ``gemm_oracle.c`` (-O2 -ffp-contract=off -fopenmp) if stale."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    return compile_source(_SRC, _LIB_PATH)


def _bind(lib):
    lib.oracle_gemm.restype = ctypes.c_int
    lib.oracle_gemm.argtypes = [
        ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_double,
        _f32p, ctypes.c_int64, _f32p, ctypes.c_int64, ctypes.c_double,
        _f32p, ctypes.c_int64, _f32p, _f64p, ctypes.c_int64, ctypes.c_int]
    lib.oracle_gemm_entries.restype = ctypes.c_int
    lib.oracle_gemm_entries.argtypes = [
        ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_double,
        _f32p, ctypes.c_int64, _f32p, ctypes.c_int64, ctypes.c_double,
        _f32p, ctypes.c_int64, ctypes.c_int64, _i64p, _i64p, _f32p, _f64p,
        ctypes.c_int]
    lib.oracle_max_threads.restype = ctypes.c_int
    return lib


def _ptr(a, t):
    return None if a is None else a.ctypes.data_as(t)


def _as_2d(x):
    x = np.asarray(x)
    assert x.dtype == np.float32 and x.ndim == 2 and x.strides[1] == 4
    return x


class Oracle:
    """The oracle routines bound to one build of ``gemm_oracle.c``."""

    def __init__(self, lib_path: str):
        self.lib = _bind(ctypes.CDLL(lib_path))

    def gemm(self, A, B, alpha=1.0, beta=0.0, C0=None, M=None, N=None, K=None,
             with_bound=False, nthreads=0):
        """C_ref = float_rn(alpha * sum_k A(i,k) B(k,j) + beta * C0(i,j)).

        A, B, C0 are 2-D float32 arrays with unit column stride (row stride =
        leading dimension).  M, N, K default to A.shape[0], B.shape[1],
        A.shape[1].  Returns C (M x N float32) or (C, D) with the per-entry
        error-bound denominator D (float64) when ``with_bound``.
        """
        A = _as_2d(A)
        B = _as_2d(B)
        M = A.shape[0] if M is None else M
        K = A.shape[1] if K is None else K
        N = B.shape[1] if N is None else N
        lda = A.strides[0] // 4
        ldb = B.strides[0] // 4
        if C0 is not None:  # read by the C code only when beta != 0
            C0 = _as_2d(C0)
            ldc = C0.strides[0] // 4
        else:
            assert beta == 0.0, "beta != 0 needs C0"
            ldc = max(N, 1)
        out = np.empty((M, N), dtype=np.float32)
        D = np.empty((M, N), dtype=np.float64) if with_bound else None
        rc = self.lib.oracle_gemm(M, N, K, float(alpha), _ptr(A, _f32p), lda, _ptr(B, _f32p),
                                  ldb, float(beta), _ptr(C0, _f32p), ldc, _ptr(out, _f32p),
                                  _ptr(D, _f64p), max(N, 1), nthreads)
        if rc != 0:
            raise ValueError("oracle_gemm: bad arguments")
        return (out, D) if with_bound else out

    def gemm_entries(self, A, B, rows, cols, alpha=1.0, beta=0.0, C0=None, M=None, N=None,
                     K=None, nthreads=0):
        """(values float32[n], bounds float64[n]) of C_ref at (rows[t], cols[t])."""
        A = _as_2d(A)
        B = _as_2d(B)
        M = A.shape[0] if M is None else M
        K = A.shape[1] if K is None else K
        N = B.shape[1] if N is None else N
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        cols = np.ascontiguousarray(cols, dtype=np.int64)
        n = rows.size
        if C0 is not None:  # read by the C code only when beta != 0
            C0 = _as_2d(C0)
            ldc = C0.strides[0] // 4
        else:
            assert beta == 0.0, "beta != 0 needs C0"
            ldc = max(N, 1)
        out = np.empty(n, dtype=np.float32)
        D = np.empty(n, dtype=np.float64)
        rc = self.lib.oracle_gemm_entries(M, N, K, float(alpha), _ptr(A, _f32p),
                                          A.strides[0] // 4, _ptr(B, _f32p), B.strides[0] // 4,
                                          float(beta), _ptr(C0, _f32p), ldc, n,
                                          _ptr(rows, _i64p), _ptr(cols, _i64p),
                                          _ptr(out, _f32p), _ptr(D, _f64p), nthreads)
        if rc != 0:
            raise ValueError("oracle_gemm_entries: bad arguments")
        return out, D

    def max_threads(self) -> int:
        return int(self.lib.oracle_max_threads())


_default = None


def default() -> Oracle:
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
    return _default


def gemm(*args, **kwargs):
    return default().gemm(*args, **kwargs)


def gemm_entries(*args, **kwargs):
    return default().gemm_entries(*args, **kwargs)


def max_threads() -> int:
    return default().max_threads()


# ---------------------------------------------------------------- metrics

def err_normalised(C, C_ref, D) -> float:
    """E1 = max |C - C_ref| / D, with D the per-entry bound
    |alpha| sum_k |A_ik||B_kj| + |beta||C_old_ij|.  0/0 counts as 0; a NaN
    or a nonzero error over a zero bound counts as inf."""
    C = np.asarray(C, dtype=np.float64)
    R = np.asarray(C_ref, dtype=np.float64)
    D = np.asarray(D, dtype=np.float64)
    diff = np.abs(C - R)
    if not np.all(np.isfinite(C)):
        return float("inf")
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.where(diff == 0.0, 0.0, diff / D)
    return float(np.max(q)) if q.size else 0.0


def mismatches(C, C_ref) -> int:
    """E2: number of entries that differ in value (bit-exact check for
    integer-valued inputs)."""
    C = np.asarray(C, dtype=np.float32)
    R = np.asarray(C_ref, dtype=np.float32)
    return int(np.count_nonzero(~(C == R)))


def err_pages(C, C_ref) -> float:
    """E3, the course page's check (section "Starter scaffolding"):
    max |g - r| / max(|r|, 1e-6)."""
    g = np.asarray(C, dtype=np.float64)
    r = np.asarray(C_ref, dtype=np.float64)
    return float(np.max(np.abs(g - r) / np.maximum(np.abs(r), 1e-6))) if r.size else 0.0
