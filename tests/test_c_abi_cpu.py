"""The C boundary from C (no GPU needed): include/gb300_gemm.h compiles as
C99 with warnings as errors, a C program links against libgb300gemm.so, and
the host-only calls answer as documented (status strings, the plan of a
4096^3 product, argument errors)."""
import os
import shutil
import subprocess

import pytest

from roofline_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "gb300_gemm.h"

int main(void) {
  gemm_plan_t p;
  int rc;
  if (gemm_abi_version() != GEMM_ABI_VERSION) return 10;
  if (strlen(gemm_strerror(GEMM_ERR_INVALID_ARG)) == 0) return 11;
  /* planning is host-only */
  rc = gemm_f32_plan(4096, 4096, 4096, 4096, 4096, 4096, GEMM_MODE_AUTO, 0, 0, &p);
  if (rc != GEMM_OK) return 12;
  printf("kernel %d bm %d bn %d launches %d ws %llu\n", (int)p.kernel, (int)p.bm, (int)p.bn,
         (int)p.launches, (unsigned long long)p.workspace_bytes);
  if (p.kernel != GEMM_KERNEL_TC_TF32X3 || p.flops != 2.0 * 4096.0 * 4096.0 * 4096.0) return 13;
  /* leading dimension smaller than the row: rejected before any device work */
  rc = gemm_f32_plan(64, 64, 64, 32, 64, 64, GEMM_MODE_FP32_SIMT, 0, 0, &p);
  if (rc != GEMM_ERR_INVALID_ARG) return 14;
  rc = gemm_f32(64, 64, 64, NULL, 64, NULL, 64, NULL, 64, GEMM_MODE_AUTO, 0);
  if (rc != GEMM_ERR_INVALID_ARG) return 15;
  printf("noalloc %llu %d\n", (unsigned long long)GEMM_NOALLOC_SCRATCH_BYTES,
         (int)GEMM_NOALLOC_MAX_SPLIT);
  printf("abi %d sizeof_plan %d sizeof_info %d\n", (int)GEMM_ABI_VERSION,
         (int)sizeof(gemm_plan_t), (int)sizeof(gemm_device_info_t));
  puts("ok");
  return 0;
}
"""


def _cuda_include():
    for d in [os.environ.get("CUDA_HOME", ""), "/usr/local/cuda"]:
        if d and os.path.exists(os.path.join(d, "include", "cuda_runtime_api.h")):
            return os.path.join(d, "include")
    nvcc = shutil.which("nvcc")
    if nvcc:
        d = os.path.join(os.path.dirname(os.path.dirname(nvcc)), "include")
        if os.path.exists(os.path.join(d, "cuda_runtime_api.h")):
            return d
    return None


def test_header_and_library_from_c(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    inc = _cuda_include()
    if cc is None or inc is None:
        pytest.skip("no C compiler or CUDA headers")
    lib = build.build()
    src = tmp_path / "use_gemm.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "use_gemm"
    cmd = [cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
           "-I", inc, str(src), "-o", str(exe), lib, "-Wl,-rpath," + os.path.dirname(lib)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), (r.returncode, r.stdout,
                                                                   r.stderr)
    # the binding's copies of the header's no-allocation limits
    from roofline_gb300 import gemm
    line = [l for l in r.stdout.splitlines() if l.startswith("noalloc ")][0]
    assert line.split()[1:] == [str(gemm.NOALLOC_SCRATCH_BYTES), str(gemm.NOALLOC_MAX_SPLIT)]
    # ... and of its structures: the ABI version and the C sizes of the plan
    # and device-info structs match the ctypes mirrors
    import ctypes
    line = [l for l in r.stdout.splitlines() if l.startswith("abi ")][0].split()
    assert int(line[1]) == gemm.ABI_VERSION
    assert int(line[3]) == ctypes.sizeof(gemm.GemmPlan)
    assert int(line[5]) == ctypes.sizeof(gemm.DeviceInfo)
