// Split-K CUDA-core SGEMM that never allocates device memory.
//
// Some callers cannot call cudaMalloc: code that runs under a device-memory
// budget fixed when it starts (a framework whose caching allocator has
// already reserved the free memory, or an embedded service that must never
// grow its footprint), and latency-critical loops that cannot afford the
// device-wide synchronisation cudaMalloc/cudaFree imply.  For them this
// entry point keeps the split-K partial sums in a fixed-size array that the
// library's module carries in device memory, so the call allocates nothing:
// the caller still passes A, B and C.
//
// Cost of that choice: every GPU that loads the library holds
// GEMM_NOALLOC_SCRATCH_BYTES of device memory until the process exits, and
// every call shares the one array, so calls whose kernels overlap on the GPU
// (on different streams, or from different host threads) race on it.
#include <mutex>

#include "common.cuh"

namespace gg {
namespace {

constexpr size_t kScratchFloats = GEMM_NOALLOC_SCRATCH_BYTES / sizeof(float);
// Most K slices a caller may ask for (the planner's own cap for the CUDA cores).
constexpr int kMaxSplit = GEMM_NOALLOC_MAX_SPLIT;

// The scratch array.  Host code only sees a host-side stand-in under this
// name; the device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) float g_noalloc_scratch[kScratchFloats];

constexpr int kMaxDev = 64;
std::mutex g_mu;
float *g_scratch_ptr[kMaxDev];

// Device address of the scratch array on the current device (looked up once
// per device, with that device current).
int scratch_for_device(int dev, float **out) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_ptr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return GEMM_ERR_CUDA;
    }
    g_scratch_ptr[dev] = static_cast<float *>(p);
  }
  *out = g_scratch_ptr[dev];
  return GEMM_OK;
}

}  // namespace
}  // namespace gg

using namespace gg;

extern "C" int gemm_f32_splitk_noalloc(int64_t M, int64_t N, int64_t K, float alpha,
                                       const float *A, int64_t lda, const float *B, int64_t ldb,
                                       float beta, float *C, int64_t ldc, int split_k,
                                       cudaStream_t stream) {
  if (M < 0 || N < 0 || K < 0 || split_k < 0 || split_k > kMaxSplit) return GEMM_ERR_INVALID_ARG;
  if (lda < (K > 1 ? K : 1) || ldb < (N > 1 ? N : 1) || ldc < (N > 1 ? N : 1))
    return GEMM_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return GEMM_OK;
  if (!C || (K > 0 && (!A || !B))) return GEMM_ERR_INVALID_ARG;

  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_NO_DEVICE;
  }
  if (dev < 0 || dev >= kMaxDev) return GEMM_ERR_UNSUPPORTED;
  const DeviceProps &dp = props_of(dev);
  GemmArgs p{M, N, K, alpha, beta, A, lda, B, ldb, C, ldc};
  // K == 0, or alpha == 0 (BLAS: A and B are not read): C <- beta * C
  if (K == 0 || alpha == 0.0f)
    return launch_scale(p, stream) == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;

  gemm_plan_t plan;
  int st = make_plan(M, N, K, lda, ldb, ldc, GEMM_MODE_FP32_SIMT,
                     (uintptr_t)A | (uintptr_t)B | (uintptr_t)C, beta != 0.0f, dp, &plan);
  if (st != GEMM_OK) return st;
  // Slices: the caller's count, or the planner's cut down to what the array
  // holds (one slice needs no scratch), rounded to whole BK-deep slices.
  int64_t want = split_k > 0 ? split_k : plan.split_k;
  if (split_k == 0 && want > 1) {
    const uint64_t fit = (uint64_t)kScratchFloats / ((uint64_t)M * (uint64_t)N);
    if ((uint64_t)want > fit) want = fit > 1 ? (int64_t)fit : 1;
  }
  if (want < 1) want = 1;
  {
    const int64_t kps = ceil_div(ceil_div(K, want), plan.bk) * plan.bk;
    plan.split_k = (int)ceil_div(K, kps);
  }
  if (plan.split_k > 1 &&
      (uint64_t)plan.split_k * (uint64_t)M * (uint64_t)N > (uint64_t)kScratchFloats)
    return GEMM_ERR_WORKSPACE_TOO_SMALL;

  float *scratch = nullptr;
  st = scratch_for_device(dev, &scratch);
  if (st != GEMM_OK) return st;
  // Every partial-sum element the reduction reads is written first by the
  // GEMM kernel of the same call, so the array needs no clearing.
  return launch_simt(plan, p, scratch, stream) == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}
