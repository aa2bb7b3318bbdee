// GEMM on matrices in host memory: C <- alpha * A * B + beta * C with A, B
// and C in (preferably page-locked) host memory, row-major.
//
// The course page times its kernels with the operands already on the GPU
// and leaves the host copies outside the measurement ("Project - tiled
// matrix multiply", "Starter scaffolding": cudaMemcpy in, kernel timed with
// events, cudaMemcpy out).  A caller whose data lives on the host pays for
// those copies too, and on GB300 they take longer than the GEMM: about
// 196 GB/s host-to-device and 180 GB/s device-to-host were measured on this
// machine's host link, against 137 GFLOP in 0.47 ms for a 4096^3 product
// whose 192 MB of operands and result take about 1 ms to move.  So the
// product is pipelined in row blocks over three library streams:
//
//   h2d:  B, then A rows [r0, r1) (and C rows when beta != 0), block by block
//   comp: GEMM of block i once its rows have arrived
//   d2h:  C rows [r0, r1) of block i once its GEMM is done
//
// so the copies of later blocks, the GEMM of the current one and the copy
// back of earlier ones run at the same time.  The whole problem is staged in
// device memory owned by the library (grown on demand, freed by
// gemm_shutdown()).  Every block runs in the mode resolved for the first
// block; on the tensor-core path the first block splits B into its TF32
// planes and the later blocks reuse them.
#include <mutex>

#include "common.cuh"

namespace gg {
namespace {

constexpr int kMaxDev = 64;
constexpr int kMaxBlocks = GEMM_HOST_MAX_BLOCKS;

struct HostPipe {
  bool ready = false;
  cudaStream_t h2d = nullptr, comp = nullptr, d2h = nullptr;
  cudaEvent_t in[kMaxBlocks] = {};
  cudaEvent_t out[kMaxBlocks] = {};
  void *buf = nullptr;
  size_t bytes = 0;
};

std::mutex g_host_mu[kMaxDev];
HostPipe g_pipe[kMaxDev];

void destroy(HostPipe &p) {
  if (p.h2d) cudaStreamDestroy(p.h2d);
  if (p.comp) cudaStreamDestroy(p.comp);
  if (p.d2h) cudaStreamDestroy(p.d2h);
  for (int i = 0; i < kMaxBlocks; ++i) {
    if (p.in[i]) cudaEventDestroy(p.in[i]);
    if (p.out[i]) cudaEventDestroy(p.out[i]);
  }
  if (p.buf) cudaFree(p.buf);
  cudaGetLastError();
  p = HostPipe{};
}

int setup(HostPipe &p) {
  if (p.ready) return GEMM_OK;
  bool ok = cudaStreamCreateWithFlags(&p.h2d, cudaStreamNonBlocking) == cudaSuccess &&
            cudaStreamCreateWithFlags(&p.comp, cudaStreamNonBlocking) == cudaSuccess &&
            cudaStreamCreateWithFlags(&p.d2h, cudaStreamNonBlocking) == cudaSuccess;
  for (int i = 0; ok && i < kMaxBlocks; ++i)
    ok = cudaEventCreateWithFlags(&p.in[i], cudaEventDisableTiming) == cudaSuccess &&
         cudaEventCreateWithFlags(&p.out[i], cudaEventDisableTiming) == cudaSuccess;
  if (!ok) {
    destroy(p);
    return GEMM_ERR_CUDA;
  }
  p.ready = true;
  return GEMM_OK;
}

int reserve(HostPipe &p, size_t need) {
  if (p.bytes >= need) return GEMM_OK;
  if (p.buf) {
    cudaFree(p.buf);
    p.buf = nullptr;
    p.bytes = 0;
  }
  if (cudaMalloc(&p.buf, need) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_CUDA;
  }
  p.bytes = need;
  return GEMM_OK;
}

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Row blocks for a product: one block while the GEMM is short (under
// ~8 GFLOP the copies dominate and a single launch has the least overhead),
// else blocks of at least 1024 rows, at most 4 of them.  Measured on GB300
// with pinned buffers (ms per call for 1 / 2 / 4 / 8 blocks): 4096^3 1.49 /
// 1.35 / 1.23 / 1.22, 8192^3 7.39 / 6.12 / 5.45 / 6.50, M = 65536, N = 64,
// K = 4096: 5.42 / 5.59 / 5.24 / 5.33.
int auto_blocks(int64_t M, int64_t N, int64_t K) {
  if (2.0 * (double)M * (double)N * (double)K < 8e9) return 1;
  int64_t b = M / 1024;
  if (b < 1) b = 1;
  if (b > 4) b = 4;
  return (int)b;
}

// Waits for all three streams, so no copy touches the caller's buffers
// after the call returns; returns the first error seen.
int drain(HostPipe &p, int st) {
  const cudaError_t e1 = cudaStreamSynchronize(p.h2d);
  const cudaError_t e2 = cudaStreamSynchronize(p.comp);
  const cudaError_t e3 = cudaStreamSynchronize(p.d2h);
  if (e1 != cudaSuccess || e2 != cudaSuccess || e3 != cudaSuccess) {
    cudaGetLastError();
    if (st == GEMM_OK) st = GEMM_ERR_CUDA;
  }
  return st;
}

cudaError_t copy_rows(float *dst, int64_t dld, const float *src, int64_t sld, int64_t cols,
                      int64_t rows, cudaMemcpyKind kind, cudaStream_t s) {
  if (rows <= 0 || cols <= 0) return cudaSuccess;
  return cudaMemcpy2DAsync(dst, (size_t)dld * 4, src, (size_t)sld * 4, (size_t)cols * 4,
                           (size_t)rows, kind, s);
}

}  // namespace

void host_pipeline_shutdown() {
  int cur = -1;
  const bool have_cur = cudaGetDevice(&cur) == cudaSuccess;
  for (int d = 0; d < kMaxDev; ++d) {
    std::lock_guard<std::mutex> lk(g_host_mu[d]);
    if (!g_pipe[d].ready && !g_pipe[d].buf) continue;
    cudaSetDevice(d);
    destroy(g_pipe[d]);
  }
  if (have_cur) cudaSetDevice(cur);
  cudaGetLastError();
}

}  // namespace gg

using namespace gg;

extern "C" int gemm_f32_host(int64_t M, int64_t N, int64_t K, float alpha, const float *A,
                             int64_t lda, const float *B, int64_t ldb, float beta, float *C,
                             int64_t ldc, int mode, int blocks) {
  if (M < 0 || N < 0 || K < 0 || blocks < 0 || blocks > kMaxBlocks) return GEMM_ERR_INVALID_ARG;
  if (lda < (K > 1 ? K : 1) || ldb < (N > 1 ? N : 1) || ldc < (N > 1 ? N : 1))
    return GEMM_ERR_INVALID_ARG;
  const int64_t lim = (int64_t)1 << 40;
  if (M > lim || N > lim || K > lim || lda > lim || ldb > lim || ldc > lim)
    return GEMM_ERR_INVALID_ARG;
  gemm_plan_t plan;
  int st = make_plan(M, N, K, K > 1 ? K : 1, N > 1 ? N : 1, N > 1 ? N : 1, mode, 0,
                     beta != 0.0f, default_props(), &plan);
  if (st == GEMM_ERR_INVALID_ARG) return st;
  if (M == 0 || N == 0) return GEMM_OK;
  if (!C || (K > 0 && (!A || !B))) return GEMM_ERR_INVALID_ARG;

  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_NO_DEVICE;
  }
  if (dev < 0 || dev >= kMaxDev) return GEMM_ERR_UNSUPPORTED;
  const DeviceProps &dp = props_of(dev);

  // row blocks: whole 128-row tiles except the last
  int nb = blocks > 0 ? blocks : auto_blocks(M, N, K);
  int64_t rows = ceil_div(M, nb);
  if (M > 128) rows = ceil_div(rows, 128) * 128;
  nb = (int)ceil_div(M, rows);
  const int64_t last = M - (int64_t)(nb - 1) * rows;
  const int64_t kld = K > 1 ? K : 1, nld = N > 1 ? N : 1;

  // one mode for every block: the one the first block resolves to
  gemm_plan_t p0, p1;
  st = make_plan(rows, N, K, kld, nld, nld, mode, 0, beta != 0.0f, dp, &p0);
  if (st != GEMM_OK) return st;
  const int bmode = (mode == GEMM_MODE_AUTO && K > 0) ? p0.mode : mode;
  st = make_plan(rows, N, K, kld, nld, nld, bmode, 0, beta != 0.0f, dp, &p0);
  if (st == GEMM_OK) st = make_plan(last, N, K, kld, nld, nld, bmode, 0, beta != 0.0f, dp, &p1);
  if (st != GEMM_OK) return st;
  const size_t ws_bytes = align256((size_t)(p0.workspace_bytes > p1.workspace_bytes
                                                ? p0.workspace_bytes
                                                : p1.workspace_bytes));
  const bool tc = p0.kernel == GEMM_KERNEL_TC_TF32X3 || p0.kernel == GEMM_KERNEL_TC_TF32;

  const size_t a_bytes = align256((size_t)M * K * 4), b_bytes = align256((size_t)K * N * 4);
  const size_t c_bytes = align256((size_t)M * N * 4);

  std::lock_guard<std::mutex> lk(g_host_mu[dev]);
  HostPipe &pp = g_pipe[dev];
  st = setup(pp);
  if (st == GEMM_OK) st = reserve(pp, a_bytes + b_bytes + c_bytes + ws_bytes);
  if (st != GEMM_OK) return st;
  char *base = static_cast<char *>(pp.buf);
  float *dA = reinterpret_cast<float *>(base);
  float *dB = reinterpret_cast<float *>(base + a_bytes);
  float *dC = reinterpret_cast<float *>(base + a_bytes + b_bytes);
  void *ws = ws_bytes ? base + a_bytes + b_bytes + c_bytes : nullptr;

  cudaError_t e = K > 0 ? copy_rows(dB, nld, B, ldb, N, K, cudaMemcpyHostToDevice, pp.h2d)
                        : cudaSuccess;
  for (int i = 0; i < nb && e == cudaSuccess && st == GEMM_OK; ++i) {
    const int64_t r0 = (int64_t)i * rows, nr = i + 1 < nb ? rows : last;
    if (K > 0)
      e = copy_rows(dA + r0 * kld, kld, A + r0 * lda, lda, K, nr, cudaMemcpyHostToDevice, pp.h2d);
    if (e == cudaSuccess && beta != 0.0f)
      e = copy_rows(dC + r0 * nld, nld, C + r0 * ldc, ldc, N, nr, cudaMemcpyHostToDevice, pp.h2d);
    if (e == cudaSuccess) e = cudaEventRecord(pp.in[i], pp.h2d);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(pp.comp, pp.in[i], 0);
    if (e != cudaSuccess) break;
    GemmArgs g{nr, N, K, alpha, beta, dA + r0 * kld, kld, dB, nld, dC + r0 * nld, nld};
    g.b_presplit = (tc && i > 0) ? 1 : 0;
    g.plain_order = 1;
    st = run_gemm(g, bmode, ws, ws_bytes, pp.comp);
    if (st != GEMM_OK) break;
    e = cudaEventRecord(pp.out[i], pp.comp);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(pp.d2h, pp.out[i], 0);
    if (e == cudaSuccess)
      e = copy_rows(C + r0 * ldc, ldc, dC + r0 * nld, nld, N, nr, cudaMemcpyDeviceToHost, pp.d2h);
  }
  if (e != cudaSuccess) {
    cudaGetLastError();
    if (st == GEMM_OK) st = GEMM_ERR_CUDA;
  }
  st = drain(pp, st);
  const int dev_st = tc ? tc_read_and_clear_status(pp.comp) : GEMM_OK;
  return st != GEMM_OK ? st : dev_st;
}
