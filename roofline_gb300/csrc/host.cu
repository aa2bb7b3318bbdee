// GEMM on matrices in host memory: C <- alpha * A * B + beta * C with A, B
// and C in (preferably page-locked) host memory, row-major.
//
// The course page times its kernels with the operands already on the GPU
// and leaves the host copies outside the measurement ("Project - tiled
// matrix multiply", "Starter scaffolding": cudaMemcpy in, kernel timed with
// events, cudaMemcpy out).  A caller whose data lives on the host pays for
// those copies too, and on GB300 they take longer than the GEMM: about
// 196 GB/s host-to-device and 180 GB/s device-to-host were measured on this
// machine's host link, against 137 GFLOP in 0.45 ms for a 4096^3 product
// whose 192 MB of operands and result take about 1 ms to move.  So the
// product is cut into a grid of row blocks of A (and C) and column blocks
// of B (and C), and three library streams overlap the copies with the GEMMs:
//
//   h2d:  B column block 0, A row block 0, then A row blocks and B column
//         blocks alternately, keeping the arrived fraction of A and of B
//         about equal (C row blocks travel with A's when beta != 0)
//   comp: as soon as a block arrives, the GEMMs it completes: a new A row
//         block against every B column block already there, a new B column
//         block against all the A rows already there (one GEMM)
//   d2h:  each GEMM's block of C, once that GEMM is done
//
// so the first GEMM starts once two blocks have arrived instead of after
// all of B.  The whole problem is staged in device memory owned by the
// library (grown on demand, freed by gemm_shutdown()).  Every GEMM runs in
// the mode resolved for the whole product; on the tensor-core path each B
// column block is split into its TF32 planes by its first GEMM, in a
// workspace of its own, and its later GEMMs reuse them.
#include <cuda.h>

#include <cstdlib>
#include <mutex>
#include <vector>

#include "common.cuh"

namespace gg {
namespace {

constexpr int kMaxDev = 64;
constexpr int kMaxBlocks = GEMM_HOST_MAX_BLOCKS;

constexpr int kMaxColBlocks = 8;
constexpr int kMaxStreamBlocks = 64;

// Stream memory operations of the driver (cuStreamWaitValue32 /
// cuStreamWriteValue32), looked up once; null when the driver lacks them.
typedef CUresult (*StreamValue32Fn)(CUstream, CUdeviceptr, cuuint32_t, unsigned int);
std::once_flag g_memops_once;
StreamValue32Fn g_wait32 = nullptr, g_write32 = nullptr;

bool memops() {
  std::call_once(g_memops_once, [] {
    void *w = nullptr, *r = nullptr;
    cudaDriverEntryPointQueryResult qw, qr;
    if (cudaGetDriverEntryPointByVersion("cuStreamWaitValue32", &w, 12000, cudaEnableDefault,
                                         &qw) == cudaSuccess &&
        qw == cudaDriverEntryPointSuccess &&
        cudaGetDriverEntryPointByVersion("cuStreamWriteValue32", &r, 12000, cudaEnableDefault,
                                         &qr) == cudaSuccess &&
        qr == cudaDriverEntryPointSuccess) {
      g_wait32 = reinterpret_cast<StreamValue32Fn>(w);
      g_write32 = reinterpret_cast<StreamValue32Fn>(r);
    } else {
      cudaGetLastError();
    }
  });
  return g_wait32 != nullptr && g_write32 != nullptr;
}

// Events are re-recorded freely: a stream wait takes the event's most recent
// record at the time the wait is enqueued.
struct HostPipe {
  bool ready = false;
  cudaStream_t h2d = nullptr, comp = nullptr, d2h = nullptr, rescue = nullptr;
  cudaEvent_t in = nullptr, out = nullptr;
  void *buf = nullptr;
  size_t bytes = 0;
  // streaming: in_flag[kMaxStreamBlocks], out_flag[...], tile_cnt[...] on
  // the device (zeroed once), and the value the next call publishes
  unsigned *flags = nullptr;
  unsigned epoch = 0;
};

std::mutex g_host_mu[kMaxDev];
HostPipe g_pipe[kMaxDev];

void destroy(HostPipe &p) {
  if (p.h2d) cudaStreamDestroy(p.h2d);
  if (p.comp) cudaStreamDestroy(p.comp);
  if (p.d2h) cudaStreamDestroy(p.d2h);
  if (p.rescue) cudaStreamDestroy(p.rescue);
  if (p.in) cudaEventDestroy(p.in);
  if (p.out) cudaEventDestroy(p.out);
  if (p.buf) cudaFree(p.buf);
  if (p.flags) cudaFree(p.flags);
  cudaGetLastError();
  p = HostPipe{};
}

int setup(HostPipe &p) {
  if (p.ready) return GEMM_OK;
  bool ok = cudaStreamCreateWithFlags(&p.h2d, cudaStreamNonBlocking) == cudaSuccess &&
            cudaStreamCreateWithFlags(&p.comp, cudaStreamNonBlocking) == cudaSuccess &&
            cudaStreamCreateWithFlags(&p.d2h, cudaStreamNonBlocking) == cudaSuccess &&
            cudaStreamCreateWithFlags(&p.rescue, cudaStreamNonBlocking) == cudaSuccess;
  ok = ok && cudaMalloc(&p.flags, 3 * kMaxStreamBlocks * sizeof(unsigned)) == cudaSuccess &&
       cudaMemset(p.flags, 0, 3 * kMaxStreamBlocks * sizeof(unsigned)) == cudaSuccess;
  ok = ok && cudaEventCreateWithFlags(&p.in, cudaEventDisableTiming) == cudaSuccess &&
       cudaEventCreateWithFlags(&p.out, cudaEventDisableTiming) == cudaSuccess;
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

// Blocking for a product (rows x columns).  One block while the GEMM is
// short (under ~8 GFLOP the copies dominate and a single launch has the
// least overhead).  Else, for a deep product (K >= 2048, where B is large
// and waiting for all of it delays the first GEMM), up to 3 x 3 blocks of at
// least 1024 rows and columns; otherwise row blocks only, up to 4.
// Measured on GB300 with pinned buffers (ms per call; rows x columns):
// 4096^3 1x1 1.46, 4x1 1.03, 2x2 1.14, 3x3 1.03, 4x4 1.07, 8x8 1.60;
// 8192^3 1x1 7.13, 4x1 5.14, 2x2 5.31, 3x3 4.78, 4x4 5.54, 4x8 4.92;
// 2048^3 4x1 0.321, 2x2 0.307, 3x3 0.342; 65536 x 64 x 4096 (rows only)
// 1 / 2 / 4 / 8 blocks: 5.42 / 5.59 / 5.24 / 5.33.  The copies in run at
// ~207 GB/s alone, ~275 GB/s in total with copies out at the same time;
// smaller blocks start the GEMMs earlier but each GEMM then carries its own
// fixed costs (4096^3 as 4x4: 613 us of GEMMs against 420 us for one call).
void auto_grid(int64_t M, int64_t N, int64_t K, int &nb, int &nc) {
  nb = nc = 1;
  if (2.0 * (double)M * (double)N * (double)K < 8e9) return;
  auto clamp = [](int64_t v, int64_t hi) { return (int)(v < 1 ? 1 : (v > hi ? hi : v)); };
  nc = K >= 2048 ? clamp(N / 1024, 3) : 1;
  nb = clamp(M / 1024, nc > 1 ? 3 : 4);
}

int64_t env_int(const char *name, int64_t dflt) {
  const char *v = std::getenv(name);
  return (v && *v) ? std::atoll(v) : dflt;
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

// Streaming form of the call, for a product that resolves to the
// tensor-core kernel with A split on chip: B is copied in whole, then A (and
// C, when beta != 0) in row blocks of `rows` rows, each followed by a write of
// `epoch` to its in_flag from the copy stream; one GEMM launch over the whole
// product (one CTA per tile, tiles in row order) runs once B is in and its
// CTAs wait, tile by tile, for their rows (GemmArgs::in_flag); the GEMM
// publishes each row block of C in out_flag once all its tiles are stored,
// and the copy-back stream waits for that value before copying the block
// out.  So the copies in, the GEMM and the copies out overlap with one
// launch's efficiency instead of one GEMM call per block.
int host_streaming(HostPipe &pp, const gemm_plan_t &plan, int64_t M, int64_t N, int64_t K,
                   float alpha, const float *A, int64_t lda, const float *B, int64_t ldb,
                   float beta, float *C, int64_t ldc, int bmode, int64_t rows) {
  const int nblk = (int)ceil_div(M, rows);
  const size_t a_bytes = align256((size_t)M * K * 4), b_bytes = align256((size_t)K * N * 4);
  const size_t c_bytes = align256((size_t)M * N * 4);
  const size_t ws_bytes = align256((size_t)plan.workspace_bytes);
  int st = reserve(pp, a_bytes + b_bytes + c_bytes + ws_bytes);
  if (st != GEMM_OK) return st;
  char *base = static_cast<char *>(pp.buf);
  float *dA = reinterpret_cast<float *>(base);
  float *dB = reinterpret_cast<float *>(base + a_bytes);
  float *dC = reinterpret_cast<float *>(base + a_bytes + b_bytes);
  char *ws = ws_bytes ? base + a_bytes + b_bytes + c_bytes : nullptr;
  unsigned *in_flag = pp.flags, *out_flag = pp.flags + kMaxStreamBlocks;
  unsigned *tile_cnt = pp.flags + 2 * kMaxStreamBlocks;
  if (++pp.epoch == 0) ++pp.epoch;  // flags start at 0: never publish 0
  const unsigned epoch = pp.epoch;
  auto rows_of = [&](int i) { return i + 1 < nblk ? rows : M - (int64_t)i * rows; };

  // test hook: the arrival of this row block is never published, so the
  // GEMM's waits for it run out (GEMM_DEBUG_WAIT_LIMIT_NS bounds them)
  const int64_t skip = env_int("GEMM_DEBUG_STREAM_SKIP_BLOCK", -1);
  cudaError_t e = copy_rows(dB, N, B, ldb, N, K, cudaMemcpyHostToDevice, pp.h2d);
  if (e == cudaSuccess) e = cudaEventRecord(pp.in, pp.h2d);
  for (int i = 0; i < nblk && e == cudaSuccess; ++i) {
    const int64_t r0 = (int64_t)i * rows, nr = rows_of(i);
    e = copy_rows(dA + r0 * K, K, A + r0 * lda, lda, K, nr, cudaMemcpyHostToDevice, pp.h2d);
    if (e == cudaSuccess && beta != 0.0f)
      e = copy_rows(dC + r0 * N, N, C + r0 * ldc, ldc, N, nr, cudaMemcpyHostToDevice, pp.h2d);
    if (e == cudaSuccess && i != skip &&
        g_write32(reinterpret_cast<CUstream>(pp.h2d), reinterpret_cast<CUdeviceptr>(in_flag + i),
                  epoch, CU_STREAM_WRITE_VALUE_DEFAULT) != CUDA_SUCCESS)
      e = cudaErrorUnknown;
  }
  if (e == cudaSuccess) e = cudaMemsetAsync(tile_cnt, 0, (size_t)nblk * sizeof(unsigned), pp.comp);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(pp.comp, pp.in, 0);
  bool launched = false;
  if (e == cudaSuccess) {
    GemmArgs g{M, N, K, alpha, beta, dA, K, dB, N, dC, N};
    g.plain_order = 1;
    g.in_flag = in_flag;
    g.out_flag = out_flag;
    g.tile_cnt = tile_cnt;
    g.epoch = epoch;
    g.stream_rows = rows;
    g.stream_blocks = nblk;
    st = run_gemm(g, bmode, ws, ws_bytes, pp.comp);
    launched = st == GEMM_OK;
  }
  // copies back, each behind its block's flag (only once the GEMM is
  // launched: nothing else would ever set the flags)
  for (int i = 0; launched && i < nblk && e == cudaSuccess; ++i) {
    const int64_t r0 = (int64_t)i * rows;
    if (g_wait32(reinterpret_cast<CUstream>(pp.d2h), reinterpret_cast<CUdeviceptr>(out_flag + i),
                 epoch, CU_STREAM_WAIT_VALUE_GEQ) != CUDA_SUCCESS) {
      e = cudaErrorUnknown;
      break;
    }
    e = copy_rows(C + r0 * ldc, ldc, dC + r0 * N, N, N, rows_of(i), cudaMemcpyDeviceToHost, pp.d2h);
  }
  if (e != cudaSuccess) {
    cudaGetLastError();
    if (st == GEMM_OK) st = GEMM_ERR_CUDA;
  }
  // The copies in and the GEMM always finish (the GEMM's waits are
  // bounded).  Once the GEMM has, every out_flag is written again from a
  // stream of its own, so a copy back still waiting on a block the GEMM did
  // not publish goes ahead instead of waiting for ever; then the copies back
  // are waited for.
  const cudaError_t e1 = cudaStreamSynchronize(pp.h2d);
  const cudaError_t e2 = cudaStreamSynchronize(pp.comp);
  bool released = true;
  for (int i = 0; i < nblk; ++i)
    released = released &&
               g_write32(reinterpret_cast<CUstream>(pp.rescue),
                         reinterpret_cast<CUdeviceptr>(out_flag + i), epoch,
                         CU_STREAM_WRITE_VALUE_DEFAULT) == CUDA_SUCCESS;
  const cudaError_t e3 = cudaStreamSynchronize(pp.rescue);
  const cudaError_t e4 = cudaStreamSynchronize(pp.d2h);
  if (e1 != cudaSuccess || e2 != cudaSuccess || e3 != cudaSuccess || e4 != cudaSuccess ||
      !released) {
    cudaGetLastError();
    if (st == GEMM_OK) st = GEMM_ERR_CUDA;
  }
  const int dev_st = tc_read_and_clear_status(pp.comp);
  return st != GEMM_OK ? st : dev_st;
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
  if (alpha == 0.0f) K = 0;  // BLAS: A and B are not read, C <- beta * C

  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_NO_DEVICE;
  }
  if (dev < 0 || dev >= kMaxDev) return GEMM_ERR_UNSUPPORTED;
  const DeviceProps &dp = props_of(dev);

  // The streaming form, on request (GEMM_HOST_STREAM = 1), when the library
  // picks the blocking and the product resolves to the tensor-core kernel
  // with A split on chip (A staged with K floats a row, so K % 4 == 0 for
  // TMA); rows in blocks of whole tile rows, about 8 of them
  // (GEMM_HOST_STREAM_ROWS = rows per block).  Measured per call on GB300,
  // blocked / streaming (ms): 4096^3 1.044 / 0.984, 6144^3 2.63 / 2.37, but
  // 4096 x 4096 x 2048 0.648 / 0.704, 8192^3 4.85 / 5.14, 2048^3 0.315 /
  // 0.353, 3072^3 0.614 / 0.622: the whole of B has to arrive before the
  // one launch starts, which the blocked form does not wait for, so it is
  // not the default.
  if (blocks == 0 && K > 0 && (K & 3) == 0 && env_int("GEMM_HOST_STREAM", 0) != 0 &&
      memops()) {
    gemm_plan_t ps;
    if (make_plan(M, N, K, K, N, N, mode, 0, beta != 0.0f, dp, &ps) == GEMM_OK &&
        tc_plan_streaming(ps, M, N, K) && M >= 2 * ps.bm) {
      int64_t rows = env_int("GEMM_HOST_STREAM_ROWS", ceil_div(M, 8));
      rows = ceil_div(rows < ps.bm ? ps.bm : rows, ps.bm) * ps.bm;
      if (ceil_div(M, rows) > kMaxStreamBlocks) rows = ceil_div(ceil_div(M, kMaxStreamBlocks), ps.bm) * ps.bm;
      std::lock_guard<std::mutex> lk(g_host_mu[dev]);
      HostPipe &pp = g_pipe[dev];
      st = setup(pp);
      if (st != GEMM_OK) return st;
      return host_streaming(pp, ps, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, ps.mode, rows);
    }
  }

  // Row blocks hold whole 128-row tiles and column blocks whole 256-column
  // tiles, except the last of each.  Column blocks only when the library
  // picks the blocking (blocks == 0); tuning knob GEMM_HOST_COL_BLOCKS.
  int auto_nb, auto_nc;
  auto_grid(M, N, K, auto_nb, auto_nc);
  int nb = blocks > 0 ? blocks : auto_nb;
  int64_t rows = ceil_div(M, nb);
  if (M > 128) rows = ceil_div(rows, 128) * 128;
  nb = (int)ceil_div(M, rows);
  int nc = (int)env_int("GEMM_HOST_COL_BLOCKS", blocks > 0 ? 1 : auto_nc);
  if (nc < 1) nc = 1;
  if (nc > kMaxColBlocks) nc = kMaxColBlocks;
  int64_t cols = ceil_div(N, nc);
  if (N > 256) cols = ceil_div(cols, 256) * 256;
  nc = (int)ceil_div(N, cols);
  const int64_t kld = K > 1 ? K : 1, nld = N > 1 ? N : 1;
  auto rows_of = [&](int64_t i) { return i + 1 < nb ? rows : M - i * rows; };
  auto cols_of = [&](int64_t j) { return j + 1 < nc ? cols : N - j * cols; };

  // Arrival order: B column block 0, A row block 0, then whichever of A and
  // B has the smaller arrived fraction.  Each arrival enables GEMMs: a new A
  // row block i against each arrived column block, a new column block j
  // against rows [0, i_arrived * rows) in one call.
  struct Gemm {
    int64_t r0, nr;
    int j;
  };
  struct Arrival {
    bool is_a;
    int idx;
    std::vector<Gemm> gemms;
  };
  std::vector<Arrival> order;
  {
    int ia = 0, jb = 0;
    while (ia < nb || jb < nc) {
      const bool take_a = jb > 0 && ia < nb && (jb >= nc || (double)ia / nb <= (double)jb / nc);
      Arrival ar{take_a, take_a ? ia : jb, {}};
      if (take_a) {
        for (int j = 0; j < jb; ++j) ar.gemms.push_back(Gemm{ia * rows, rows_of(ia), j});
        ++ia;
      } else {
        if (ia > 0) ar.gemms.push_back(Gemm{0, (int64_t)ia * rows < M ? (int64_t)ia * rows : M, jb});
        ++jb;
      }
      order.push_back(ar);
    }
  }

  // one mode for every GEMM: the one the whole product resolves to
  gemm_plan_t whole;
  st = make_plan(M, N, K, kld, nld, nld, mode, 0, beta != 0.0f, dp, &whole);
  if (st != GEMM_OK) return st;
  const int bmode = (mode == GEMM_MODE_AUTO && K > 0) ? whole.mode : mode;
  size_t ws_bytes = 0;
  bool tc = false;
  for (const Arrival &ar : order)
    for (const Gemm &g : ar.gemms) {
      gemm_plan_t pg;
      st = make_plan(g.nr, cols_of(g.j), K, kld, nld, nld, bmode, 0, beta != 0.0f, dp, &pg);
      if (st != GEMM_OK) return st;
      if ((size_t)pg.workspace_bytes > ws_bytes) ws_bytes = (size_t)pg.workspace_bytes;
      tc = tc || pg.kernel == GEMM_KERNEL_TC_TF32X3 || pg.kernel == GEMM_KERNEL_TC_TF32;
    }
  ws_bytes = align256(ws_bytes);

  const size_t a_bytes = align256((size_t)M * K * 4), b_bytes = align256((size_t)K * N * 4);
  const size_t c_bytes = align256((size_t)M * N * 4);

  std::lock_guard<std::mutex> lk(g_host_mu[dev]);
  HostPipe &pp = g_pipe[dev];
  st = setup(pp);
  if (st == GEMM_OK) st = reserve(pp, a_bytes + b_bytes + c_bytes + (size_t)nc * ws_bytes);
  if (st != GEMM_OK) return st;
  char *base = static_cast<char *>(pp.buf);
  float *dA = reinterpret_cast<float *>(base);
  float *dB = reinterpret_cast<float *>(base + a_bytes);
  float *dC = reinterpret_cast<float *>(base + a_bytes + b_bytes);
  char *ws0 = base + a_bytes + b_bytes + c_bytes;  // column block j: ws0 + j * ws_bytes

  cudaError_t e = cudaSuccess;
  // per column block: its B planes are in that block's workspace (written by
  // an earlier GEMM of the column that split B with the pass; GEMMs that
  // split B on chip write none, and the next one that needs them writes them)
  int planes[kMaxColBlocks] = {};
  for (const Arrival &ar : order) {
    if (e != cudaSuccess || st != GEMM_OK) break;
    if (ar.is_a) {
      const int64_t r0 = (int64_t)ar.idx * rows, nr = rows_of(ar.idx);
      if (K > 0)
        e = copy_rows(dA + r0 * kld, kld, A + r0 * lda, lda, K, nr, cudaMemcpyHostToDevice,
                      pp.h2d);
      if (e == cudaSuccess && beta != 0.0f)
        e = copy_rows(dC + r0 * nld, nld, C + r0 * ldc, ldc, N, nr, cudaMemcpyHostToDevice,
                      pp.h2d);
    } else if (K > 0) {
      const int64_t c0 = (int64_t)ar.idx * cols;
      e = copy_rows(dB + c0, nld, B + c0, ldb, cols_of(ar.idx), K, cudaMemcpyHostToDevice,
                    pp.h2d);
    }
    if (ar.gemms.empty()) continue;
    if (e == cudaSuccess) e = cudaEventRecord(pp.in, pp.h2d);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(pp.comp, pp.in, 0);
    for (const Gemm &gm : ar.gemms) {
      if (e != cudaSuccess || st != GEMM_OK) break;
      const int64_t c0 = (int64_t)gm.j * cols, w = cols_of(gm.j);
      GemmArgs g{gm.nr, w, K, alpha, beta, dA + gm.r0 * kld, kld, dB + c0, nld,
                 dC + gm.r0 * nld + c0, nld};
      g.b_presplit = (tc && planes[gm.j]) ? 1 : 0;
      g.b_planes_written = &planes[gm.j];
      g.plain_order = 1;
      st = run_gemm(g, bmode, ws_bytes ? ws0 + (size_t)gm.j * ws_bytes : nullptr, ws_bytes,
                    pp.comp);
      if (st != GEMM_OK) break;
      e = cudaEventRecord(pp.out, pp.comp);
      if (e == cudaSuccess) e = cudaStreamWaitEvent(pp.d2h, pp.out, 0);
      if (e == cudaSuccess)
        e = copy_rows(C + gm.r0 * ldc + c0, ldc, dC + gm.r0 * nld + c0, nld, w, gm.nr,
                      cudaMemcpyDeviceToHost, pp.d2h);
    }
  }
  if (e != cudaSuccess) {
    cudaGetLastError();
    if (st == GEMM_OK) st = GEMM_ERR_CUDA;
  }
  st = drain(pp, st);
  const int dev_st = tc ? tc_read_and_clear_status(pp.comp) : GEMM_OK;
  return st != GEMM_OK ? st : dev_st;
}
