// Register-tiled FP32 SGEMM on the CUDA cores (sm_103a).
//
// This is the step the tiled-matmul course page leaves for later ("Project -
// tiled matrix multiply", sections "The results table" and "What comes
// next"): each thread computes an 8 x 8 output tile held in registers, the
// next shared-memory tiles are fetched while the current one is consumed,
// and global traffic moves in wide asynchronous copies.
//
// One CTA: 128 threads as 1 x 4 warps, output tile 64 (M) x 128 (N), K in
// 16-deep stages of a 4-stage cp.async ring (~53 KB of shared memory, two
// CTAs per SM).  A warp covers 64 x 32 outputs with its lanes in an 8 x 4
// grid; a thread's 8 x 8 tile is four 4 x 4 blocks spaced 32 rows and 16
// columns apart, so each k step reads its A and B fragments with four
// 128-bit shared loads that the warp serves in one wavefront each.
// Accumulators are column pairs updated with packed f32x2 FMAs (two FMAs per
// issued instruction, each rounded as a scalar FFMA would be).
// A is K-contiguous in global memory but the inner product wants it
// M-contiguous, so it is the operand that gets transposed: copied element
// by element into a k-major tile whose rows are 68 floats apart, with lanes
// arranged 8 (k) x 4 (rows) so one warp instruction reads four 32-byte
// sectors and writes 32 distinct banks.  B is already N-contiguous and moves
// in 16-byte copies.  The copies' source-size operand zero-fills elements
// outside the matrices; stores outside C are skipped (the course page's edge
// handling in "Stage 2").
// Transposed storage (A stored K x M, B stored N x K) swaps the two copy
// kinds per operand: an M- or N-contiguous operand moves in 16-byte copies,
// a K-contiguous one is scattered element by element into padded rows.
// Split-K: grid.z slices K; slices write raw partial sums to the workspace
// and splitk_reduce applies alpha/beta, summing slices in a fixed order.
//
// (Measured on GB300 while choosing this layout: transposing the 128-row
// operand with 8-row-spread copies caused 2x the shared-memory wavefronts and
// ran at 46 TFLOP/s; the earlier register-staged 128 x 128 x 16 kernel with
// scalar FFMA reached 51-53 TFLOP/s; this one reaches 58.8 at 4096^3 and
// 62.3 at 8192^3.)
#include <cstdlib>

#include "common.cuh"

namespace gg {
namespace {

__device__ __forceinline__ void cp_async4(void *smem, const void *gmem, bool valid) {
  const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(s), "l"(gmem),
               "r"(valid ? 4 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
  const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem) : "memory");
}
// Programmatic dependent launch: wait until the kernel before this one in
// the stream has finished and its writes are visible / let the next kernel
// be scheduled (it waits the same way before touching memory).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

constexpr int kThreadsP = 128;
// Row-tiles per column sweep (tile order).  GB300, 8192^3: 8 cuts the
// kernel's DRAM traffic from 27 GB to ~3 GB at the same speed when B is
// stored K x N; with B stored N x K plain row order (1) is 3-4 % faster.
constexpr int kGroupM = 8;

// Three CTAs per SM (12 warps): 150 registers a thread fit 3 x 128 threads in
// the SM's 65536 (capping at 128 registers for four spills and ran 2-10 %
// slower on GB300).
template <int BM, int BN, int BK, int STAGES, bool VEC, bool TA, bool TB>
__global__ void __launch_bounds__(kThreadsP, 3)
simt_packed_kernel(GemmArgs p, int64_t k_per_split, float *__restrict__ ws, int ws_vec,
                   int group_m, unsigned long long *stamps) {
  constexpr int TM = 8, TN = 8;
  // k-major tiles As[k][m], Bs[k][n].  An operand stored with K contiguous (A
  // as M x K, or B as N x K) is copied element by element into rows of
  // (tile width + 4) floats: an odd multiple of 4, so a warp's 8 k x 4 rows
  // scatter lands in 32 distinct banks.  An operand stored with M or N
  // contiguous moves in 16-byte copies into unpadded-width rows.
  constexpr int LDA_S = BM + 4;
  constexpr int LDB_S = BN + (TB ? 4 : 0);
  constexpr int WTM = TM * 8;   // 64
  constexpr int WTN = TN * 4;   // 32
  constexpr int WARPS_N = BN / WTN;
  static_assert((BM / WTM) * WARPS_N * 32 == kThreadsP, "warp grid must cover the CTA");
  static_assert(BK % 8 == 0, "element copies go 8 k at a time");
  // element copy e: k = 8 * (e / (8 * rows)) + e % 8, row = (e / 8) % rows, so
  // one warp instruction reads 4 rows x 32 contiguous bytes.
  // vector copy e: k = e / (cols / 4), first column = 4 * (e % (cols / 4)).
  constexpr int A_COPIES = TA ? BK * BM / 4 : BM * BK;
  constexpr int B_COPIES = TB ? BK * BN : BK * BN / 4;
  static_assert(A_COPIES % kThreadsP == 0 && B_COPIES % kThreadsP == 0, "whole copies per thread");
  static_assert(BM % 16 == 0 && BN % 16 == 0 && 512 % BM == 0 && 512 % BN == 0 &&
                BM / 16 <= 32 && BN / 16 <= 32, "copy strides below assume these tile sizes");
  constexpr int A_PER_T = A_COPIES / kThreadsP;
  constexpr int B_PER_T = B_COPIES / kThreadsP;

  extern __shared__ __align__(16) float smp[];
  float(*As)[BK][LDA_S] = reinterpret_cast<float(*)[BK][LDA_S]>(smp);
  float(*Bs)[BK][LDB_S] = reinterpret_cast<float(*)[BK][LDB_S]>(smp + STAGES * BK * LDA_S);

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int wm = warp / WARPS_N, wn = warp % WARPS_N;
  const int lr = lane >> 2, lc = lane & 3;
  // Tile order: CTAs are issued in blockIdx order; consecutive ones take
  // group_m row-tiles of one column-tile before moving right, so the CTAs
  // resident at one time share a band of A rows and a band of B columns
  // (both held in L2) instead of sweeping every column of B per row band.
  // group_m = 1 is plain row order.
  const int64_t tiles_n = gridDim.x, tiles_m = gridDim.y;
  const int64_t id = (int64_t)blockIdx.y * tiles_n + blockIdx.x;
  const int64_t first_m = (id / (group_m * tiles_n)) * group_m;
  const int64_t gm = min(tiles_m - first_m, (int64_t)group_m);
  const int64_t local = id % (group_m * tiles_n);
  const int64_t m0 = (first_m + local % gm) * BM;
  const int64_t n0 = (local / gm) * BN;
  pdl_wait();  // A, B and C may come from the kernel before this one
  // measurement aid: earliest start of any CTA (see gemm_set_profile_stamps)
  if (stamps != nullptr && tid == 0) atomicMin(&stamps[0], globaltimer_ns());
  const int64_t kbeg = (int64_t)blockIdx.z * k_per_split;
  const int64_t kend = min(p.K, kbeg + k_per_split);
  const int64_t klen = kend > kbeg ? kend - kbeg : 0;
  const int ntiles = (int)((klen + BK - 1) / BK);

  // Copies.  Copy j of this thread (e = tid + 128 j of the stage's copies)
  // reaches, for each operand, one base pointer plus a fixed stride:
  //   element copies of A stored M x K: row a_r0 + 16 (j % AJ), k a_k0 +
  //     8 (j / AJ), AJ = BM / 16;  16-byte copies of A stored K x M: k row
  //     a_r0 + (512 / BM) j, columns a_q .. a_q + 3;
  //   16-byte copies of B stored K x N: k row b_r0 + (512 / BN) j, columns
  //     b_q .. b_q + 3;  element copies of B stored N x K: column b_r0 +
  //     16 (j % BJ), k b_k0 + 8 (j / BJ), BJ = BN / 16.
  // A bit mask (element copies) or a count of in-range columns (16-byte
  // copies) says which lie inside the matrix; pointers to the rest are
  // formed but never read (the copy's source size is 0).  Holding one base
  // per operand instead of one pointer per copy keeps the registers for the
  // accumulators.
  constexpr int AJ = BM / 16, BJ = BN / 16;
  const float *a_base;
  uint32_t a_mask = 0;
  int a_cols = 0, a_r0, a_k0 = 0;
  if (!TA) {
    a_r0 = tid / 8;
    a_k0 = tid % 8;
#pragma unroll
    for (int j = 0; j < AJ; ++j)
      if (m0 + a_r0 + 16 * j < p.M) a_mask |= 1u << j;
    a_base = p.A + (m0 + a_r0) * p.lda + kbeg + a_k0;
  } else {
    a_r0 = tid / (BM / 4);
    const int64_t a_q = (tid % (BM / 4)) * 4, left = p.M - (m0 + a_q);
    a_cols = (int)(left > 4 ? 4 : (left < 0 ? 0 : left));
    a_base = p.A + (kbeg + a_r0) * p.lda + m0 + a_q;
  }
  const float *b_base;
  uint32_t b_mask = 0;
  int b_cols = 0, b_r0, b_k0 = 0;
  if (!TB) {
    b_r0 = tid / (BN / 4);
    const int64_t b_q = (tid % (BN / 4)) * 4, left = p.N - (n0 + b_q);
    b_cols = (int)(left > 4 ? 4 : (left < 0 ? 0 : left));
    b_base = p.B + (kbeg + b_r0) * p.ldb + n0 + b_q;
  } else {
    b_r0 = tid / 8;
    b_k0 = tid % 8;
#pragma unroll
    for (int j = 0; j < BJ; ++j)
      if (n0 + b_r0 + 16 * j < p.N) b_mask |= 1u << j;
    b_base = p.B + (n0 + b_r0) * p.ldb + kbeg + b_k0;
  }
  const int a_q = TA ? (tid % (BM / 4)) * 4 : 0;
  const int b_q = TB ? 0 : (tid % (BN / 4)) * 4;

  // copy c of the stage of tile t: A's copies first, then B's
  auto issue_copy = [&](int t, int c) {
    const int buf = t % STAGES;
    const int rem = (int)min(klen - (int64_t)t * BK, (int64_t)BK);
    if (c < A_PER_T) {
      const int j = c;
      if (!TA) {
        const int jr = j % AJ, jk = j / AJ;
        const int kk = a_k0 + 8 * jk;
        const bool ok = ((a_mask >> jr) & 1u) && kk < rem;
        const float *src = a_base + (int64_t)(16 * jr) * p.lda + (int64_t)t * BK + 8 * jk;
        cp_async4(&As[buf][kk][a_r0 + 16 * jr], ok ? src : p.A, ok);
      } else {
        const int kr = a_r0 + (512 / BM) * j;
        const float *src = a_base + ((int64_t)t * BK + (512 / BM) * j) * p.lda;
        float *dst = &As[buf][kr][a_q];
        const bool row_ok = kr < rem;
        if (VEC && row_ok && a_cols == 4) {
          cp_async16(dst, src);
        } else {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const bool ok = row_ok && i < a_cols;
            cp_async4(dst + i, ok ? src + i : p.A, ok);
          }
        }
      }
    } else {
      const int j = c - A_PER_T;
      if (!TB) {
        const int kr = b_r0 + (512 / BN) * j;
        const float *src = b_base + ((int64_t)t * BK + (512 / BN) * j) * p.ldb;
        float *dst = &Bs[buf][kr][b_q];
        const bool row_ok = kr < rem;
        if (VEC && row_ok && b_cols == 4) {
          cp_async16(dst, src);
        } else {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const bool ok = row_ok && i < b_cols;
            cp_async4(dst + i, ok ? src + i : p.B, ok);
          }
        }
      } else {
        const int jr = j % BJ, jk = j / BJ;
        const int kk = b_k0 + 8 * jk;
        const bool ok = ((b_mask >> jr) & 1u) && kk < rem;
        const float *src = b_base + (int64_t)(16 * jr) * p.ldb + (int64_t)t * BK + 8 * jk;
        cp_async4(&Bs[buf][kk][b_r0 + 16 * jr], ok ? src : p.B, ok);
      }
    }
  };
  constexpr int NCOPY = A_PER_T + B_PER_T;
  auto issue = [&](int t) {
#pragma unroll
    for (int c = 0; c < NCOPY; ++c) issue_copy(t, c);
  };

  float2 acc[TM][TN / 2];
#pragma unroll
  for (int i = 0; i < TM; ++i)
#pragma unroll
    for (int j = 0; j < TN / 2; ++j) acc[i][j] = make_float2(0.f, 0.f);
  const int a_off = wm * WTM + lr * 4;
  const int b_off = wn * WTN + lc * 4;

#pragma unroll
  for (int t = 0; t < STAGES - 1; ++t) {
    if (t < ntiles) issue(t);
    cp_async_commit();
  }
  for (int t = 0; t < ntiles; ++t) {
    cp_async_wait<STAGES - 2>();
    __syncthreads();  // tile t landed for everyone; tile t-1's buffer is free
    if (t + STAGES - 1 < ntiles) issue(t + STAGES - 1);
    cp_async_commit();
    const int cur = t % STAGES;
#pragma unroll
    for (int k = 0; k < BK; ++k) {
      float2 b[TN / 2];
#pragma unroll
      for (int in = 0; in < TN / 4; ++in) {
        const float4 v = *reinterpret_cast<const float4 *>(&Bs[cur][k][b_off + in * 16]);
        b[2 * in] = make_float2(v.x, v.y);
        b[2 * in + 1] = make_float2(v.z, v.w);
      }
      float a[TM];
#pragma unroll
      for (int im = 0; im < TM / 4; ++im)
        *reinterpret_cast<float4 *>(&a[im * 4]) =
            *reinterpret_cast<const float4 *>(&As[cur][k][a_off + im * 32]);
#pragma unroll
      for (int i = 0; i < TM; ++i) {
        const float2 aa = make_float2(a[i], a[i]);
#pragma unroll
        for (int j = 0; j < TN / 2; ++j) acc[i][j] = __ffma2_rn(aa, b[j], acc[i][j]);
      }
    }
  }
  cp_async_wait<0>();
  pdl_trigger();  // the split-K reduction (or the next call) may be scheduled

#pragma unroll
  for (int i = 0; i < TM; ++i) {
    const int64_t row = m0 + a_off + (i / 4) * 32 + (i % 4);
    if (row >= p.M) continue;
#pragma unroll
    for (int jn = 0; jn < TN / 4; ++jn) {
      const int64_t col = n0 + b_off + jn * 16;
      const float v[4] = {acc[i][jn * 2].x, acc[i][jn * 2].y, acc[i][jn * 2 + 1].x,
                          acc[i][jn * 2 + 1].y};
      if (ws != nullptr) {
        float *dst = ws + (int64_t)blockIdx.z * p.M * p.N + row * p.N + col;
        if (ws_vec && col + 4 <= p.N) {
          *reinterpret_cast<float4 *>(dst) = make_float4(v[0], v[1], v[2], v[3]);
        } else {
#pragma unroll
          for (int q = 0; q < 4; ++q)
            if (col + q < p.N) dst[q] = v[q];
        }
        continue;
      }
      float *dst = p.C + row * p.ldc + col;
      if (VEC && col + 4 <= p.N) {
        float4 o = make_float4(p.alpha * v[0], p.alpha * v[1], p.alpha * v[2], p.alpha * v[3]);
        if (p.beta != 0.0f) {
          const float4 c = *reinterpret_cast<const float4 *>(dst);
          o.x = fmaf(p.beta, c.x, o.x);
          o.y = fmaf(p.beta, c.y, o.y);
          o.z = fmaf(p.beta, c.z, o.z);
          o.w = fmaf(p.beta, c.w, o.w);
        }
        *reinterpret_cast<float4 *>(dst) = o;
      } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          if (col + q < p.N) {
            float o = p.alpha * v[q];
            if (p.beta != 0.0f) o = fmaf(p.beta, dst[q], o);
            dst[q] = o;
          }
        }
      }
    }
  }
  if (stamps != nullptr) {  // latest end of any CTA
    __syncthreads();
    if (tid == 0) atomicMax(&stamps[1], globaltimer_ns());
  }
}

// C <- alpha * sum_{z < splits} ws[z] + beta * C.  Slice z goes to chain
// z % 8 (each chain summed in z order), then the chains are combined in a
// fixed tree, so the result does not depend on timing; the eight chains keep
// eight loads in flight per thread, which matters with many slices and a
// small C (32 x 32 x 65536 uses 241 slices).
__global__ void splitk_reduce_kernel(GemmArgs p, const float *__restrict__ ws, int splits) {
  pdl_wait();  // the GEMM's slices
  pdl_trigger();
  const int64_t total = p.M * p.N;
  for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < total;
       t += (int64_t)gridDim.x * blockDim.x) {
    float c[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    int z = 0;
    for (; z + 8 <= splits; z += 8) {
      float v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) v[u] = ws[(int64_t)(z + u) * total + t];
#pragma unroll
      for (int u = 0; u < 8; ++u) c[u] += v[u];
    }
#pragma unroll
    for (int u = 0; u < 8; ++u)
      if (z + u < splits) c[u] += ws[(int64_t)(z + u) * total + t];
    const float s = ((c[0] + c[1]) + (c[2] + c[3])) + ((c[4] + c[5]) + (c[6] + c[7]));
    const int64_t r = t / p.N, col = t % p.N;
    float *dst = p.C + r * p.ldc + col;
    float o = p.alpha * s;
    if (p.beta != 0.0f) o = fmaf(p.beta, *dst, o);
    *dst = o;
  }
}

}  // namespace

SimtConfig simt_config() { return SimtConfig{64, 128, 16, kThreadsP}; }

bool simt_config_valid(int bk, int stages) {
#define GG_SIMT(BK_, ST_) \
  if (bk == BK_ && stages == ST_) return true;
  GG_SIMT_CONFIGS(GG_SIMT)
#undef GG_SIMT
  return false;
}

// Launch with the programmatic-dependent-launch attribute unless the caller
// needs plain stream order (profiling events around the main kernel, or
// chaining behind cross-stream event waits).
template <typename... Args>
cudaError_t launch_pdl(void (*kern)(Args...), dim3 grid, dim3 block, size_t smem, bool pdl,
                       cudaStream_t s, Args... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = grid;
  lc.blockDim = block;
  lc.dynamicSmemBytes = smem;
  lc.stream = s;
  lc.attrs = attr;
  lc.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&lc, kern, args...);
}

cudaError_t launch_splitk_reduce(const GemmArgs &p, const float *ws, int splits, cudaStream_t s) {
  int64_t blocks = ceil_div(p.M * p.N, 256);
  if (blocks > 4096) blocks = 4096;
  const bool pdl = !profile_events_set() && !p.plain_order;
  const cudaError_t e =
      launch_pdl(splitk_reduce_kernel, dim3((unsigned)blocks), dim3(256), 0, pdl, s, p, ws, splits);
  return e != cudaSuccess ? e : cudaGetLastError();
}

template <int BM, int BN, int BK, int STAGES, bool TA, bool TB>
cudaError_t launch_packed(const gemm_plan_t &plan, const GemmArgs &p, float *ws, cudaStream_t s) {
  const int split = plan.split_k > 1 ? plan.split_k : 1;
  int64_t kps = ceil_div(p.K, split);
  kps = ceil_div(kps, BK) * BK;
  dim3 grid((unsigned)ceil_div(p.N, BN), (unsigned)ceil_div(p.M, BM), (unsigned)split);
  float *w = split > 1 ? ws : nullptr;
  const int ws_vec = (p.N % 4 == 0) ? 1 : 0;
  // Tuning knob: GEMM_SIMT_GROUP=g sets the row-tiles per column sweep (>= 1).
  int group_m = TB ? 1 : kGroupM;
  if (const char *g = std::getenv("GEMM_SIMT_GROUP")) {
    const int v = std::atoi(g);
    if (v >= 1) group_m = v;
  }
  constexpr int smem = STAGES * BK * ((BM + 4) + BN + (TB ? 4 : 0)) * 4;
  auto kv = simt_packed_kernel<BM, BN, BK, STAGES, true, TA, TB>;
  auto ks = simt_packed_kernel<BM, BN, BK, STAGES, false, TA, TB>;
  if (smem > 48 * 1024) {
    if (cudaFuncSetAttribute(kv, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess ||
        cudaFuncSetAttribute(ks, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
      return cudaGetLastError();
  }
  // The GEMM kernel itself goes in plain stream order (measured on GB300:
  // with programmatic launch its CTAs wait on SMs the kernel before it still
  // needs; 1023 x 1025 x 777 split 2 went from 57.4 to 71.9 us per call).
  profile_mark_before(s);
  cudaError_t e = launch_pdl(plan.vec ? kv : ks, grid, dim3(kThreadsP), (size_t)smem, false, s,
                             p, kps, w, ws_vec, group_m, profile_stamps());
  profile_mark_after(s);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess || split == 1) return e;
  return launch_splitk_reduce(p, ws, split, s);
}

cudaError_t launch_simt(const gemm_plan_t &plan, const GemmArgs &p, float *ws, cudaStream_t s) {
  if (plan.bm != 64 || plan.bn != 128) return cudaErrorInvalidValue;
#define GG_SIMT(BK_, ST_)                                                              \
  if (plan.bk == BK_ && plan.stages == ST_) {                                          \
    if (!p.ta && !p.tb) return launch_packed<64, 128, BK_, ST_, false, false>(plan, p, ws, s); \
    if (p.ta && !p.tb) return launch_packed<64, 128, BK_, ST_, true, false>(plan, p, ws, s);   \
    if (!p.ta && p.tb) return launch_packed<64, 128, BK_, ST_, false, true>(plan, p, ws, s);   \
    return launch_packed<64, 128, BK_, ST_, true, true>(plan, p, ws, s);                       \
  }
  GG_SIMT_CONFIGS(GG_SIMT)
#undef GG_SIMT
  return cudaErrorInvalidValue;
}

}  // namespace gg
