// Register-tiled FP32 SGEMM on the CUDA cores with a duplicated A tile.
//
// Same CTA tile, thread tile, tile order, split-K and epilogue as the packed
// kernel in simt.cu (64 x 128 outputs, 128 threads, 8 x 8 per thread as
// column pairs, packed f32x2 FMA), with two changes in the inner loop:
//
//  * The f32x2 FMA multiplies a pair of B values by a pair (a, a).  Built
//    from one A value in a register, that pair costs a register move per A
//    value per k step (8 per thread per k, on top of 32 packed FMAs).  Here
//    the copy into shared memory writes every A value twice, next to each
//    other, so the pairs come straight out of 128-bit shared loads: four for
//    A and two for B per k step, and nothing else besides the 32 FMAs.
//  * The fragments of step k+1 are loaded before the FMAs of step k, and
//    the barrier that publishes the next tile comes before the last k step's
//    FMAs, so the loads of the next tile's first fragments overlap them.
//
// Shared-memory layout of one k line of the A tile (64 rows, 2 floats a row,
// plus 4 floats of padding: 132 floats, 4 mod 32): row r = 32*im + 4*lr + q
// (q = 2*h + qb) keeps its pair at 64*im + 32*h + 4*lr + 2*qb.  A thread's
// rows are 32*im + 4*lr + (0..3), so for each (im, h) one 128-bit load gives
// it two pairs, and the 8 distinct lr of a warp read 128 contiguous bytes:
// one wavefront.  The copy writes each element twice with 4-byte cp.async;
// the lanes of one instruction cover 8 k x 2 rows x 2 copies (A stored
// M x K) or 16 rows x 2 copies of one k (A stored K x M), which land in 32
// distinct banks.
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

constexpr int kThreads = 128;
constexpr int kBM = 64, kBN = 128;

template <int BK, int STAGES, bool VEC, bool TA, bool TB>
__global__ void __launch_bounds__(kThreads, 2)
simt_dup_kernel(GemmArgs p, int64_t k_per_split, float *__restrict__ ws, int ws_vec,
                int group_m, unsigned long long *stamps) {
  constexpr int BM = kBM, BN = kBN;
  constexpr int TM = 8, TN = 8;
  static_assert(STAGES >= 3, "the next tile is waited for one k step early");
  static_assert(BK % 8 == 0, "A copies go 8 k at a time");
  constexpr int LDA2 = 2 * BM + 4;              // floats per k line of the pair tile
  constexpr int LDB_S = BN + (TB ? 4 : 0);
  constexpr int A_COPIES = 2 * BM * BK;         // each element twice
  constexpr int B_COPIES = TB ? BK * BN : BK * BN / 4;
  static_assert(A_COPIES % kThreads == 0 && B_COPIES % kThreads == 0, "whole copies per thread");
  constexpr int A_PER_T = A_COPIES / kThreads;  // 16 for BK = 16
  constexpr int B_PER_T = B_COPIES / kThreads;
  // A stored M x K: copy j of a thread takes row group j % 8 and k group j / 8
  constexpr int A_ROWS = TA ? 1 : 8;

  extern __shared__ __align__(16) float smp[];
  float(*As)[BK][LDA2] = reinterpret_cast<float(*)[BK][LDA2]>(smp);
  float(*Bs)[BK][LDB_S] = reinterpret_cast<float(*)[BK][LDB_S]>(smp + STAGES * BK * LDA2);

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int lr = lane >> 2, lc = lane & 3;
  // grouped tile order, as in simt.cu
  const int64_t tiles_n = gridDim.x, tiles_m = gridDim.y;
  const int64_t id = (int64_t)blockIdx.y * tiles_n + blockIdx.x;
  const int64_t first_m = (id / (group_m * tiles_n)) * group_m;
  const int64_t gm = min(tiles_m - first_m, (int64_t)group_m);
  const int64_t local = id % (group_m * tiles_n);
  const int64_t m0 = (first_m + local % gm) * BM;
  const int64_t n0 = (local / gm) * BN;
  pdl_wait();  // A, B and C may come from the kernel before this one
  if (stamps != nullptr && tid == 0) atomicMin(&stamps[0], globaltimer_ns());
  const int64_t kbeg = (int64_t)blockIdx.z * k_per_split;
  const int64_t kend = min(p.K, kbeg + k_per_split);
  const int64_t klen = kend > kbeg ? kend - kbeg : 0;
  const int ntiles = (int)((klen + BK - 1) / BK);

  // ---- A copies: (row, k, copy d) of copy j of this thread, and its slot
  // e = tid + 128 j, lane = e % 32, w = e / 32.
  //   M x K: kk = lane % 8, qb = lane / 8 % 2, d = lane / 16; lr' = w % 8,
  //          h = w / 8 % 2, im = w / 16 % 2, kgroup = w / 32.
  //   K x M: d = lane % 2, qb = lane / 2 % 2, lr' = lane / 4; h = w % 2,
  //          im = w / 2 % 2, k = w / 4.
  // row = 32 im + 4 lr' + 2 h + qb; slot = 64 im + 32 h + 4 lr' + 2 qb + d.
  const float *a_src[A_ROWS];
  int a_ok[A_ROWS];
  int a_slot[A_ROWS];
  int a_k0 = 0;  // M x K: this thread's k within a group of 8
#pragma unroll
  for (int j = 0; j < A_ROWS; ++j) {
    const int e = tid + j * kThreads, ln = e & 31, w = e >> 5;
    int r, slot;
    if (!TA) {
      const int kk = ln & 7, qb = (ln >> 3) & 1, d = ln >> 4;
      const int lrr = w & 7, h = (w >> 3) & 1, im = (w >> 4) & 1;
      r = 32 * im + 4 * lrr + 2 * h + qb;
      slot = 64 * im + 32 * h + 4 * lrr + 2 * qb + d;
      a_k0 = kk;
      a_ok[j] = m0 + r < p.M;
      a_src[j] = p.A + (a_ok[j] ? (m0 + r) * p.lda + kbeg + kk : 0);
    } else {
      const int d = ln & 1, qb = (ln >> 1) & 1, lrr = ln >> 2;
      const int h = w & 1, im = (w >> 1) & 1;
      r = 32 * im + 4 * lrr + 2 * h + qb;
      slot = 64 * im + 32 * h + 4 * lrr + 2 * qb + d;
      a_ok[j] = m0 + r < p.M;
      a_src[j] = p.A + (a_ok[j] ? kbeg * p.lda + m0 + r : 0);
    }
    a_slot[j] = slot;
  }
  const float *b_src[B_PER_T];
  int b_ok[B_PER_T];
#pragma unroll
  for (int s = 0; s < B_PER_T; ++s) {
    const int e = tid + s * kThreads;
    if (!TB) {
      const int kr = e / (BN / 4), cq = (e % (BN / 4)) * 4;
      const int64_t left = p.N - (n0 + cq);
      b_ok[s] = (int)(left > 4 ? 4 : (left < 0 ? 0 : left));
      b_src[s] = p.B + (kbeg + kr < p.K && b_ok[s] > 0 ? (kbeg + kr) * p.ldb + n0 + cq : 0);
    } else {
      const int kk = 8 * (e / (8 * BN)) + e % 8, c = (e / 8) % BN;
      b_ok[s] = n0 + c < p.N;
      b_src[s] = p.B + (b_ok[s] ? (n0 + c) * p.ldb + kbeg + kk : 0);
    }
  }
  const int64_t b_step = TB ? BK : (int64_t)BK * p.ldb;

  auto issue = [&](int t) {
    const int buf = t % STAGES;
    const int rem = (int)min(klen - (int64_t)t * BK, (int64_t)BK);
#pragma unroll
    for (int j = 0; j < A_PER_T; ++j) {
      if (!TA) {
        // row group j % 8, k group j / 8
        const int jr = j % 8, kg = j / 8;
        const int kk = kg * 8 + a_k0;
        const bool ok = a_ok[jr] && kk < rem;
        const float *src = a_src[jr] + (int64_t)t * BK + kg * 8;
        cp_async4(&As[buf][kk][a_slot[jr]], ok ? src : p.A, ok);
      } else {
        // this thread's one row, k = j (plus the warp's offset below)
        const int e = tid + j * kThreads, w = e >> 5;
        const int kk = w >> 2;
        const bool ok = a_ok[0] && kk < rem;
        const float *src = a_src[0] + ((int64_t)t * BK + kk) * p.lda;
        cp_async4(&As[buf][kk][a_slot[0]], ok ? src : p.A, ok);
      }
    }
#pragma unroll
    for (int s = 0; s < B_PER_T; ++s) {
      const int e = tid + s * kThreads;
      const float *src = b_src[s] + (int64_t)t * b_step;
      if (!TB) {
        const int kr = e / (BN / 4), cq = (e % (BN / 4)) * 4;
        float *dst = &Bs[buf][kr][cq];
        const bool row_ok = kr < rem;
        if (VEC && row_ok && b_ok[s] == 4) {
          cp_async16(dst, src);
        } else {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const bool ok = row_ok && i < b_ok[s];
            cp_async4(dst + i, ok ? src + i : p.B, ok);
          }
        }
      } else {
        const int kk = 8 * (e / (8 * BN)) + e % 8, c = (e / 8) % BN;
        const bool ok = b_ok[s] && kk < rem;
        cp_async4(&Bs[buf][kk][c], ok ? src : p.B, ok);
      }
    }
  };

  float2 acc[TM][TN / 2];
#pragma unroll
  for (int i = 0; i < TM; ++i)
#pragma unroll
    for (int j = 0; j < TN / 2; ++j) acc[i][j] = make_float2(0.f, 0.f);
  const int b_off = warp * 32 + lc * 4;

  // fragments of one k step: 8 (a, a) pairs (rows 32 im + 4 lr + q, pair
  // index 4 im + q) and 4 B pairs (columns b_off + {0,1}, {2,3}, 16 + ...)
  float2 af[2][TM], bf[2][TN / 2];
  auto load_frag = [&](int buf, int k, int slot) {
    const float *line = &As[buf][k][0];
#pragma unroll
    for (int im = 0; im < 2; ++im)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const float4 v = *reinterpret_cast<const float4 *>(line + 64 * im + 32 * h + 4 * lr);
        af[slot][4 * im + 2 * h] = make_float2(v.x, v.y);
        af[slot][4 * im + 2 * h + 1] = make_float2(v.z, v.w);
      }
#pragma unroll
    for (int in = 0; in < 2; ++in) {
      const float4 v = *reinterpret_cast<const float4 *>(&Bs[buf][k][b_off + 16 * in]);
      bf[slot][2 * in] = make_float2(v.x, v.y);
      bf[slot][2 * in + 1] = make_float2(v.z, v.w);
    }
  };

#pragma unroll
  for (int t = 0; t < STAGES - 1; ++t) {
    if (t < ntiles) issue(t);
    cp_async_commit();
  }
  if (ntiles > 0) {
    cp_async_wait<STAGES - 2>();
    __syncthreads();  // tile 0 landed for everyone
    load_frag(0, 0, 0);
  }
  for (int t = 0; t < ntiles; ++t) {
    const int cur = t % STAGES;
#pragma unroll
    for (int k = 0; k < BK; ++k) {
      if (k < BK - 1) {
        load_frag(cur, k + 1, (k + 1) & 1);
      } else if (t + 1 < ntiles) {
        // tile t+1 landed for everyone, and everyone is past tile t-1, whose
        // buffer the next copy overwrites
        cp_async_wait<STAGES - 3>();
        __syncthreads();
        if (t + STAGES - 1 < ntiles) issue(t + STAGES - 1);
        cp_async_commit();
        load_frag((t + 1) % STAGES, 0, (k + 1) & 1);
      }
      const int sl = k & 1;
#pragma unroll
      for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN / 2; ++j) acc[i][j] = __ffma2_rn(af[sl][i], bf[sl][j], acc[i][j]);
    }
  }
  cp_async_wait<0>();
  pdl_trigger();  // the split-K reduction (or the next call) may be scheduled

  const int a_off = lr * 4;
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
  if (stamps != nullptr) {
    __syncthreads();
    if (tid == 0) atomicMax(&stamps[1], globaltimer_ns());
  }
}

template <typename... Args>
cudaError_t launch_plain(void (*kern)(Args...), dim3 grid, dim3 block, size_t smem,
                         cudaStream_t s, Args... args) {
  cudaLaunchConfig_t lc = {};
  lc.gridDim = grid;
  lc.blockDim = block;
  lc.dynamicSmemBytes = smem;
  lc.stream = s;
  return cudaLaunchKernelEx(&lc, kern, args...);
}

template <int BK, int STAGES, bool TA, bool TB>
cudaError_t launch_dup(const gemm_plan_t &plan, const GemmArgs &p, float *ws, cudaStream_t s) {
  const int split = plan.split_k > 1 ? plan.split_k : 1;
  int64_t kps = ceil_div(p.K, split);
  kps = ceil_div(kps, BK) * BK;
  dim3 grid((unsigned)ceil_div(p.N, kBN), (unsigned)ceil_div(p.M, kBM), (unsigned)split);
  float *w = split > 1 ? ws : nullptr;
  const int ws_vec = (p.N % 4 == 0) ? 1 : 0;
  int group_m = TB ? 1 : 8;
  if (const char *g = std::getenv("GEMM_SIMT_GROUP")) {
    const int v = std::atoi(g);
    if (v >= 1) group_m = v;
  }
  constexpr int smem = STAGES * BK * ((2 * kBM + 4) + kBN + (TB ? 4 : 0)) * 4;
  auto kv = simt_dup_kernel<BK, STAGES, true, TA, TB>;
  auto ks = simt_dup_kernel<BK, STAGES, false, TA, TB>;
  if (smem > 48 * 1024) {
    if (cudaFuncSetAttribute(kv, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess ||
        cudaFuncSetAttribute(ks, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
      return cudaGetLastError();
  }
  profile_mark_before(s);
  cudaError_t e = launch_plain(plan.vec ? kv : ks, grid, dim3(kThreads), (size_t)smem, s, p, kps,
                               w, ws_vec, group_m, profile_stamps());
  profile_mark_after(s);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess || split == 1) return e;
  return launch_splitk_reduce(p, ws, split, s);
}

}  // namespace

#define GG_SIMT2_CONFIGS(X) X(16, 4) X(16, 6) X(32, 3)

bool simt2_config_valid(int bk, int stages) {
#define GG_V(BK_, ST_) \
  if (bk == BK_ && stages == ST_) return true;
  GG_SIMT2_CONFIGS(GG_V)
#undef GG_V
  return false;
}

cudaError_t launch_simt2(const gemm_plan_t &plan, const GemmArgs &p, float *ws, cudaStream_t s) {
  if (plan.bm != kBM || plan.bn != kBN) return cudaErrorInvalidValue;
#define GG_L(BK_, ST_)                                                                \
  if (plan.bk == BK_ && plan.stages == ST_) {                                         \
    if (!p.ta && !p.tb) return launch_dup<BK_, ST_, false, false>(plan, p, ws, s);    \
    if (p.ta && !p.tb) return launch_dup<BK_, ST_, true, false>(plan, p, ws, s);      \
    if (!p.ta && p.tb) return launch_dup<BK_, ST_, false, true>(plan, p, ws, s);      \
    return launch_dup<BK_, ST_, true, true>(plan, p, ws, s);                          \
  }
  GG_SIMT2_CONFIGS(GG_L)
#undef GG_L
  return cudaErrorInvalidValue;
}

}  // namespace gg
