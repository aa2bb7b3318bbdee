// Register-tiled FP32 SGEMM on the CUDA cores (sm_103a).
//
// This is the step the tiled-matmul course page leaves for later ("Project -
// tiled matrix multiply", sections "The results table" and "What comes
// next"): each thread computes a TM x TN output tile held in registers
// (8 x 8 here), the next shared-memory tile is fetched while the current
// one is consumed (double buffering), and global loads are 128-bit wide.
//
// Layout of one CTA (BM x BN output tile, 256 threads = 8 warps):
//   * warps form a WARPS_M x WARPS_N grid; a warp covers WTM x WTN outputs
//     with its lanes in an 8 (rows) x 4 (cols) arrangement;
//   * each thread's TM x TN tile is made of 4 x 4 sub-tiles spaced 32 rows
//     and 16 columns apart, so every fragment read is one 128-bit shared
//     load that the warp serves in a single wavefront (A: 8 distinct
//     16-byte chunks, B: 4 distinct chunks broadcast);
//   * A is stored k-major in shared memory (As[k][m], transposed on the way
//     in through registers) with 4 floats of row padding, so the transposing
//     stores of two k-quads land on disjoint bank halves; B keeps its
//     row-major layout (Bs[k][n]).
//   * BK = 16 for the 128 x 128 tile: one barrier per 16 k-steps.  (Measured
//     on GB300: BK = 16 beats BK = 8 by 19% at 4096^3; packed f32x2 FMAs did
//     not beat scalar FFMA at this tile shape, with or without the register
//     headroom of one CTA per SM.)
//   * Out-of-range loads are zero-filled and out-of-range stores skipped
//     (the course page's edge handling in "Stage 2").
// Split-K: grid.z slices K; slices write raw partial sums to the workspace
// and splitk_reduce applies alpha/beta, summing slices in a fixed order.
#include "common.cuh"

namespace gg {
namespace {

constexpr int kThreads = 256;

template <int BM, int BN, int BK, int TM, int TN, bool VEC>
__global__ void __launch_bounds__(kThreads, 2)
simt_sgemm_kernel(GemmArgs p, int64_t k_per_split, float *__restrict__ ws, int ws_vec) {
  constexpr int PAD = 4;
  constexpr int LDA_S = BM + PAD;
  constexpr int WTM = TM * 8;
  constexpr int WTN = TN * 4;
  constexpr int WARPS_N = BN / WTN;
  static_assert((BM / WTM) * WARPS_N * 32 == kThreads, "warp grid must cover the CTA");
  static_assert(TM % 4 == 0 && TN % 4 == 0 && BK % 4 == 0, "4x4 sub-tiles");
  constexpr int A_SLOTS = BM * BK / 4;
  constexpr int B_SLOTS = BK * BN / 4;
  constexpr int A_PER_T = (A_SLOTS + kThreads - 1) / kThreads;
  constexpr int B_PER_T = (B_SLOTS + kThreads - 1) / kThreads;

  __shared__ __align__(16) float As[2][BK][LDA_S];
  __shared__ __align__(16) float Bs[2][BK][BN];

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int wm = warp / WARPS_N, wn = warp % WARPS_N;
  const int lr = lane >> 2, lc = lane & 3;
  const int64_t m0 = (int64_t)blockIdx.y * BM;
  const int64_t n0 = (int64_t)blockIdx.x * BN;
  const int64_t kbeg = (int64_t)blockIdx.z * k_per_split;
  const int64_t kend = min(p.K, kbeg + k_per_split);
  const int64_t ntiles = kend > kbeg ? (kend - kbeg + BK - 1) / BK : 0;

  float4 ra[A_PER_T], rb[B_PER_T];

  // Per-thread source pointers, advanced by one BK tile per iteration.
  const float *a_src[A_PER_T];
  bool a_ok[A_PER_T];
#pragma unroll
  for (int s = 0; s < A_PER_T; ++s) {
    const int slot = tid + s * kThreads;
    const int r = slot / (BK / 4), kq = (slot % (BK / 4)) * 4;
    a_ok[s] = (A_SLOTS % kThreads == 0 || slot < A_SLOTS) && (m0 + r < p.M);
    a_src[s] = p.A + (a_ok[s] ? (m0 + r) * p.lda + kbeg + kq : 0);
  }
  const float *b_src[B_PER_T];
  int b_cols[B_PER_T];  // valid columns from this slot's first column (<= 4 matters)
#pragma unroll
  for (int s = 0; s < B_PER_T; ++s) {
    const int slot = tid + s * kThreads;
    const int kr = slot / (BN / 4), cq = (slot % (BN / 4)) * 4;
    const bool ok = (B_SLOTS % kThreads == 0 || slot < B_SLOTS);
    const int64_t left = p.N - (n0 + cq);
    b_cols[s] = ok ? (int)(left > 4 ? 4 : (left < 0 ? 0 : left)) : 0;
    b_src[s] = p.B + (ok && kbeg + kr < p.K ? (kbeg + kr) * p.ldb + n0 + cq : 0);
  }
  const int64_t b_step = (int64_t)BK * p.ldb;

  // rem: K elements left in this slice from the tile's first k.
  auto load_global = [&](int rem) {
#pragma unroll
    for (int s = 0; s < A_PER_T; ++s) {
      const int slot = tid + s * kThreads;
      const int kq = (slot % (BK / 4)) * 4;
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (a_ok[s]) {
        const float *src = a_src[s];
        if (VEC && kq + 4 <= rem) {
          v = __ldg(reinterpret_cast<const float4 *>(src));
        } else {
          if (kq + 0 < rem) v.x = __ldg(src + 0);
          if (kq + 1 < rem) v.y = __ldg(src + 1);
          if (kq + 2 < rem) v.z = __ldg(src + 2);
          if (kq + 3 < rem) v.w = __ldg(src + 3);
        }
      }
      ra[s] = v;
      a_src[s] += BK;
    }
#pragma unroll
    for (int s = 0; s < B_PER_T; ++s) {
      const int slot = tid + s * kThreads;
      const int kr = slot / (BN / 4);
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (kr < rem && b_cols[s] > 0) {
        const float *src = b_src[s];
        if (VEC && b_cols[s] == 4) {
          v = __ldg(reinterpret_cast<const float4 *>(src));
        } else {
          v.x = __ldg(src + 0);
          if (b_cols[s] > 1) v.y = __ldg(src + 1);
          if (b_cols[s] > 2) v.z = __ldg(src + 2);
          if (b_cols[s] > 3) v.w = __ldg(src + 3);
        }
      }
      rb[s] = v;
      b_src[s] += b_step;
    }
  };

  auto store_smem = [&](int buf) {
#pragma unroll
    for (int s = 0; s < A_PER_T; ++s) {
      const int slot = tid + s * kThreads;
      if (A_SLOTS % kThreads == 0 || slot < A_SLOTS) {
        const int r = slot / (BK / 4);
        const int kq = (slot % (BK / 4)) * 4;
        As[buf][kq + 0][r] = ra[s].x;
        As[buf][kq + 1][r] = ra[s].y;
        As[buf][kq + 2][r] = ra[s].z;
        As[buf][kq + 3][r] = ra[s].w;
      }
    }
#pragma unroll
    for (int s = 0; s < B_PER_T; ++s) {
      const int slot = tid + s * kThreads;
      if (B_SLOTS % kThreads == 0 || slot < B_SLOTS) {
        const int kr = slot / (BN / 4);
        const int cq = (slot % (BN / 4)) * 4;
        *reinterpret_cast<float4 *>(&Bs[buf][kr][cq]) = rb[s];
      }
    }
  };

  // Accumulators as column pairs: acc[i][jp] holds columns 2jp, 2jp+1 of
  // row i, so the packed FMA (two lanes per instruction) needs no repacking.
  float2 acc[TM][TN / 2];
#pragma unroll
  for (int i = 0; i < TM; ++i)
#pragma unroll
    for (int j = 0; j < TN / 2; ++j) acc[i][j] = make_float2(0.f, 0.f);

  const int a_off = wm * WTM + lr * 4;
  const int b_off = wn * WTN + lc * 4;

  const int64_t klen = kend - kbeg;
  if (ntiles > 0) {
    load_global((int)(klen < (1 << 30) ? klen : (1 << 30)));
    store_smem(0);
    __syncthreads();
  }
  for (int64_t t = 0; t < ntiles; ++t) {
    const int cur = (int)(t & 1);
    const bool more = t + 1 < ntiles;
    if (more) {
      const int64_t rem = klen - (t + 1) * BK;
      load_global((int)(rem < (1 << 30) ? rem : (1 << 30)));
    }
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
      for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN / 2; ++j) {
          acc[i][j].x = fmaf(a[i], b[j].x, acc[i][j].x);
          acc[i][j].y = fmaf(a[i], b[j].y, acc[i][j].y);
        }
    }
    if (more) store_smem(cur ^ 1);
    __syncthreads();
  }

  // Epilogue: fused alpha/beta (or raw partials for split-K).
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
}

// C <- alpha * sum_{z < splits} ws[z] + beta * C, slices summed in order z = 0..splits-1.
__global__ void splitk_reduce_kernel(GemmArgs p, const float *__restrict__ ws, int splits) {
  const int64_t total = p.M * p.N;
  for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < total;
       t += (int64_t)gridDim.x * blockDim.x) {
    float s = ws[t];
    for (int z = 1; z < splits; ++z) s += ws[(int64_t)z * total + t];
    const int64_t r = t / p.N, c = t % p.N;
    float *dst = p.C + r * p.ldc + c;
    float o = p.alpha * s;
    if (p.beta != 0.0f) o = fmaf(p.beta, *dst, o);
    *dst = o;
  }
}

template <int BM, int BN, int BK, int TM, int TN>
cudaError_t launch_cfg(const gemm_plan_t &plan, const GemmArgs &p, float *ws, cudaStream_t s) {
  const int split = plan.split_k > 1 ? plan.split_k : 1;
  int64_t kps = ceil_div(p.K, split);
  kps = ceil_div(kps, BK) * BK;
  dim3 grid((unsigned)ceil_div(p.N, BN), (unsigned)ceil_div(p.M, BM), (unsigned)split);
  float *w = split > 1 ? ws : nullptr;
  const int ws_vec = (p.N % 4 == 0) ? 1 : 0;
  profile_mark_before(s);
  if (plan.vec)
    simt_sgemm_kernel<BM, BN, BK, TM, TN, true><<<grid, kThreads, 0, s>>>(p, kps, w, ws_vec);
  else
    simt_sgemm_kernel<BM, BN, BK, TM, TN, false><<<grid, kThreads, 0, s>>>(p, kps, w, ws_vec);
  profile_mark_after(s);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || split == 1) return e;
  return launch_splitk_reduce(p, ws, split, s);
}

}  // namespace

SimtConfig simt_config(int id) {
  if (id == 1) return SimtConfig{64, 64, 16, kThreads};
  return SimtConfig{128, 128, 16, kThreads};
}

int simt_config_for_tile(int bm, int bn) {
  if (bm == 64 && bn == 64) return 1;
  if (bm == 128 && bn == 128) return 0;
  return -1;
}

cudaError_t launch_splitk_reduce(const GemmArgs &p, const float *ws, int splits, cudaStream_t s) {
  int64_t blocks = ceil_div(p.M * p.N, 256);
  if (blocks > 4096) blocks = 4096;
  splitk_reduce_kernel<<<(unsigned)blocks, 256, 0, s>>>(p, ws, splits);
  return cudaGetLastError();
}

cudaError_t launch_simt(const gemm_plan_t &plan, const GemmArgs &p, float *ws, cudaStream_t s) {
  if (plan.bm == 128 && plan.bn == 128) return launch_cfg<128, 128, 16, 8, 8>(plan, p, ws, s);
  if (plan.bm == 64 && plan.bn == 64) return launch_cfg<64, 64, 16, 4, 4>(plan, p, ws, s);
  return cudaErrorInvalidValue;
}

}  // namespace gg
