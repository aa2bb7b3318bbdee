// Passes around the tensor-core GEMM kernel: the TF32 hi/lo split of an
// operand into the workspace (row by row, or transposed so that it becomes
// K-major), and the stream-K fix-up that sums the parts of tiles shared
// between CTAs.  All are HBM-bound copies.
#include "tc_common.cuh"

namespace gg {
namespace tc {
namespace {

// Stream-K fix-up: an output tile whose K blocks were split between CTAs
// gets C = alpha * (sum of its partial tiles, in CTA order) + beta * C.
// Block j looks at the boundary between CTAs j and j+1 in the stream-K unit
// space; the block whose boundary is the first one strictly inside a tile
// handles that tile, all other blocks return at once (whole tiles were
// written by the GEMM).
constexpr int kFixRows = 16;  // tile rows per fix-up block
__device__ int g_fix_status;  // 0 = ok, else a GEMM_ERR_* code
constexpr int kTrK = 32, kTrN = 128;  // transposed split: k x n tile per block

__global__ void __launch_bounds__(256)
streamk_fixup_kernel(TcParams p, int BM, int BN, int64_t G) {
  __shared__ int64_t part_off[kFixMaxParts];
  __shared__ int nparts;
  grid_dependency_wait();  // the GEMM's partial tiles
  const int64_t c = (int64_t)blockIdx.x + 1;  // boundary between CTAs c-1 and c
  // boundaries live in the stream-K unit space (tiles after the whole-tile waves)
  const int64_t b = unit_begin(p.sk_units, c, G);
  const int64_t tl = b / p.num_kb;
  const int64_t t = p.dp_tiles + tl;
  const int64_t first = tl * p.num_kb, last = first + p.num_kb - 1;
  if (b == first || b > last) return;                       // not strictly inside a tile
  if (unit_begin(p.sk_units, c - 1, G) > first) return;     // an earlier boundary owns it
  if (threadIdx.x == 0) {
    int n = 0;
    for (int64_t cta = c - 1; cta < G && unit_begin(p.sk_units, cta, G) <= last; ++cta) {
      const int64_t ub = unit_begin(p.sk_units, cta, G), ue = unit_begin(p.sk_units, cta + 1, G);
      if (ub == ue) continue;  // no work
      if (n == kFixMaxParts) {  // more parts than this kernel sums: report, write nothing
        n = -1;
        break;
      }
      // the tile is this CTA's first segment (slot 0) or its last (slot 1)
      const int slot = (ub >= first) ? 0 : 1;
      part_off[n++] = (cta * 2 + slot) * (int64_t)BM * BN;
    }
    if (n < 0) atomicExch(&g_fix_status, GEMM_ERR_UNSUPPORTED);
    nparts = n;
  }
  __syncthreads();
  const int n = nparts;
  if (n < 0) return;
  // blockIdx.y picks 32 of the tile's BM rows; each thread keeps four
  // independent 16-byte sums so several loads are in flight
  int64_t mt, nt;
  tile_coords(p, t, mt, nt);
  const int64_t m0 = mt * BM + blockIdx.y * kFixRows;
  const int64_t n0 = nt * BN;
  const int64_t row0 = (int64_t)blockIdx.y * kFixRows * BN;  // offset of these rows in a part
  const bool vec = ((p.ldc & 3) == 0) && ((reinterpret_cast<uintptr_t>(p.C) & 15) == 0);
  const int span = kFixRows * BN;
  for (int e0 = threadIdx.x * 4; e0 < span; e0 += blockDim.x * 16) {
    float4 acc[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int i = 0; i < n; ++i) {
      const float *base = p.partial + part_off[i] + row0;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int e = e0 + u * blockDim.x * 4;
        if (e < span) {
          const float4 v = *reinterpret_cast<const float4 *>(base + e);
          acc[u].x += v.x;
          acc[u].y += v.y;
          acc[u].z += v.z;
          acc[u].w += v.w;
        }
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int e = e0 + u * blockDim.x * 4;
      if (e >= span) continue;
      const int r = e / BN, col = e % BN;
      const int64_t gr = m0 + r, gc = n0 + col;
      if (gr >= p.M || gc >= p.N) continue;
      float *dst = p.C + gr * p.ldc + gc;
      const float a4[4] = {acc[u].x, acc[u].y, acc[u].z, acc[u].w};
      if (vec && gc + 4 <= p.N) {
        float4 o = make_float4(p.alpha * a4[0], p.alpha * a4[1], p.alpha * a4[2], p.alpha * a4[3]);
        if (p.beta != 0.0f) {
          const float4 old = *reinterpret_cast<const float4 *>(dst);
          o.x = fmaf(p.beta, old.x, o.x);
          o.y = fmaf(p.beta, old.y, o.y);
          o.z = fmaf(p.beta, old.z, o.z);
          o.w = fmaf(p.beta, old.w, o.w);
        }
        *reinterpret_cast<float4 *>(dst) = o;
      } else {
        for (int q = 0; q < 4 && gc + q < p.N; ++q) {
          float o = p.alpha * a4[q];
          if (p.beta != 0.0f) o = fmaf(p.beta, dst[q], o);
          dst[q] = o;
        }
      }
    }
  }
}

// Row split: dst_hi/dst_lo (rows x kp, row-major) <- split of src (rows x
// k, ld), zero for k <= c < kp (lo == nullptr: the hi part only, for
// 1xTF32).  Block `blk` of the job's `blocks` walks the 4-float groups
// grid-stride.
__device__ __forceinline__ void split_rows_block(const SplitJob &j, int64_t blk) {
  const int64_t rows = j.a, k = j.b, kp = j.kp;
  const int64_t groups = rows * (kp / 4);
  for (int64_t g = blk * (int64_t)blockDim.x + threadIdx.x; g < groups;
       g += j.blocks * (int64_t)blockDim.x) {
    const int64_t r = g / (kp / 4);
    const int64_t c = (g % (kp / 4)) * 4;
    const float *s = j.src + r * j.ld + c;
    float v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = (c + i < k) ? __ldg(s + i) : 0.0f;
    float4 h, l;
    // 3xTF32 (lo written): the truncated split; 1xTF32: hi rounded to nearest
    h.x = j.lo ? tf32_trunc(v[0]) : tf32_rna(v[0]); l.x = v[0] - h.x;
    h.y = j.lo ? tf32_trunc(v[1]) : tf32_rna(v[1]); l.y = v[1] - h.y;
    h.z = j.lo ? tf32_trunc(v[2]) : tf32_rna(v[2]); l.z = v[2] - h.z;
    h.w = j.lo ? tf32_trunc(v[3]) : tf32_rna(v[3]); l.w = v[3] - h.w;
    *reinterpret_cast<float4 *>(j.hi + r * kp + c) = h;
    if (j.lo) *reinterpret_cast<float4 *>(j.lo + r * kp + c) = l;
  }
}

// Transposed split: src (k x n, ld, row-major) -> hi/lo (n x kp, row-major),
// columns k <= c < kp zero.  One block of 256 threads moves a 32 (k) x 128
// (n) tile: each thread loads four 16-byte pieces along n (all in flight at
// once), the tile goes through shared memory, and each thread then stores
// four 16-byte pieces of hi and of lo along k.  `vec` (ld % 4 == 0 and a
// 16-byte aligned source) enables the 16-byte loads; the stores are 16-byte
// aligned because kp is a multiple of 32.
__device__ __forceinline__ void split_transpose_block(const SplitJob &j, int64_t blk,
                                                      float (*tile)[kTrN + 1]) {
  const int64_t k = j.a, n = j.b, kp = j.kp;
  const int64_t k0 = (blk / j.grid_x) * kTrK;
  const int64_t n0 = (blk % j.grid_x) * kTrN;
  const int t = threadIdx.x;
  // loads: piece p = t + 256 * i covers row p / 32, columns 4 * (p % 32) .. +3
  float4 v[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int p = t + 256 * i;
    const int64_t kk = k0 + p / 32, nn = n0 + 4 * (p % 32);
    float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
    if (kk < k) {
      const float *s = j.src + kk * j.ld + nn;
      if (j.vec && nn + 4 <= n) {
        x = __ldg(reinterpret_cast<const float4 *>(s));
      } else {
        if (nn + 0 < n) x.x = __ldg(s + 0);
        if (nn + 1 < n) x.y = __ldg(s + 1);
        if (nn + 2 < n) x.z = __ldg(s + 2);
        if (nn + 3 < n) x.w = __ldg(s + 3);
      }
    }
    v[i] = x;
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int p = t + 256 * i;
    float *row = &tile[p / 32][4 * (p % 32)];
    row[0] = v[i].x;
    row[1] = v[i].y;
    row[2] = v[i].z;
    row[3] = v[i].w;
  }
  __syncthreads();
  // stores: piece q = t + 256 * i covers output row n0 + q / 8, k quad q % 8
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int q = t + 256 * i;
    const int nl = q / 8, kq = 4 * (q % 8);
    const int64_t nn = n0 + nl, kk = k0 + kq;
    if (nn < n && kk < kp) {
      float4 h, l;
      const float a0 = tile[kq + 0][nl], a1 = tile[kq + 1][nl];
      const float a2 = tile[kq + 2][nl], a3 = tile[kq + 3][nl];
      h.x = j.lo ? tf32_trunc(a0) : tf32_rna(a0); l.x = a0 - h.x;
      h.y = j.lo ? tf32_trunc(a1) : tf32_rna(a1); l.y = a1 - h.y;
      h.z = j.lo ? tf32_trunc(a2) : tf32_rna(a2); l.z = a2 - h.z;
      h.w = j.lo ? tf32_trunc(a3) : tf32_rna(a3); l.w = a3 - h.w;
      *reinterpret_cast<float4 *>(j.hi + nn * kp + kk) = h;
      if (j.lo) *reinterpret_cast<float4 *>(j.lo + nn * kp + kk) = l;
    }
  }
}

// One launch for one or two split jobs (A's and B's): the first job's
// blocks come first, then the second's.
__global__ void __launch_bounds__(256) split_kernel(SplitJob j0, SplitJob j1) {
  __shared__ float tile[kTrK][kTrN + 1];
  grid_dependency_wait();   // the kernel before this one is done
  grid_launch_dependents();  // the GEMM may launch; it waits for this grid to finish
  int64_t blk = blockIdx.x;
  const bool second = blk >= j0.blocks;
  const SplitJob j = second ? j1 : j0;
  if (second) blk -= j0.blocks;
  if (j.transposed)
    split_transpose_block(j, blk, tile);
  else
    split_rows_block(j, blk);
}

}  // namespace

// One launch with the programmatic-dependent-launch attribute when `pdl`.
template <typename... Args>
cudaError_t launch(void (*kern)(Args...), dim3 grid, dim3 block, bool pdl, cudaStream_t s,
                   Args... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = grid;
  lc.blockDim = block;
  lc.stream = s;
  lc.attrs = attr;
  lc.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&lc, kern, args...);
}

SplitJob split_rows_job(const float *src, int64_t ld, int64_t rows, int64_t k, int64_t kp,
                        float *hi, float *lo) {
  SplitJob j{src, ld, rows, k, kp, hi, lo, 0, 0, 0, 1};
  j.blocks = ceil_div(rows * (kp / 4), 256);
  if (j.blocks > 152 * 16) j.blocks = 152 * 16;
  if (j.blocks < 1) j.blocks = 1;
  return j;
}

SplitJob split_transposed_job(const float *src, int64_t ld, int64_t k, int64_t cols, int64_t kp,
                              float *hi, float *lo) {
  SplitJob j{src, ld, k, cols, kp, hi, lo, 1, 0, 0, 1};
  j.vec = ((ld & 3) == 0 && (reinterpret_cast<uintptr_t>(src) & 15) == 0) ? 1 : 0;
  j.grid_x = ceil_div(cols, kTrN);
  j.blocks = j.grid_x * ceil_div(kp, kTrK);
  return j;
}

cudaError_t launch_splits(const SplitJob &a, const SplitJob *b, bool pdl, cudaStream_t s) {
  SplitJob none{};
  const SplitJob &second = b ? *b : none;
  const int64_t blocks = a.blocks + second.blocks;
  if (blocks < 1 || blocks > 0x7fffffff) return cudaErrorInvalidValue;
  return launch(split_kernel, dim3((unsigned)blocks), dim3(256), pdl, s, a, second);
}

int fixup_read_and_clear_status(cudaStream_t s) {
  int v = 0;
  if (cudaMemcpyFromSymbolAsync(&v, g_fix_status, sizeof(int), 0, cudaMemcpyDeviceToHost, s) !=
          cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_CUDA;
  }
  if (v == 0) return GEMM_OK;
  const int zero = 0;
  if (cudaMemcpyToSymbolAsync(g_fix_status, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, s) !=
          cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_CUDA;
  }
  return v;
}

cudaError_t launch_fixup(const TcParams &p, int bm, int bn, int64_t G, bool pdl, cudaStream_t s) {
  return launch(streamk_fixup_kernel, dim3((unsigned)(G - 1), (unsigned)(bm / kFixRows)),
                dim3(256), pdl, s, p, bm, bn, G);
}

}  // namespace tc
}  // namespace gg
