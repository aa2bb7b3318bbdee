// The course page's GEMM ladder ("Project - tiled matrix multiply"), kept as
// comparison modes, plus the K == 0 scaling kernel.  Each kernel computes
// one output per thread; they are generalised here from square N x N to
// M x N x K with leading dimensions and the alpha/beta epilogue.
#include "common.cuh"

namespace gg {
namespace {

__device__ __forceinline__ void store_out(const GemmArgs &p, int64_t r, int64_t c, float acc) {
  float *dst = p.C + r * p.ldc + c;
  float v = p.alpha * acc;
  if (p.beta != 0.0f) v = fmaf(p.beta, *dst, v);
  *dst = v;
}

// K == 0 or alpha == 0: C <- beta*C (beta == 0 writes zeros without reading C).
__global__ void scale_kernel(GemmArgs p) {
  int64_t total = p.M * p.N;
  for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < total;
       t += (int64_t)gridDim.x * blockDim.x) {
    int64_t r = t / p.N, c = t % p.N;
    float *dst = p.C + r * p.ldc + c;
    *dst = (p.beta != 0.0f) ? p.beta * *dst : 0.0f;
  }
}

// "Stage 0 - the naive baseline": thread x -> output row, y -> column, so
// adjacent lanes touch addresses a whole row apart (uncoalesced).
__global__ void naive_kernel(GemmArgs p) {
  int64_t row = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  int64_t col = blockIdx.y * (int64_t)blockDim.y + threadIdx.y;
  if (row < p.M && col < p.N) {
    float sum = 0.0f;
    for (int64_t k = 0; k < p.K; ++k) sum += p.A[row * p.lda + k] * p.B[k * p.ldb + col];
    store_out(p, row, col, sum);
  }
}

// "Stage 1 - global memory coalescing": x -> column, so a warp reads one
// broadcast A element and 32 consecutive B elements per k.
__global__ void coalesced_kernel(GemmArgs p) {
  int64_t col = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  int64_t row = blockIdx.y * (int64_t)blockDim.y + threadIdx.y;
  if (row < p.M && col < p.N) {
    float sum = 0.0f;
    for (int64_t k = 0; k < p.K; ++k) sum += p.A[row * p.lda + k] * p.B[k * p.ldb + col];
    store_out(p, row, col, sum);
  }
}

// "Stage 2 - shared memory tiling": TILE x TILE tiles of A and B staged in
// shared memory, zero-filled outside the matrices, two barriers per tile.
template <int TILE>
__global__ void tiled_kernel(GemmArgs p) {
  __shared__ float As[TILE][TILE];
  __shared__ float Bs[TILE][TILE];
  int tx = threadIdx.x, ty = threadIdx.y;
  int64_t row = blockIdx.y * (int64_t)TILE + ty;
  int64_t col = blockIdx.x * (int64_t)TILE + tx;
  float sum = 0.0f;
  for (int64_t t = 0; t < p.K; t += TILE) {
    int64_t ak = t + tx, bk = t + ty;
    As[ty][tx] = (row < p.M && ak < p.K) ? p.A[row * p.lda + ak] : 0.0f;
    Bs[ty][tx] = (bk < p.K && col < p.N) ? p.B[bk * p.ldb + col] : 0.0f;
    __syncthreads();
#pragma unroll
    for (int k = 0; k < TILE; ++k) sum += As[ty][k] * Bs[k][tx];
    __syncthreads();
  }
  if (row < p.M && col < p.N) store_out(p, row, col, sum);
}

}  // namespace

cudaError_t launch_scale(const GemmArgs &p, cudaStream_t s) {
  int64_t total = p.M * p.N;
  int64_t blocks = ceil_div(total, 256);
  if (blocks > 65535) blocks = 65535;
  scale_kernel<<<(unsigned)blocks, 256, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_ladder(int kernel, int tile, const GemmArgs &p, cudaStream_t s) {
  if (kernel == GEMM_KERNEL_NAIVE) {
    dim3 block(16, 16);
    dim3 grid((unsigned)ceil_div(p.M, 16), (unsigned)ceil_div(p.N, 16));
    naive_kernel<<<grid, block, 0, s>>>(p);
  } else if (kernel == GEMM_KERNEL_COALESCED) {
    dim3 block(16, 16);
    dim3 grid((unsigned)ceil_div(p.N, 16), (unsigned)ceil_div(p.M, 16));
    coalesced_kernel<<<grid, block, 0, s>>>(p);
  } else if (kernel == GEMM_KERNEL_TILED && tile == 16) {
    dim3 block(16, 16);
    dim3 grid((unsigned)ceil_div(p.N, 16), (unsigned)ceil_div(p.M, 16));
    tiled_kernel<16><<<grid, block, 0, s>>>(p);
  } else if (kernel == GEMM_KERNEL_TILED && tile == 32) {
    dim3 block(32, 32);
    dim3 grid((unsigned)ceil_div(p.N, 32), (unsigned)ceil_div(p.M, 32));
    tiled_kernel<32><<<grid, block, 0, s>>>(p);
  } else {
    return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace gg
