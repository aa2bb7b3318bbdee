// Device-to-device copy used to measure the HBM roof ("Bandwidths and peak
// rate - exercises", exercise 2: a grid-stride copy out[i] = in[i], each
// element read once and written once, bandwidth = 2 * n * 4 bytes / time).
//
// GB300 version: 128-bit accesses with streaming cache hints (the data is
// touched once, far larger than L2), four independent 16-byte loads in
// flight per thread before any store, and a grid of 8 CTAs x 256 threads
// per SM so every SM keeps enough bytes in flight to cover HBM latency.
#include "common.cuh"

namespace gg {
namespace {

constexpr int kCopyThreads = 256;
constexpr int kUnroll = 4;

__global__ void __launch_bounds__(kCopyThreads)
copy_vec_kernel(const float4 *__restrict__ src, float4 *__restrict__ dst, size_t n4) {
  const size_t stride = (size_t)gridDim.x * kCopyThreads;
  size_t i = (size_t)blockIdx.x * kCopyThreads + threadIdx.x;
  for (; i + (kUnroll - 1) * stride < n4; i += kUnroll * stride) {
    float4 v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) v[u] = __ldcs(src + i + u * stride);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) __stcs(dst + i + u * stride, v[u]);
  }
  for (; i < n4; i += stride) __stcs(dst + i, __ldcs(src + i));
}

__global__ void copy_scalar_kernel(const float *__restrict__ src, float *__restrict__ dst,
                                   size_t begin, size_t n) {
  for (size_t i = begin + (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x)
    dst[i] = src[i];
}

}  // namespace

cudaError_t launch_copy(const float *src, float *dst, size_t n, int sm_count, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  const bool aligned = ((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst)) & 15) == 0;
  size_t done = 0;
  if (aligned) {
    const size_t n4 = n / 4;
    if (n4 > 0) {
      int64_t blocks = (int64_t)sm_count * 8;
      const int64_t need = ceil_div((int64_t)n4, kCopyThreads);
      if (blocks > need) blocks = need;
      copy_vec_kernel<<<(unsigned)blocks, kCopyThreads, 0, s>>>(
          reinterpret_cast<const float4 *>(src), reinterpret_cast<float4 *>(dst), n4);
      cudaError_t e = cudaGetLastError();
      if (e != cudaSuccess) return e;
    }
    done = n4 * 4;
  }
  if (done < n) {
    int64_t blocks = ceil_div((int64_t)(n - done), 256);
    const int64_t cap = (int64_t)sm_count * 8;
    if (blocks > cap) blocks = cap;
    copy_scalar_kernel<<<(unsigned)blocks, 256, 0, s>>>(src, dst, done, n);
    return cudaGetLastError();
  }
  return cudaSuccess;
}

}  // namespace gg
