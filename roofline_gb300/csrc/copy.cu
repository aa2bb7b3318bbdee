// Device-to-device copy used to measure the HBM roof ("Bandwidths and peak
// rate - exercises", exercise 2: a grid-stride copy out[i] = in[i], each
// element read once and written once, bandwidth = 2 * n * 4 bytes / time).
//
// GB300 version: 128-bit accesses with streaming cache hints (the data is
// touched once, far larger than L2), four independent 16-byte loads in
// flight per thread before any store, and a grid of 8 CTAs x 256 threads
// per SM so every SM keeps enough bytes in flight to cover HBM latency.
#include <cstdlib>

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

template <int UNROLL, bool HINTS>
__global__ void __launch_bounds__(kCopyThreads)
copy_var_kernel(const float4 *__restrict__ src, float4 *__restrict__ dst, size_t n4) {
  const size_t stride = (size_t)gridDim.x * kCopyThreads;
  size_t i = (size_t)blockIdx.x * kCopyThreads + threadIdx.x;
  for (; i + (UNROLL - 1) * stride < n4; i += UNROLL * stride) {
    float4 v[UNROLL];
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) v[u] = HINTS ? __ldcs(src + i + u * stride) : src[i + u * stride];
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      if (HINTS) __stcs(dst + i + u * stride, v[u]);
      else dst[i + u * stride] = v[u];
    }
  }
  for (; i < n4; i += stride) dst[i] = src[i];
}

// Block-contiguous chunks: each CTA copies CHUNK = 256 x UNROLL float4
// contiguous elements per iteration (grid-stride over chunks).
template <int UNROLL>
__global__ void __launch_bounds__(kCopyThreads)
copy_chunk_kernel(const float4 *__restrict__ src, float4 *__restrict__ dst, size_t n4) {
  constexpr size_t CH = (size_t)kCopyThreads * UNROLL;
  const size_t nch = n4 / CH;
  for (size_t c = blockIdx.x; c < nch; c += gridDim.x) {
    const float4 *s = src + c * CH + threadIdx.x;
    float4 *d = dst + c * CH + threadIdx.x;
    float4 v[UNROLL];
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) v[u] = __ldcs(s + u * kCopyThreads);
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) __stcs(d + u * kCopyThreads, v[u]);
  }
  for (size_t i = nch * CH + (size_t)blockIdx.x * kCopyThreads + threadIdx.x; i < n4;
       i += (size_t)gridDim.x * kCopyThreads)
    dst[i] = src[i];
}

// Bulk-copy ring: one thread per CTA streams CHUNK-byte pieces global ->
// shared (cp.async.bulk, mbarrier completion) -> global (bulk store group).
constexpr int kChunk = 16384, kRing = 4;

__global__ void __launch_bounds__(32)
copy_bulk_kernel(const char *__restrict__ src, char *__restrict__ dst, size_t nchunks) {
  extern __shared__ __align__(128) char ring[];
  __shared__ __align__(8) uint64_t bar[kRing];
  if (threadIdx.x != 0) return;
  auto sa = [](const void *p) { return (uint32_t)__cvta_generic_to_shared(p); };
  for (int s = 0; s < kRing; ++s)
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(sa(&bar[s])));
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  const size_t G = gridDim.x;
  const size_t mine = nchunks > blockIdx.x ? (nchunks - blockIdx.x + G - 1) / G : 0;
  auto load = [&](size_t k) {
    const int s = (int)(k % kRing);
    const size_t c = blockIdx.x + k * G;
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(sa(&bar[s])),
                 "r"(kChunk) : "memory");
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(sa(ring + s * kChunk)), "l"(src + c * kChunk), "r"(kChunk), "r"(sa(&bar[s]))
        : "memory");
  };
  for (size_t k = 0; k < mine && k < kRing; ++k) load(k);
  uint64_t t0;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  for (size_t k = 0; k < mine; ++k) {
    const int s = (int)(k % kRing);
    const uint32_t par = (uint32_t)(k / kRing) & 1u;
    uint32_t ok = 0;
    for (uint32_t spin = 0; !ok; ++spin) {
      asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                   "selp.u32 %0, 1, 0, p;\n\t}" : "=r"(ok) : "r"(sa(&bar[s])), "r"(par) : "memory");
      if (!ok && (spin & 255) == 255) {
        uint64_t t;
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
        if (t - t0 > 1000000000ull) return;  // gave up (bounded wait)
      }
    }
    const size_t c = blockIdx.x + k * G;
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst + c * kChunk),
                 "r"(sa(ring + s * kChunk)), "r"(kChunk) : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    if (k + kRing < mine) {
      asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
      load(k + kRing);
    }
  }
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

}  // namespace

cudaError_t launch_copy(const float *src, float *dst, size_t n, int sm_count, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  const bool aligned = ((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst)) & 15) == 0;
  size_t done = 0;
  const char *var_env = getenv("GEMM_COPY_VARIANT");  // experiment hook
  const int var = var_env ? atoi(var_env) : 0;
  if (aligned && var != 0) {
    const size_t n4 = n / 4;
    if (var == 5) {
      const size_t nchunks = (n * 4) / kChunk;
      cudaFuncSetAttribute(copy_bulk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kRing * kChunk);
      copy_bulk_kernel<<<(unsigned)(sm_count * 3), 32, kRing * kChunk, s>>>(
          reinterpret_cast<const char *>(src), reinterpret_cast<char *>(dst), nchunks);
      done = nchunks * kChunk / 4;
    } else {
      const int per_sm = (var == 3 || var == 6 || var == 8 || var == 9 || var == 10) ? 16 : 8;
      int64_t blocks = (int64_t)sm_count * per_sm;
      if (var == 1) copy_var_kernel<8, true><<<(unsigned)blocks, kCopyThreads, 0, s>>>(
          reinterpret_cast<const float4 *>(src), reinterpret_cast<float4 *>(dst), n4);
      if (var == 2) copy_var_kernel<4, false><<<(unsigned)blocks, kCopyThreads, 0, s>>>(
          reinterpret_cast<const float4 *>(src), reinterpret_cast<float4 *>(dst), n4);
      if (var == 3) copy_var_kernel<4, true><<<(unsigned)blocks, kCopyThreads, 0, s>>>(
          reinterpret_cast<const float4 *>(src), reinterpret_cast<float4 *>(dst), n4);
      if (var == 4) copy_var_kernel<8, false><<<(unsigned)blocks, kCopyThreads, 0, s>>>(
          reinterpret_cast<const float4 *>(src), reinterpret_cast<float4 *>(dst), n4);
      if (var == 6) copy_var_kernel<8, true><<<(unsigned)blocks, kCopyThreads, 0, s>>>(
          reinterpret_cast<const float4 *>(src), reinterpret_cast<float4 *>(dst), n4);
      if (var == 7) copy_var_kernel<16, true><<<(unsigned)blocks, kCopyThreads, 0, s>>>(
          reinterpret_cast<const float4 *>(src), reinterpret_cast<float4 *>(dst), n4);
      if (var == 8) copy_var_kernel<16, true><<<(unsigned)blocks, kCopyThreads, 0, s>>>(
          reinterpret_cast<const float4 *>(src), reinterpret_cast<float4 *>(dst), n4);
      if (var == 9) copy_chunk_kernel<4><<<(unsigned)blocks, kCopyThreads, 0, s>>>(
          reinterpret_cast<const float4 *>(src), reinterpret_cast<float4 *>(dst), n4);
      if (var == 10) copy_chunk_kernel<8><<<(unsigned)blocks, kCopyThreads, 0, s>>>(
          reinterpret_cast<const float4 *>(src), reinterpret_cast<float4 *>(dst), n4);
      if (var == 11) copy_chunk_kernel<8><<<(unsigned)blocks, kCopyThreads, 0, s>>>(
          reinterpret_cast<const float4 *>(src), reinterpret_cast<float4 *>(dst), n4);
      done = n4 * 4;
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  } else if (aligned) {
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
