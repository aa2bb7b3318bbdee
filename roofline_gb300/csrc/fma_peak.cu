// FP32 FMA-throughput probe ("Bandwidths and peak rate - exercises",
// exercise 5): every thread runs register-only chains acc = acc * x + y,
// several independent chains so the FMA pipe never waits on a dependency,
// and writes its result to global memory so the work is not removed.
// FLOP = threads x iterations x chains x 2 (x2 again for the packed form,
// which updates two lanes per instruction).  Grid: 8 CTAs of 256 threads
// per SM.
#include "common.cuh"

namespace gg {
namespace {

constexpr int kChains = 8;
constexpr int kFmaThreads = 256;

__global__ void __launch_bounds__(kFmaThreads)
fma_chain_kernel(float x, float y, int64_t iters, float *__restrict__ sink) {
  float acc[kChains];
#pragma unroll
  for (int c = 0; c < kChains; ++c) acc[c] = (float)(threadIdx.x + c);
  for (int64_t i = 0; i < iters; ++i) {
#pragma unroll
    for (int c = 0; c < kChains; ++c) acc[c] = fmaf(acc[c], x, y);
  }
  float s = 0.f;
#pragma unroll
  for (int c = 0; c < kChains; ++c) s += acc[c];
  sink[blockIdx.x * kFmaThreads + threadIdx.x] = s;
}

__global__ void __launch_bounds__(kFmaThreads)
fma2_chain_kernel(float x, float y, int64_t iters, float *__restrict__ sink) {
  float2 acc[kChains];
#pragma unroll
  for (int c = 0; c < kChains; ++c) acc[c] = make_float2((float)threadIdx.x, (float)c);
  const float2 xx = make_float2(x, x), yy = make_float2(y, y);
  for (int64_t i = 0; i < iters; ++i) {
#pragma unroll
    for (int c = 0; c < kChains; ++c) acc[c] = __ffma2_rn(acc[c], xx, yy);
  }
  float s = 0.f;
#pragma unroll
  for (int c = 0; c < kChains; ++c) s += acc[c].x + acc[c].y;
  sink[blockIdx.x * kFmaThreads + threadIdx.x] = s;
}

}  // namespace

int fma_peak_blocks(int sm_count) { return sm_count * 8; }

cudaError_t launch_fma_peak(int64_t iters, int packed, int sm_count, float *sink, cudaStream_t s,
                            double *flops) {
  const int blocks = fma_peak_blocks(sm_count);
  // values that keep the chains finite for any iteration count
  const float x = 0.999999f, y = 1e-6f;
  if (packed)
    fma2_chain_kernel<<<blocks, kFmaThreads, 0, s>>>(x, y, iters, sink);
  else
    fma_chain_kernel<<<blocks, kFmaThreads, 0, s>>>(x, y, iters, sink);
  *flops = (double)blocks * kFmaThreads * (double)iters * kChains * 2.0 * (packed ? 2.0 : 1.0);
  return cudaGetLastError();
}

}  // namespace gg
