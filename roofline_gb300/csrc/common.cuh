// Internal declarations shared by the library's translation units.
// Nothing here is part of the C ABI (include/gb300_gemm.h is).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "gb300_gemm.h"

namespace gg {

// One GEMM problem, C <- alpha*A*B + beta*C, row-major (see gb300_gemm.h).
struct GemmArgs {
  int64_t M, N, K;
  float alpha, beta;
  const float *A;
  int64_t lda;
  const float *B;
  int64_t ldb;
  float *C;
  int64_t ldc;
  // operand storage: ta = 1 means A is stored K x M (A(i,k) = A[k*lda + i]),
  // tb = 1 means B is stored N x K (B(k,j) = B[j*ldb + k]); 0 is the
  // row-major M x K / K x N storage of gemm_f32.
  int ta = 0, tb = 0;
  // b_presplit = 1 (tensor-core path only): the workspace already holds the
  // B_hi / B_lo planes of this B (same N, K and mode, written by an earlier
  // call on the same stream), so the B split pass is skipped.  plain_order =
  // 1: launch without programmatic dependent launch (each kernel waits for
  // everything before it in the stream), for callers that chain the GEMM
  // behind cross-stream event waits.
  int b_presplit = 0, plain_order = 0;
  // b_planes_written (host memory, or nullptr): set to 1 when this call's
  // launches write the B_hi / B_lo planes into the workspace (a call that
  // splits B on chip writes none), so a caller knows when a later call may
  // take b_presplit = 1.
  int *b_planes_written = nullptr;
  // Streaming (tensor-core path with A split on chip, one CTA per tile):
  // A's rows, and C's when beta != 0, are still arriving in row blocks of
  // stream_rows rows (a multiple of the tile height) while the GEMM runs.
  // Row block i is in device memory once in_flag[i] - epoch >= 0 (32-bit
  // cyclic compare); the GEMM sets out_flag[i] = epoch once every tile of
  // block i is stored, counting in tile_cnt[i] (zero on entry, zero again
  // when the block completes).  in_flag == nullptr: no streaming.
  const unsigned *in_flag = nullptr;
  unsigned *out_flag = nullptr, *tile_cnt = nullptr;
  unsigned epoch = 0;
  int64_t stream_rows = 0;
  int stream_blocks = 0;
};

// Cached properties of one device (or the built-in GB300 figures).
struct DeviceProps {
  int device;
  int sm_count;
  int cc_major, cc_minor;
  int clock_khz;
  int mem_clock_khz;
  int mem_bus_width;
  int regs_per_sm;
  int smem_per_sm;
  int smem_optin;
  int64_t l2_bytes;
  int64_t hbm_bytes;
  int from_device;
  char name[128];
};

// Returns the props of the current device, or GB300 defaults when none is
// visible (from_device = 0).  Thread-safe; queried once per device.
const DeviceProps &current_props();
const DeviceProps &props_of(int dev);
const DeviceProps &default_props();

// Measurement hooks (abi.cu): record the caller's profiling events around
// the main kernel launch, if set for this host thread.
void profile_mark_before(cudaStream_t s);
void profile_mark_after(cudaStream_t s);
bool profile_events_set();
// The caller's stamp pair for the next main-kernel launch on this host thread
// (gemm_set_profile_stamps), or nullptr.
unsigned long long *profile_stamps();

// %globaltimer: the GPU's nanosecond clock, common to all SMs.
__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Planner (plan.cu).
// ta / tb: operand storage as in GemmArgs.
int make_plan(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
              int64_t ldc, int mode, uintptr_t align_hint, int beta_nonzero,
              const DeviceProps &dp, gemm_plan_t *out, int ta = 0, int tb = 0);
bool tc_supported(const DeviceProps &dp);

// One row-major GEMM through the planner and the kernels (abi.cu): the body
// of gemm_f32_ex / gemm_f32_op.  workspace == nullptr: the library's
// per-device buffer.  Returns a GEMM_* status.
int run_gemm(const GemmArgs &p, int mode, void *workspace, size_t ws_bytes, cudaStream_t stream);

// Host-buffer pipeline (host.cu): frees its device staging, streams and events.
void host_pipeline_shutdown();

// Kernel launchers.  Each returns cudaSuccess or the launch error.
cudaError_t launch_scale(const GemmArgs &p, cudaStream_t s);
cudaError_t launch_ladder(int kernel, int tile, const GemmArgs &p, cudaStream_t s);
cudaError_t launch_simt(const gemm_plan_t &plan, const GemmArgs &p, float *ws,
                        cudaStream_t s);
cudaError_t launch_splitk_reduce(const GemmArgs &p, const float *ws, int splits,
                                 cudaStream_t s);
cudaError_t launch_copy(const float *src, float *dst, size_t n, int sm_count,
                        cudaStream_t s);
int fma_peak_blocks(int sm_count);
cudaError_t launch_fma_peak(int64_t iters, int packed, int sm_count, float *sink, cudaStream_t s,
                            double *flops);
// Tensor-core path (tc_tf32x3.cu).  Returns a GEMM_* status.
int launch_tc(const gemm_plan_t &plan, const GemmArgs &p, void *ws, size_t ws_bytes,
              cudaStream_t s);
uint64_t tc_workspace_bytes(const gemm_plan_t &plan, int64_t M, int64_t N, int64_t K);
// The plan of a streaming call (GemmArgs::in_flag): the same tile
// configuration, one CTA per tile (no stream-K, so every tile is finished by
// the CTA that computes it; measured faster than waves plus stream-K here),
// and the workspace that needs.  False when the plan cannot stream: not the
// tensor-core path, or A not split on chip.
bool tc_plan_streaming(gemm_plan_t &plan, int64_t M, int64_t N, int64_t K);
bool tc_config_valid(int bm, int bn, int bk, int stages, int a_inkernel, int concat, int nprod,
                     int b_inkernel);
int tc_ctas_per_sm(int bm, int bn, int bk, int stages, int a_inkernel, int concat, int nprod,
                   int b_inkernel, int smem_per_sm);
int tc_read_and_clear_status(cudaStream_t s);

// CUDA-core tile (simt.cu): 64 x 128, 8 x 8 per thread, 128 threads, K in
// BK-deep stages.
struct SimtConfig {
  int bm, bn, bk, threads;
};
SimtConfig simt_config();
// Built (BK, stages) pairs of the 64 x 128 CUDA-core tile; the first is the default.
#define GG_SIMT_CONFIGS(X) X(16, 4) X(32, 2)
bool simt_config_valid(int bk, int stages);


inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace gg
