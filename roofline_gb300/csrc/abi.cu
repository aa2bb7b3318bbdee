// The C ABI (include/gb300_gemm.h): argument checks, device properties,
// workspace, dispatch to the kernels, and status reporting.
//
// The course pages wrap every CUDA call in a macro that prints and exits
// ("Project - tiled matrix multiply", section "Starter scaffolding"); a
// library must not exit, so every failure becomes a returned status code.
#include <cstdio>
#include <cstring>
#include <mutex>

#include "common.cuh"

namespace gg {

namespace {

constexpr int kMaxDevices = 64;

std::mutex g_props_mu;
DeviceProps g_props[kMaxDevices];
bool g_props_valid[kMaxDevices];

std::mutex g_ws_mu;
void *g_ws_ptr[kMaxDevices];
size_t g_ws_bytes[kMaxDevices];

DeviceProps make_default_props() {
  DeviceProps d{};
  d.device = -1;
  d.sm_count = 152;
  d.cc_major = 10;
  d.cc_minor = 3;
  d.clock_khz = 2070000;
  d.mem_clock_khz = 3996000;
  d.mem_bus_width = 8192;
  d.regs_per_sm = 65536;
  d.smem_per_sm = 233472;
  d.smem_optin = 232448;
  d.l2_bytes = 129LL * 1024 * 1024;
  d.hbm_bytes = 284208LL * 1024 * 1024;
  d.from_device = 0;
  std::snprintf(d.name, sizeof(d.name), "%s", "GB300 (built-in figures)");
  return d;
}

bool query_props(int dev, DeviceProps *d) {
  DeviceProps p{};
  p.device = dev;
  auto attr = [&](cudaDeviceAttr a, int *v) { return cudaDeviceGetAttribute(v, a, dev) == cudaSuccess; };
  bool ok = attr(cudaDevAttrMultiProcessorCount, &p.sm_count) &&
            attr(cudaDevAttrComputeCapabilityMajor, &p.cc_major) &&
            attr(cudaDevAttrComputeCapabilityMinor, &p.cc_minor) &&
            attr(cudaDevAttrClockRate, &p.clock_khz) &&
            attr(cudaDevAttrMemoryClockRate, &p.mem_clock_khz) &&
            attr(cudaDevAttrGlobalMemoryBusWidth, &p.mem_bus_width) &&
            attr(cudaDevAttrMaxRegistersPerMultiprocessor, &p.regs_per_sm) &&
            attr(cudaDevAttrMaxSharedMemoryPerMultiprocessor, &p.smem_per_sm) &&
            attr(cudaDevAttrMaxSharedMemoryPerBlockOptin, &p.smem_optin);
  if (!ok) return false;
  int l2 = 0;
  if (!attr(cudaDevAttrL2CacheSize, &l2)) return false;
  p.l2_bytes = l2;
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return false;
  p.hbm_bytes = (int64_t)prop.totalGlobalMem;
  std::snprintf(p.name, sizeof(p.name), "%.127s", prop.name);
  p.from_device = 1;
  *d = p;
  return true;
}

bool valid_ld(int64_t ld, int64_t width) { return ld >= (width > 1 ? width : 1); }

int check_args(int64_t M, int64_t N, int64_t K, const float *A, int64_t lda, const float *B,
               int64_t ldb, const float *C, int64_t ldc, int ta = 0, int tb = 0) {
  if (M < 0 || N < 0 || K < 0) return GEMM_ERR_INVALID_ARG;
  if (!valid_ld(lda, ta ? M : K) || !valid_ld(ldb, tb ? K : N) || !valid_ld(ldc, N))
    return GEMM_ERR_INVALID_ARG;
  // keep every element offset well inside int64
  const int64_t lim = (int64_t)1 << 40;
  if (M > lim || N > lim || K > lim || lda > lim || ldb > lim || ldc > lim) return GEMM_ERR_INVALID_ARG;
  if (M > 0 && N > 0) {
    if (!C) return GEMM_ERR_INVALID_ARG;
    if (K > 0 && (!A || !B)) return GEMM_ERR_INVALID_ARG;
  }
  return GEMM_OK;
}

int current_device(int *dev) {
  if (cudaGetDevice(dev) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_NO_DEVICE;
  }
  if (*dev < 0 || *dev >= kMaxDevices) return GEMM_ERR_UNSUPPORTED;
  return GEMM_OK;
}

// Per-device library workspace, grown on demand.
int library_workspace(int dev, size_t need, void **out) {
  std::lock_guard<std::mutex> lk(g_ws_mu);
  if (g_ws_bytes[dev] < need) {
    if (g_ws_ptr[dev]) {
      cudaFree(g_ws_ptr[dev]);
      g_ws_ptr[dev] = nullptr;
      g_ws_bytes[dev] = 0;
    }
    void *p = nullptr;
    if (cudaMalloc(&p, need) != cudaSuccess) {
      cudaGetLastError();
      return GEMM_ERR_CUDA;
    }
    g_ws_ptr[dev] = p;
    g_ws_bytes[dev] = need;
  }
  *out = g_ws_ptr[dev];
  return GEMM_OK;
}

int to_status(cudaError_t e) { return e == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA; }

thread_local cudaEvent_t t_prof_before = nullptr;
thread_local cudaEvent_t t_prof_after = nullptr;
thread_local unsigned long long *t_prof_stamps = nullptr;

}  // namespace

void profile_mark_before(cudaStream_t s) {
  if (t_prof_before) cudaEventRecord(t_prof_before, s);
}
void profile_mark_after(cudaStream_t s) {
  if (t_prof_after) cudaEventRecord(t_prof_after, s);
}
bool profile_events_set() { return t_prof_before != nullptr; }
unsigned long long *profile_stamps() { return t_prof_stamps; }

const DeviceProps &default_props() {
  static const DeviceProps d = make_default_props();
  return d;
}

const DeviceProps &props_of(int dev) {
  if (dev < 0 || dev >= kMaxDevices) return default_props();
  std::lock_guard<std::mutex> lk(g_props_mu);
  if (!g_props_valid[dev]) {
    if (!query_props(dev, &g_props[dev])) {
      cudaGetLastError();
      return default_props();
    }
    g_props_valid[dev] = true;
  }
  return g_props[dev];
}

const DeviceProps &current_props() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return default_props();
  }
  return props_of(dev);
}

}  // namespace gg

using namespace gg;

extern "C" {

int gemm_abi_version(void) { return GEMM_ABI_VERSION; }

int gemm_set_profile_events(cudaEvent_t before_main, cudaEvent_t after_main) {
  if ((before_main == nullptr) != (after_main == nullptr)) return GEMM_ERR_INVALID_ARG;
  t_prof_before = before_main;
  t_prof_after = after_main;
  return GEMM_OK;
}

int gemm_set_profile_stamps(unsigned long long *stamps) {
  if (stamps && (reinterpret_cast<uintptr_t>(stamps) & 7)) return GEMM_ERR_INVALID_ARG;
  t_prof_stamps = stamps;
  return GEMM_OK;
}

const char *gemm_strerror(int code) {
  switch (code) {
    case GEMM_OK: return "success";
    case GEMM_ERR_INVALID_ARG: return "invalid argument (size, leading dimension, pointer or mode)";
    case GEMM_ERR_UNSUPPORTED: return "mode not supported for this device or shape";
    case GEMM_ERR_CUDA: return "CUDA runtime error or kernel launch failure";
    case GEMM_ERR_DEVICE_TIMEOUT: return "a bounded wait inside a kernel ran out";
    case GEMM_ERR_WORKSPACE_TOO_SMALL: return "workspace smaller than the plan requires";
    case GEMM_ERR_NO_DEVICE: return "no CUDA device visible";
    default: return "unknown status code";
  }
}

int gemm_device_info(int dev, gemm_device_info_t *out) {
  if (!out) return GEMM_ERR_INVALID_ARG;
  const DeviceProps *d = &default_props();
  if (dev >= 0) {
    int count = 0;
    if (cudaGetDeviceCount(&count) != cudaSuccess) {
      cudaGetLastError();
      count = 0;
    }
    if (count > 0) {
      if (dev >= count) return GEMM_ERR_INVALID_ARG;
      d = &props_of(dev);
    }
  }
  gemm_device_info_t o{};
  o.device = d->device;
  o.sm_count = d->sm_count;
  o.cc_major = d->cc_major;
  o.cc_minor = d->cc_minor;
  o.clock_khz = d->clock_khz;
  o.mem_clock_khz = d->mem_clock_khz;
  o.mem_bus_width_bits = d->mem_bus_width;
  o.fp32_lanes_per_sm = 128;
  o.regs_per_sm = d->regs_per_sm;
  o.smem_per_sm = d->smem_per_sm;
  o.smem_per_block_optin = d->smem_optin;
  o.from_device = d->from_device;
  o.l2_bytes = d->l2_bytes;
  o.hbm_bytes = d->hbm_bytes;
  o.fp32_peak_tflops = (double)d->sm_count * 128.0 * 2.0 * (double)d->clock_khz * 1e3 / 1e12;
  std::snprintf(o.name, sizeof(o.name), "%s", d->name);
  *out = o;
  return GEMM_OK;
}

int gemm_f32_plan(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                  int mode, uintptr_t align_hint, int beta_nonzero, gemm_plan_t *out) {
  if (!out) return GEMM_ERR_INVALID_ARG;
  if (M < 0 || N < 0 || K < 0) return GEMM_ERR_INVALID_ARG;
  return make_plan(M, N, K, lda, ldb, ldc, mode, align_hint, beta_nonzero, current_props(), out);
}

}  // extern "C"

namespace gg {

// One row-major GEMM (operand storage per p.ta / p.tb): checks, plan,
// workspace, launch.
int run_gemm(const GemmArgs &p, int mode, void *workspace, size_t ws_bytes, cudaStream_t stream) {
  const int64_t M = p.M, N = p.N, K = p.K;
  int st = check_args(M, N, K, p.A, p.lda, p.B, p.ldb, p.C, p.ldc, p.ta, p.tb);
  if (st != GEMM_OK) return st;
  gemm_plan_t plan;
  const uintptr_t align = (uintptr_t)p.A | (uintptr_t)p.B | (uintptr_t)p.C;
  // Mode and shape checks first (host only), then the device.
  st = make_plan(M, N, K, p.lda, p.ldb, p.ldc, mode, align, p.beta != 0.0f, default_props(),
                 &plan, p.ta, p.tb);
  if (st == GEMM_ERR_INVALID_ARG) return st;
  if (M == 0 || N == 0) return GEMM_OK;
  if (workspace && (((uintptr_t)workspace) & 255)) return GEMM_ERR_INVALID_ARG;

  int dev = -1;
  st = current_device(&dev);
  if (st != GEMM_OK) return st;
  const DeviceProps &dp = props_of(dev);
  st = make_plan(M, N, K, p.lda, p.ldb, p.ldc, mode, align, p.beta != 0.0f, dp, &plan, p.ta,
                 p.tb);
  if (st != GEMM_OK) return st;
  if (p.in_flag != nullptr && (p.alpha == 0.0f || !tc_plan_streaming(plan, M, N, K)))
    return GEMM_ERR_UNSUPPORTED;
  // K == 0, or alpha == 0 (BLAS: A and B are not read): C <- beta * C
  if (plan.kernel == GEMM_KERNEL_SCALE || p.alpha == 0.0f)
    return to_status(launch_scale(p, stream));

  void *ws = nullptr;
  size_t wsb = 0;
  if (plan.workspace_bytes > 0) {
    if (workspace) {
      if (ws_bytes < plan.workspace_bytes) return GEMM_ERR_WORKSPACE_TOO_SMALL;
      ws = workspace;
      wsb = ws_bytes;
    } else {
      st = library_workspace(dev, (size_t)plan.workspace_bytes, &ws);
      if (st != GEMM_OK) return st;
      wsb = (size_t)plan.workspace_bytes;
    }
  }

  switch (plan.kernel) {
    case GEMM_KERNEL_NAIVE:
    case GEMM_KERNEL_COALESCED:
    case GEMM_KERNEL_TILED: {
      profile_mark_before(stream);
      cudaError_t e = launch_ladder(plan.kernel, plan.bm, p, stream);
      profile_mark_after(stream);
      return to_status(e);
    }
    case GEMM_KERNEL_SIMT:
      return to_status(launch_simt(plan, p, static_cast<float *>(ws), stream));
    case GEMM_KERNEL_TC_TF32X3:
    case GEMM_KERNEL_TC_TF32:
      return launch_tc(plan, p, ws, wsb, stream);
    default:
      return GEMM_ERR_UNSUPPORTED;
  }
}

namespace {

// gemm_f32_op's problem as a row-major one.  Column-major storage is the
// row-major storage of the transpose, so C^T = op(B)^T * op(A)^T: the
// operands swap places, M and N swap, and each operand keeps its storage
// flag (a column-major B stored K x N is a row-major N x K matrix, i.e. the
// new A stored as M' x K with no transpose).
int op_args(int layout, int op_a, int op_b, int64_t M, int64_t N, int64_t K, float alpha,
            const float *A, int64_t lda, const float *B, int64_t ldb, float beta, float *C,
            int64_t ldc, GemmArgs *out) {
  if ((layout != GEMM_ROW_MAJOR && layout != GEMM_COL_MAJOR) ||
      (op_a != GEMM_OP_N && op_a != GEMM_OP_T) || (op_b != GEMM_OP_N && op_b != GEMM_OP_T))
    return GEMM_ERR_INVALID_ARG;
  if (layout == GEMM_ROW_MAJOR)
    *out = GemmArgs{M, N, K, alpha, beta, A, lda, B, ldb, C, ldc, op_a, op_b};
  else
    *out = GemmArgs{N, M, K, alpha, beta, B, ldb, A, lda, C, ldc, op_b, op_a};
  return GEMM_OK;
}

}  // namespace
}  // namespace gg

extern "C" {

int gemm_f32_ex(int64_t M, int64_t N, int64_t K, float alpha, const float *A, int64_t lda,
                const float *B, int64_t ldb, float beta, float *C, int64_t ldc, int mode,
                void *workspace, size_t ws_bytes, cudaStream_t stream) {
  return run_gemm(GemmArgs{M, N, K, alpha, beta, A, lda, B, ldb, C, ldc}, mode, workspace,
                  ws_bytes, stream);
}

int gemm_f32_op(int layout, int op_a, int op_b, int64_t M, int64_t N, int64_t K, float alpha,
                const float *A, int64_t lda, const float *B, int64_t ldb, float beta, float *C,
                int64_t ldc, int mode, void *workspace, size_t ws_bytes, cudaStream_t stream) {
  GemmArgs p;
  int st = op_args(layout, op_a, op_b, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, &p);
  if (st != GEMM_OK) return st;
  return run_gemm(p, mode, workspace, ws_bytes, stream);
}

int gemm_f32_op_plan(int layout, int op_a, int op_b, int64_t M, int64_t N, int64_t K,
                     int64_t lda, int64_t ldb, int64_t ldc, int mode, uintptr_t align_hint,
                     int beta_nonzero, gemm_plan_t *out) {
  if (!out) return GEMM_ERR_INVALID_ARG;
  if (M < 0 || N < 0 || K < 0) return GEMM_ERR_INVALID_ARG;
  GemmArgs p;
  int st = op_args(layout, op_a, op_b, M, N, K, 1.0f, nullptr, lda, nullptr, ldb, 0.0f, nullptr,
                   ldc, &p);
  if (st != GEMM_OK) return st;
  return make_plan(p.M, p.N, p.K, p.lda, p.ldb, p.ldc, mode, align_hint, beta_nonzero,
                   current_props(), out, p.ta, p.tb);
}

int gemm_f32(int64_t M, int64_t N, int64_t K, const float *A, int64_t lda, const float *B,
             int64_t ldb, float *C, int64_t ldc, int mode, cudaStream_t stream) {
  return gemm_f32_ex(M, N, K, 1.0f, A, lda, B, ldb, 0.0f, C, ldc, mode, nullptr, 0, stream);
}

int hbm_copy_f32(const float *src, float *dst, size_t n, cudaStream_t stream) {
  if (n == 0) return GEMM_OK;
  if (!src || !dst) return GEMM_ERR_INVALID_ARG;
  int dev = -1;
  int st = current_device(&dev);
  if (st != GEMM_OK) return st;
  return to_status(launch_copy(src, dst, n, props_of(dev).sm_count, stream));
}

int hbm_copy_calibrate(const float *src, float *dst, size_t n, int iters, cudaStream_t stream,
                       double *gbps_out) {
  if (!src || !dst || !gbps_out || n == 0 || iters < 1) return GEMM_ERR_INVALID_ARG;
  int dev = -1;
  int st = current_device(&dev);
  if (st != GEMM_OK) return st;
  const int sms = props_of(dev).sm_count;
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  if (cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess) {
    cudaGetLastError();
    if (e0) cudaEventDestroy(e0);
    return GEMM_ERR_CUDA;
  }
  cudaError_t e = launch_copy(src, dst, n, sms, stream);  // warm-up, untimed
  if (e == cudaSuccess) e = cudaEventRecord(e0, stream);
  for (int i = 0; i < iters && e == cudaSuccess; ++i) e = launch_copy(src, dst, n, sms, stream);
  if (e == cudaSuccess) e = cudaEventRecord(e1, stream);
  if (e == cudaSuccess) e = cudaEventSynchronize(e1);
  float ms = 0.f;
  if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, e0, e1);
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  if (e != cudaSuccess || ms <= 0.f) {
    cudaGetLastError();
    return GEMM_ERR_CUDA;
  }
  *gbps_out = 2.0 * (double)n * sizeof(float) * (double)iters / ((double)ms * 1e-3) / 1e9;
  return GEMM_OK;
}

int64_t fp32_fma_peak_sink_floats(void) {
  return (int64_t)fma_peak_blocks(current_props().sm_count) * 256;
}

int fp32_fma_peak(int64_t iters, int packed, float *sink, cudaStream_t stream,
                  double *tflops_out) {
  if (!sink || !tflops_out || iters < 1) return GEMM_ERR_INVALID_ARG;
  int dev = -1;
  int st = current_device(&dev);
  if (st != GEMM_OK) return st;
  const int sms = props_of(dev).sm_count;
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  if (cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess) {
    cudaGetLastError();
    if (e0) cudaEventDestroy(e0);
    return GEMM_ERR_CUDA;
  }
  double flops = 0.0;
  cudaError_t e = launch_fma_peak(iters < 1024 ? iters : 1024, packed, sms, sink, stream, &flops);
  if (e == cudaSuccess) e = cudaEventRecord(e0, stream);
  if (e == cudaSuccess) e = launch_fma_peak(iters, packed, sms, sink, stream, &flops);
  if (e == cudaSuccess) e = cudaEventRecord(e1, stream);
  if (e == cudaSuccess) e = cudaEventSynchronize(e1);
  float ms = 0.f;
  if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, e0, e1);
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  if (e != cudaSuccess || ms <= 0.f) {
    cudaGetLastError();
    return GEMM_ERR_CUDA;
  }
  *tflops_out = flops / ((double)ms * 1e-3) / 1e12;
  return GEMM_OK;
}

int gemm_check_status(cudaStream_t stream) {
  if (cudaStreamSynchronize(stream) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_CUDA;
  }
  return tc_read_and_clear_status(stream);
}

void gemm_shutdown(void) {
  host_pipeline_shutdown();
  std::lock_guard<std::mutex> lk(g_ws_mu);
  for (int d = 0; d < kMaxDevices; ++d) {
    if (g_ws_ptr[d]) {
      int cur = -1;
      cudaGetDevice(&cur);
      cudaSetDevice(d);
      cudaFree(g_ws_ptr[d]);
      if (cur >= 0) cudaSetDevice(cur);
      g_ws_ptr[d] = nullptr;
      g_ws_bytes[d] = 0;
    }
  }
  cudaGetLastError();
}

}  // extern "C"
