// tcgen05 3xTF32 tensor-core GEMM (placeholder until the kernel lands).
#include "common.cuh"

namespace gg {

bool tc_supported(const DeviceProps &) { return false; }

uint64_t tc_workspace_bytes(const gemm_plan_t &, int64_t, int64_t, int64_t) { return 0; }

int launch_tc(const gemm_plan_t &, const GemmArgs &, void *, size_t, cudaStream_t) {
  return GEMM_ERR_UNSUPPORTED;
}

int tc_read_and_clear_status(cudaStream_t) { return GEMM_OK; }

}  // namespace gg
