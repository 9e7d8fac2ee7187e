// Allocation-free variant of the backward entry point.
//
// Some callers cannot call cudaMalloc at all: plugin or custom-op interfaces
// that hand a library only its input and output buffers and offer no
// workspace, runtimes whose memory pool owns all device memory and forbids
// allocations from elsewhere, and latency-critical paths that cannot afford
// cudaMalloc's implicit device synchronisation.  For them this file keeps the
// backward pass's scratch (status word, D, fp32 dQ accumulator) in one
// fixed-size array in device global memory, reserved when the library's
// device code is loaded and held by every GPU that loads it until the
// process exits.
#include <cuda_runtime.h>

#include <mutex>

#include "csbp.h"
#include "csbp_internal.h"

namespace {

constexpr size_t kScratchBytes = static_cast<size_t>(64) << 20;  // 64 MiB

// Shared by every call of csbp_attn_bwd_noalloc on a device.
static __device__ __align__(256) unsigned char g_bwd_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_dev[kMaxDevices] = {};

// Device address of g_bwd_scratch on the current device.  In host code the
// array's name only stands in for the symbol; the address is looked up once
// per device (with that device current) and cached.
csbp_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return CSBP_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return CSBP_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_dev[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_bwd_scratch) != cudaSuccess || p == nullptr)
      return CSBP_ERR_CUDA;
    g_scratch_dev[dev] = p;
  }
  *out = g_scratch_dev[dev];
  return CSBP_OK;
}

}  // namespace

extern "C" csbp_status csbp_attn_bwd_noalloc(
    const csbp_problem* problem, const csbp_inputs* in, const void* work_dev,
    const csbp_schedule_info* info, const void* o_clean, const void* o_corr, const float* lse,
    const void* do_clean, const void* do_corr, void* dq_clean, void* dq_corr, void* dk_clean,
    void* dv_clean, void* dk_corr, void* dv_corr, void* stream) {
  const csbp_status st = csbp::validate_problem(problem);
  if (st != CSBP_OK) return st;
  const size_t need = csbp_workspace_bytes(problem, 1);
  if (need == 0) return CSBP_ERR_INVALID;
  if (need > kScratchBytes) return CSBP_ERR_WORKSPACE;  // beyond the built-in scratch
  void* scratch = nullptr;
  const csbp_status sa = scratch_address(&scratch);
  if (sa != CSBP_OK) return sa;
  // The status word must start at zero; D and the dQ accumulator are fully
  // rewritten by the backward pass itself.
  if (cudaMemsetAsync(scratch, 0, 256, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return CSBP_ERR_CUDA;
  return csbp_attn_bwd(problem, in, work_dev, info, o_clean, o_corr, lse, do_clean, do_corr,
                       dq_clean, dq_corr, dk_clean, dv_clean, dk_corr, dv_corr, scratch,
                       kScratchBytes, stream);
}
