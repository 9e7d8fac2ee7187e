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
#include <cuda.h>
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
struct ScratchAddr {
  CUcontext ctx;  // context the address was looked up in
  void* addr;
};
ScratchAddr g_scratch_dev[kMaxDevices] = {};

// The CUDA context current on this thread (the device's primary context for
// callers of the runtime API), through the runtime's driver entry point so
// that the library needs no link against the driver library.
CUcontext current_context() {
  using Fn = CUresult (*)(CUcontext*);
  static Fn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<Fn>(f);
  });
  CUcontext c = nullptr;
  if (!fn || fn(&c) != CUDA_SUCCESS) return nullptr;
  return c;
}

// Device address of g_bwd_scratch on the current device.  In host code the
// array's name only stands in for the symbol; the address is looked up (with
// that device current) the first time a context uses it, and cached for that
// device and context.  A call from another context of the same device (a
// driver-API context made current) looks it up again.
csbp_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return CSBP_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return CSBP_ERR_UNSUPPORTED;
  const CUcontext ctx = current_context();
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  ScratchAddr& e = g_scratch_dev[dev];
  if (!e.addr || e.ctx != ctx) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_bwd_scratch) != cudaSuccess || p == nullptr)
      return CSBP_ERR_CUDA;
    // the runtime makes a context current if none was: key on that one
    e.ctx = ctx ? ctx : current_context();
    e.addr = p;
  }
  *out = e.addr;
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

extern "C" csbp_status csbp_attn_bwd_noalloc_status(void* stream) {
  void* scratch = nullptr;
  const csbp_status sa = scratch_address(&scratch);
  if (sa != CSBP_OK) return sa;
  return csbp_check_status(scratch, stream);  // the status word opens the scratch
}
