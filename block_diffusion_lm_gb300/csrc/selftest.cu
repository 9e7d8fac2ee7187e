// Self-test of the device-side hang guard: a kernel waits, through the same
// bounded-wait helpers the attention and GEMM kernels use, on an mbarrier
// that nothing ever arrives on.  The wait gives up after the given budget,
// records the timeout in the status word and returns, so the host sees
// CSBP_ERR_TIMEOUT from csbp_check_status and the context stays usable.
// Nothing else is in flight while it waits: no copy, MMA or TMEM holding.
#include <cuda_runtime.h>

#include <cstdint>

#include "csbp.h"
#include "csbp_internal.h"
#include "mbar_spin.cuh"
#include "ptx_sm100.cuh"

namespace csbp {
namespace {

// Thread 0 waits with mbar_wait, warp 1 with the warp-collective form and
// thread 64 with the polling form the backward's MMA issuer uses; all on a
// barrier with no arrivals.  Any of them giving up records DEV_TIMEOUT and
// raises the abort flag, which ends the others' waits too.
__global__ void wait_selftest_kernel(int* status, uint64_t budget_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbarrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(&bar, 0, status, &abort_flag, budget_ns);
  if ((threadIdx.x >> 5) == 1) mbar_wait_warp(&bar, 0, status, &abort_flag, budget_ns);
  if (threadIdx.x == 64) mbar_wait_spin(&bar, 0, status, &abort_flag, budget_ns);
  __syncthreads();
}

}  // namespace
}  // namespace csbp

extern "C" csbp_status csbp_wait_selftest(int64_t budget_ns, void* workspace, void* stream) {
  if (!workspace || budget_ns < 1000 || budget_ns > 2000000000) return CSBP_ERR_INVALID;
  if ((reinterpret_cast<uintptr_t>(workspace) & 15u) != 0) return CSBP_ERR_INVALID;
  csbp::wait_selftest_kernel<<<1, 96, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<int*>(workspace), static_cast<uint64_t>(budget_ns));
  return cudaGetLastError() == cudaSuccess ? CSBP_OK : CSBP_ERR_CUDA;
}
