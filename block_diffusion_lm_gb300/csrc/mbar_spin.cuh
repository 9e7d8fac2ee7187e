// Bounded mbarrier wait that polls with the non-blocking test (no thread
// suspension between polls), for the single MMA-issuing thread of the
// attention kernels: every cycle between an MMA group's completion and the
// issue of the next group leaves the tensor pipe idle.  Same bound and error
// reporting as mbar_wait.  Written from the public PTX ISA description of
// mbarrier.test_wait.
#pragma once

#include <cstdint>

#include "ptx_sm100.cuh"

namespace csbp {

__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ bool mbar_wait_spin(uint64_t* bar, uint32_t parity, int* status,
                                               volatile int* abort_flag,
                                               uint64_t budget_ns = 2000000000ull) {
  if (mbar_test_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_test_wait(bar, parity)) return true;
    if (abort_flag && *abort_flag) return false;
    if (globaltimer_ns() - t0 > budget_ns) {
      if (status) atomicExch(status, DEV_TIMEOUT);
      if (abort_flag) *abort_flag = 1;
      return false;
    }
  }
}

}  // namespace csbp
