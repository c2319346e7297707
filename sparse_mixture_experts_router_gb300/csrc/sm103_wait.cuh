// Bounded mbarrier waits shared by the tcgen05 kernels: every wait gives
// up after a fixed time, records MOE_ERR_TIMEOUT in the call's status word
// and raises a shared-memory abort flag that ends the other warp roles'
// loops, so a kernel never hangs the GPU.
#pragma once

#include <stdint.h>

#include "device_util.cuh"
#include "moe_internal.h"
#include "sm103_ptx.cuh"

namespace moe {

constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s
constexpr uint64_t kDrainLimitNs = 50000000ull;    // 50 ms

// Bounded wait on one mbarrier phase. Returns false if the wait ran out (and
// then records the timeout and raises the abort flag) or if another role
// already aborted.
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                           int* status) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      *abort_flag = 1;
      set_status(status, MOE_ERR_TIMEOUT);
      return false;
    }
  }
}
// Short bounded wait used only while draining after an abort.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!ptx::mbar_try_wait(bar, parity))
    if (globaltimer_ns() - t0 > kDrainLimitNs) return;
}

}  // namespace moe
