// Device-side status word and bounded mbarrier waits shared by every kernel.
//
// No kernel in this library may trap or spin forever. Every wait on an
// mbarrier polls with try_wait and gives up after a deadline measured on
// %globaltimer; it then records FA_DEV_TIMEOUT (with a code naming the wait
// and the CTA) in a per-translation-unit status word and raises a CTA-local
// abort flag so the CTA's other roles stop waiting too. The host reads and
// clears the status words through fa_device_status().
#pragma once
#include <cstdint>

#include "ptx.cuh"

namespace fa {

enum : uint32_t { FA_DEV_OK = 0, FA_DEV_TIMEOUT = 1, FA_DEV_BAD_INDEX = 2 };

struct DevStatus {
  uint32_t code;   // first error code recorded (0 = none)
  uint32_t where;  // which wait / check recorded it
  uint32_t block;  // linear CTA index that recorded it
  uint32_t count;  // number of reports
};

// One status word per translation unit (static: no relocatable device code needed).
static __device__ DevStatus g_status;

__device__ __forceinline__ void report_status(uint32_t code, uint32_t where) {
  if (atomicCAS(&g_status.code, 0u, code) == 0u) {
    g_status.where = where;
    g_status.block = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
  }
  atomicAdd(&g_status.count, 1u);
}

// Wait until the phase with the given parity of mbarrier `bar` has completed.
// Returns false (after recording a timeout, or seeing another role's abort) if
// it did not complete before `timeout_ns`. After one immediate test the thread
// sleeps in the barrier (up to kWaitSleepNs per try, woken when the phase
// completes) instead of spinning, so waiting warps do not take issue slots from
// the warps they share a sub-partition with; the abort flag and the deadline are
// checked between tries.
constexpr uint32_t kWaitSleepNs = 200000;
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, uint64_t timeout_ns,
                                         volatile uint32_t* abort_flag, uint32_t where) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait_sleep(bar, parity, kWaitSleepNs)) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > timeout_ns) {
      report_status(FA_DEV_TIMEOUT, where);
      *abort_flag = 1u;
      return false;
    }
  }
}


// Host-side reader for this translation unit's status word (defined per TU).
}  // namespace fa
