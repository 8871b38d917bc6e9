// Bounded mbarrier waits.  Every wait in the kernels goes through these: a
// wait that exceeds its time limit records a timeout in the device status
// word, raises the CTA's abort flag and returns false, so the kernel can
// release its tensor memory and return instead of hanging.
#pragma once

#include "kernels.cuh"
#include "sm103_ptx.cuh"

namespace slope {

// Longest hardware sleep per try_wait (the thread wakes as soon as the phase completes).
constexpr uint32_t kWaitSleepNs = 100000;

__device__ __forceinline__ void record_timeout(int* status, int site) {
  if (atomicCAS(status, 0, kStatusTimeout) == 0) atomicExch(status + 1, site);
}

// Waits for the phase of `bar` with the given parity to complete.  Gives up
// when the CTA-local abort flag is raised by another role or when
// `limit_ns` elapses (then raises the flag itself).
__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity, volatile int* cta_abort,
                                             int* status, uint64_t limit_ns, int site) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait_sleep(bar, parity, kWaitSleepNs)) return true;
    if (*cta_abort) return false;
    if (globaltimer_ns() - t0 > limit_ns) {
      *cta_abort = 1;
      record_timeout(status, site);
      return false;
    }
  }
}

// Same, but ignores the abort flag: used after an abort to let operations
// already in flight land before the CTA releases its resources.
__device__ __forceinline__ bool wait_final(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait_sleep(bar, parity, kWaitSleepNs)) {
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
  return true;
}

}  // namespace slope
