// Bounded mbarrier waits shared by the forward and backward kernels.
// `Params` supplies `status` (device status word) and `timeout_ns`.
#pragma once

#include <cstdint>

#include "sm103_ptx.cuh"

namespace attn {

// Compile-time flag passed to generic lambdas, to compile a loop twice (for
// instance with and without a mask test the compiler would otherwise turn
// into a select on every element).
template <bool B>
struct BoolTag {
  static constexpr bool value = B;
};

// Bounded wait.  Returns false if the CTA is aborting or the wait ran out.
// After one immediate test the thread sleeps in try_wait (woken when the
// phase completes, or after at most 20 us), so waiting warps do not take
// issue slots from the working ones; abort flag and clock are checked
// between sleeps.
template <class Params>
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity,
                                             volatile int* abort_flag,
                                             const Params& p, int role) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  while (true) {
    if (ptx::mbar_try_wait_sleep(bar, parity, 20000u)) return true;
    if (*abort_flag) return false;
    if (ptx::globaltimer_ns() - t0 > p.timeout_ns) {
      *abort_flag = 1;
      atomicOr(p.status, 1u | (static_cast<unsigned>(role) << 8));
      return false;
    }
  }
}

// Wait used while tearing down after an abort: ignores the abort flag.
template <class Params>
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity,
                                           const Params& p) {
  const uint64_t t0 = ptx::globaltimer_ns();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (ptx::globaltimer_ns() - t0 > p.timeout_ns) return;
  }
}

}  // namespace attn
