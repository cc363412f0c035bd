// Bounded mbarrier waits shared by the tensor-core kernels.  Every wait
// has a time limit (globaltimer); a wait that runs out sets a CTA-wide abort
// flag and the device status word, so that all roles leave their loops and
// the kernel can drain its copies and MMAs, free TMEM and return.
#pragma once

#include "msa_common.cuh"
#include "tc_ptx.cuh"

namespace msa {

constexpr uint64_t kDrainLimitNs = 4000000000ull;

struct WaitCtl {
  volatile int* abort;
  int* status;
  uint64_t limit;
};

// Bounded wait on phase `parity` of an mbarrier.  Returns false when the
// CTA is aborting (flag set by another role, or this wait ran out).  The
// first probe does not block; a limit of at most 1 ns (a test setting) makes
// every wait that this probe does not find complete run out.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const WaitCtl& c) {
  if (ptx::mbar_test_wait(bar, parity)) return true;
  if (c.limit > 1) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer();
    while (true) {
      if (ptx::mbar_try_wait(bar, parity)) return true;
      if (*c.abort) return false;
      if (ptx::globaltimer() - t0 > c.limit) break;
    }
  } else if (*c.abort) {
    return false;
  }
  *c.abort = 1;
  record_status(c.status, MSA_ERR_TIMEOUT);
  return false;
}

// Bounded wait taken by a whole warp, with one result for all its lanes.
__device__ __forceinline__ bool wait_w(uint32_t bar, uint32_t parity, const WaitCtl& ctl) {
  return __all_sync(0xffffffffu, wait_bar(bar, parity, ctl));
}

// Wait used while draining: ignores the abort flag, fixed limit.
__device__ __forceinline__ void drain_bar(uint32_t bar, uint32_t parity, int* status) {
  if (ptx::mbar_try_wait(bar, parity)) return;
  const uint64_t t0 = ptx::globaltimer();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (ptx::globaltimer() - t0 > kDrainLimitNs) {
      record_status(status, MSA_ERR_TIMEOUT);
      return;
    }
  }
}

}  // namespace msa
