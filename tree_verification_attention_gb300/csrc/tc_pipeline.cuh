// tc_pipeline.cuh - pieces shared by the two tensor-core partials kernels
// (k_partials_tc.cu: one CTA per worker; k_partials_pair.cu: a CTA pair per worker).
#pragma once

#include <cstdint>

#include "tc_ptx.cuh"
#include "tva_common.cuh"

namespace tva {

constexpr uint64_t kDrainNs = 2000000000ull;  // drain waits, and the default main-loop limit
constexpr uint32_t kNegInfBits = 0xff800000u;

// A bounded wait taken by a whole converged warp; the result is the same in every lane.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort, uint64_t limit_ns) {
  return __all_sync(0xffffffffu, ptx::mbar_wait(bar, parity, abort, limit_ns));
}

// Waits that ignore the abort flag (used only while draining).
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  volatile int never = 0;
  ptx::mbar_wait(bar, parity, &never, kDrainNs);
}

}  // namespace tva
