// Grid-wide barrier for cooperative launches (all blocks co-resident), with a bounded wait.
#pragma once

#include "dh_internal.cuh"
#include "sm100.cuh"

namespace dh {

struct GridBar {
  unsigned int count;
  unsigned int gen;
};

__device__ __forceinline__ unsigned int ld_acquire_u32(const unsigned int* p) {
  unsigned int v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Sense-reversing barrier over `expected` blocks: the last arrival resets the counter and bumps the
// generation; the others poll the generation.  A block that waits longer than limit_ns raises
// DH_ERR_TIMEOUT in *status, sets *s_fail and returns false.  The counter must start at zero
// (zero-filled workspace); every completed barrier leaves it at zero.
__device__ inline bool grid_sync(GridBar* bar, unsigned int expected, uint64_t limit_ns, int* status,
                                 volatile int* s_fail) {
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned int g = ld_acquire_u32(&bar->gen);
    __threadfence();
    const unsigned int arrived = atomicAdd(&bar->count, 1u) + 1u;
    if (arrived == expected) {
      bar->count = 0u;
      __threadfence();
      atomicAdd(&bar->gen, 1u);
    } else {
      const uint64_t t0 = sm100::globaltimer_ns();
      while (ld_acquire_u32(&bar->gen) == g) {
        if (sm100::globaltimer_ns() - t0 > limit_ns) {
          atomicOr(status, 1 << DH_ERR_TIMEOUT);
          *s_fail = 1;
          break;
        }
        __nanosleep(64);
      }
    }
    __threadfence();
  }
  __syncthreads();
  return *s_fail == 0;
}

}  // namespace dh
