// One grid-wide barrier per launch for the library's cooperative kernels
// (every block of the launch is resident at once), on two 32-bit words of
// device memory that start at zero: bar[0] counts arrivals, bar[1]
// departures.  Every block calls grid_barrier_wait once and
// grid_barrier_depart once, on every path out of the kernel; the last block to
// depart sets both words back to zero, so the next launch needs no memset
// (a graph replays the kernel alone).  The wait is bounded by wall time.
#pragma once
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace cbmoe {

__device__ __forceinline__ unsigned int ld_acquire_gpu_u32(const unsigned int* p) {
  unsigned int v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// All threads of the block call it.  The block's global writes before the
// call are visible to every block after it.  Returns false (and records
// CB_ERR_TIMEOUT in *err) when `expected` arrivals did not come within
// limit_ns.  `ok_smem` is a shared int for the result.
__device__ __forceinline__ bool grid_barrier_wait(unsigned int* bar, unsigned int expected, uint64_t limit_ns,
                                                  int* err, int* ok_smem) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(bar, 1u);
    const uint64_t start = globaltimer_ns();
    int ok = 1;
    while (ld_acquire_gpu_u32(bar) < expected) {
      if (globaltimer_ns() - start > limit_ns) {
        set_error(err, kErrTimeout);
        ok = 0;
        break;
      }
      __nanosleep(64);
    }
    __threadfence();
    *ok_smem = ok;
  }
  __syncthreads();
  return *ok_smem != 0;
}

// One thread of the block calls it, after the block's barrier wait has ended
// (passed or timed out); the last of the G blocks zeroes the two words.
__device__ __forceinline__ void grid_barrier_depart(unsigned int* bar, unsigned int G) {
  if (atomicAdd(bar + 1, 1u) == G - 1) {
    atomicExch(bar, 0u);
    atomicExch(bar + 1, 0u);
  }
}

}  // namespace cbmoe
