// Completion counters between grids on one stream.
#pragma once

#include "ess_device.cuh"

namespace ess {

// Completion counters between a grid that writes per-request results and a
// later grid on the stream that may already run beside it.  The writer's CTA,
// once all of its threads' writes are done (a __syncthreads first), makes them
// visible at device scope and adds n; the reader polls with acquire loads.
// The reader may only wait on a writer whose CTAs are all resident (the
// writer launched the grids between them before the reader could launch).
__device__ __forceinline__ void count_done(int* ctr, int n) {
  __threadfence();
  atomicAdd(ctr, n);
}
// Bounded wait until *ctr >= target; false when the limit passes.
__device__ __forceinline__ bool wait_count(const int* ctr, int target) {
  const long long t0 = clock64();
  while (true) {
    int v;
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
    if (v >= target) return true;
    if (clock64() - t0 > kWaitLimitCycles) return false;
    __nanosleep(64);
  }
}

}  // namespace ess
