// Completion counters between grids on one stream.
#pragma once

#include "ess_device.cuh"

namespace ess {

// Ints from one counter to the next: each sits in a 128-byte line of its own,
// so the readers polling different counters load different L2 lines.
constexpr int kCounterStride = 32;

// Completion counters between a grid that writes per-request results and a
// later grid on the stream that may already run beside it.  The writer's CTA,
// once all of its threads' writes are done (a __syncthreads first), makes them
// visible at device scope and adds n; the reader polls with acquire loads.
// The reader may only wait on a writer whose CTAs are all resident (the
// writer launched the grids between them before the reader could launch).
// Orders this thread's completed bulk (async-proxy) writes to global memory
// before its later generic accesses, ahead of a count_done.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}
__device__ __forceinline__ void count_done(int* ctr, int n) {
  __threadfence();
  atomicAdd(ctr, n);
}
// Bounded wait until *ctr >= target; false when the limit passes.  The polls
// back off from 64 to 512 ns apart, so that many waiting CTAs load the
// counter's line a few hundred million times a second at most.
__device__ __forceinline__ bool wait_count(const int* ctr, int target) {
  const long long t0 = clock64();
  unsigned ns = 64;
  while (true) {
    int v;
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
    if (v >= target) return true;
    if (clock64() - t0 > kWaitLimitCycles) return false;
    __nanosleep(ns);
    if (ns < 512) ns <<= 1;
  }
}

}  // namespace ess
