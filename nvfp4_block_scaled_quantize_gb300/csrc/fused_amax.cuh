// Single-launch amax for the quantize kernel: every CTA reduces the tiles it is about to
// quantize (plain and, for the columnwise RHT, transformed maxima), folds them into two
// launch-tagged maxima words with an atomic max, counts its arrival, and waits until every
// CTA has arrived (a grid barrier that carries the result). These are the reduction and
// exchange pieces; the tile walk is in the quantize kernel.
//
// Page cited: "[nvfp4_training] Optimize CuteDSL kernels for NVFP4 training" (pytorch/ao pull
// request #4798), "Performance": its pipelines are an amax kernel followed by a quantize
// kernel; this folds the two into one launch.
#pragma once

#include "nvfp4_device.cuh"
#include "nvfp4_internal.h"

namespace nvfp4 {
namespace qk {

constexpr uint64_t kBarrierLimitNs = 2000000000ull;  // 2 s

// Max over the CTA of a 16-bit magnitude held in a 32-bit word (every thread gets it).
// red: 32 words of shared memory, free on entry.
__device__ __forceinline__ uint32_t cta_max(uint32_t v, volatile uint32_t* red) {
  v = __reduce_max_sync(0xFFFFFFFFu, v);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) red[warp] = v;
  __syncthreads();
  uint32_t r = 0;
  for (int w = 0; w < (int)(blockDim.x >> 5); w++) r = max(r, red[w]);
  __syncthreads();
  return r;
}

// Arrival of this CTA (one thread): fold its maxima (16-bit magnitudes) into the launch's two
// maxima words, then count itself; the release orders the maxima before the count.
__device__ __forceinline__ void fuse_arrive(uint32_t* ws, uint64_t epoch, uint32_t mr,
                                            uint32_t mc) {
  unsigned long long* mx = reinterpret_cast<unsigned long long*>(ws + 2);
  const unsigned long long vr = (epoch << 16) | mr, vc = (epoch << 16) | mc;
  asm volatile("red.relaxed.gpu.global.max.u64 [%0], %1;" ::"l"(mx), "l"(vr) : "memory");
  asm volatile("red.relaxed.gpu.global.max.u64 [%0], %1;" ::"l"(mx + 1), "l"(vc) : "memory");
  asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(ws) : "memory");
}

// Wait (one thread, bounded) until the arrival count reaches `target`, then read the maxima
// of every CTA. Returns false when the wait passed its limit or the maxima carry another epoch.
__device__ __forceinline__ bool fuse_wait(uint32_t* ws, uint32_t target, uint64_t epoch,
                                          uint32_t& mr, uint32_t& mc) {
  uint32_t c;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(c) : "l"(ws) : "memory");
  if ((int32_t)(c - target) < 0) {
    uint64_t t0, t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
    do {
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
      if (t - t0 > kBarrierLimitNs) return false;
      asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(c) : "l"(ws) : "memory");
    } while ((int32_t)(c - target) < 0);
  }
  unsigned long long vr, vc;
  const unsigned long long* mx = reinterpret_cast<const unsigned long long*>(ws + 2);
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(vr) : "l"(mx) : "memory");
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(vc) : "l"(mx + 1) : "memory");
  if ((vr >> 16) != epoch || (vc >> 16) != epoch) return false;
  mr = (uint32_t)vr & 0xFFFFu;
  mc = (uint32_t)vc & 0xFFFFu;
  return true;
}

}  // namespace qk
}  // namespace nvfp4
