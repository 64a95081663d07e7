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

// Workspace words of the single-launch amax (kFuseWsWords, 8-byte aligned): [0] and [1] the
// arrival counts of launches with even and odd epochs, [2..3] and [4..5] the rowwise and
// columnwise maxima as (epoch << 16) | 16-bit magnitude, [6..7] the epoch (64 bits, so tags
// stay below 2^48 for longer than any process runs). A launch reads the epoch E when it starts,
// counts its arrivals on word E & 1 and tags its maxima with E + 1; once CTA 0 has seen every
// arrival (or given up) it zeroes the other count, which the next launch uses, and stores
// E + 1. Every CTA has read E before it arrives, and the next launch on the stream reads the
// words only once this one has ended (even when it starts early, it waits for this launch at
// entry), so plain stores suffice and no launch depends on host-side state: launches can be
// captured in a CUDA graph and replayed, and a launch whose barrier timed out leaves the words
// ready for the next. Launches sharing a workspace must be ordered (one stream): launches on
// unordered streams would use the words at the same time.

// The epoch (one thread per CTA, at the start of the launch; the value is needed only at the
// arrival, so the load's latency hides behind the amax phase).
__device__ __forceinline__ uint64_t fuse_epoch(const uint32_t* ws) {
  unsigned long long e;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(e) : "l"(ws + 6) : "memory");
  return e;
}

// Arrival of this CTA (one thread): fold its maxima (16-bit magnitudes) into the two maxima
// words under the launch's tag, then count itself; the release orders the maxima before the
// count. Tags grow from launch to launch, so the atomic max needs no clearing in between.
__device__ __forceinline__ void fuse_arrive(uint32_t* ws, uint64_t epoch, uint32_t mr, uint32_t mc) {
  unsigned long long* mx = reinterpret_cast<unsigned long long*>(ws + 2);
  const unsigned long long tag = epoch + 1u;
  const unsigned long long vr = (tag << 16) | mr, vc = (tag << 16) | mc;
  asm volatile("red.relaxed.gpu.global.max.u64 [%0], %1;" ::"l"(mx), "l"(vr) : "memory");
  asm volatile("red.relaxed.gpu.global.max.u64 [%0], %1;" ::"l"(mx + 1), "l"(vc) : "memory");
  asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(ws + (epoch & 1u)) : "memory");
}

// Wait (one thread, bounded) until `target` CTAs have arrived, then read the maxima of every
// CTA. Returns false when the wait passed its limit or the maxima carry another tag.
__device__ __forceinline__ bool fuse_wait(const uint32_t* ws, uint64_t epoch, uint32_t target,
                                          uint32_t& mr, uint32_t& mc) {
  const uint32_t* count = ws + (epoch & 1u);
  uint32_t c;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(c) : "l"(count) : "memory");
  if (c < target) {
    uint64_t t0, t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
    do {
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
      if (t - t0 > kBarrierLimitNs) return false;
      asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(c) : "l"(count) : "memory");
    } while (c < target);
  }
  unsigned long long vr, vc;
  const unsigned long long* mx = reinterpret_cast<const unsigned long long*>(ws + 2);
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(vr) : "l"(mx) : "memory");
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(vc) : "l"(mx + 1) : "memory");
  if ((vr >> 16) != epoch + 1u || (vc >> 16) != epoch + 1u) return false;
  mr = (uint32_t)vr & 0xFFFFu;
  mc = (uint32_t)vc & 0xFFFFu;
  return true;
}

// CTA 0, once its wait has ended (passed or not): ready the words for the next launch.
__device__ __forceinline__ void fuse_advance(uint32_t* ws, uint64_t epoch) {
  const unsigned long long next = epoch + 1u;
  asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(ws + (next & 1u)), "r"(0u) : "memory");
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(ws + 6), "l"(next) : "memory");
}

}  // namespace qk
}  // namespace nvfp4
