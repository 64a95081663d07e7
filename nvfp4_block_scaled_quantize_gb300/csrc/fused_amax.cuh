// Single-launch amax for the quantize kernel: every CTA reduces the tiles it is about to
// quantize (plain and, for the columnwise RHT, transformed maxima), the CTAs meet at a grid
// barrier, and each reads the per-CTA partials back. These are the reduction and barrier
// pieces; the tile walk is in the quantize kernel.
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

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_gpu(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void st_relaxed_gpu(uint32_t* p, uint32_t v) {
  asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t atom_add_acq_rel_gpu(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// Grid barrier for a launch whose CTAs are all resident: one thread per CTA calls it, after
// its own writes that the other CTAs read. ws[0] counts arrivals; the last arrival resets it
// and publishes the release by bumping the generation ws[1], which only grows, so the
// barrier needs no clearing between launches on one stream. Returns false when the wait
// passed its limit.
__device__ __forceinline__ bool grid_sync(uint32_t* ws, uint32_t nblocks) {
  const uint32_t g = ld_acquire_gpu(ws + 1);  // cannot change before this CTA arrives
  if (atom_add_acq_rel_gpu(ws, 1u) == nblocks - 1) {
    st_relaxed_gpu(ws, 0u);        // nobody else touches the count until the next launch
    st_release_gpu(ws + 1, g + 1u);
    return true;
  }
  uint64_t t0, t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  while (ld_acquire_gpu(ws + 1) == g) {
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    if (t - t0 > kBarrierLimitNs) return false;
  }
  return true;
}

}  // namespace qk
}  // namespace nvfp4
