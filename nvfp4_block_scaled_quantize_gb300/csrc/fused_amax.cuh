// Single-launch amax for the quantize kernel: every CTA reduces its share of the tensor
// (plain and, for the columnwise RHT, transformed maxima), the CTAs meet at a grid barrier,
// and each reads the per-CTA partials back. The tensor is walked from its end to its start so
// that the tiles the quantize phase reads first are the ones most recently pulled into L2.
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

// This CTA's share of max |x| (mr) and, when rht, of max |bf16(RHT(x))| over 16-row column
// blocks (mc), as 16-bit BF16 magnitudes. rows % 16 == 0 when rht.
template <bool RHT>
__device__ __forceinline__ void local_amax(const void* x, int64_t rows, int64_t cols,
                                           uint32_t sign_mask, uint32_t& mr, uint32_t& mc) {
  const int64_t gtid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t gstride = (int64_t)gridDim.x * blockDim.x;
  uint32_t m = 0, mt = 0;
  if (!RHT) {
    const uint4* p = reinterpret_cast<const uint4*>(x);
    const int64_t total = rows * cols / 8;  // 16-byte vectors
    int64_t j = gtid;
    for (; j + 3 * gstride < total; j += 4 * gstride) {
      uint4 v[4];
#pragma unroll
      for (int u = 0; u < 4; u++) v[u] = p[total - 1 - (j + u * gstride)];
#pragma unroll
      for (int u = 0; u < 4; u++)
        m = vmax2(m, vmax2(vmax2(abs2(v[u].x), abs2(v[u].y)), vmax2(abs2(v[u].z), abs2(v[u].w))));
    }
    for (; j < total; j += gstride) {
      const uint4 v = p[total - 1 - j];
      m = vmax2(m, vmax2(vmax2(abs2(v.x), abs2(v.y)), vmax2(abs2(v.z), abs2(v.w))));
    }
  } else {
    const uint2* p = reinterpret_cast<const uint2*>(x);
    const int64_t chunks = cols / 4;               // 4-column pieces of a row
    const int64_t items = (rows / 16) * chunks;    // 16-row x 4-column items
    for (int64_t j = gtid; j < items; j += gstride) {
      const int64_t it = items - 1 - j;
      const int64_t rb = it / chunks, ch = it - rb * chunks;
      uint32_t w0[16], w1[16];
#pragma unroll
      for (int i = 0; i < 16; i++) {
        const uint2 v = p[(rb * 16 + i) * chunks + ch];
        w0[i] = v.x;
        w1[i] = v.y;
      }
#pragma unroll
      for (int i = 0; i < 16; i++) m = vmax2(m, vmax2(abs2(w0[i]), abs2(w1[i])));
      rht16_pair(w0, sign_mask);
      rht16_pair(w1, sign_mask);
#pragma unroll
      for (int i = 0; i < 16; i++) mt = vmax2(mt, vmax2(abs2(w0[i]), abs2(w1[i])));
    }
  }
  mr = max(m & 0xFFFFu, m >> 16);
  mc = RHT ? max(mt & 0xFFFFu, mt >> 16) : mr;
}

// Grid barrier for a launch whose CTAs are all resident: one thread per CTA calls it.
// ws[0] counts arrivals and is reset by the last one, ws[1] is a generation number that only
// grows, so the barrier needs no clearing between launches on one stream. Returns false when
// the wait passed its limit.
__device__ __forceinline__ bool grid_sync(uint32_t* ws, uint32_t nblocks) {
  volatile uint32_t* gen = ws + 1;
  const uint32_t g = *gen;
  __threadfence();
  const uint32_t old = atomicAdd(ws, 1u);
  if (old == nblocks - 1) {
    atomicExch(ws, 0u);
    __threadfence();
    atomicAdd(ws + 1, 1u);
    return true;
  }
  uint64_t t0, t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  while (*gen == g) {
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    if (t - t0 > kBarrierLimitNs) return false;
    __nanosleep(128);
  }
  __threadfence();
  return true;
}

}  // namespace qk
}  // namespace nvfp4
