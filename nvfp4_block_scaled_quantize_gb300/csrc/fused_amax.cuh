// Single-launch amax for the quantize kernel: the amax of the whole tensor is needed before
// any block can be quantized, so every CTA first reduces its share of the tiles, folds the
// maxima into two workspace words with an atomic max and counts the share as arrived; once
// every share has arrived the maxima are final. These are the reduction and exchange pieces;
// the tile walk is in the quantize kernel.
//
// Page cited: "[nvfp4_training] Optimize CuteDSL kernels for NVFP4 training" (pytorch/ao pull
// request #4798), "Performance": its pipelines are an amax kernel followed by a quantize
// kernel; this folds the two into one launch.
//
// No CTA waits for another CTA to start. The tiles are split into G shares ("ranks", G = the
// grid size; rank r is every G-th tile from tile r). CTA b claims rank b when it starts, but
// a CTA that has waited a while for the arrivals claims any rank still unclaimed and does
// that share's amax itself. A CTA that has not started yet (its SM held by another stream's
// kernel, a reduced MPS share, a green context) thus never holds the others up: the waiters
// take over its share, and when it starts it finds its rank taken and only quantizes. A CTA
// quantizes every rank whose amax it computed, its own included even when its own rank was
// taken meanwhile (both CTAs then write the same bytes).
//
// Workspace words (kFuseWsWords, zero before the first launch):
//   [0] ranks arrived   [1] CTAs done with the words   [2] rowwise max   [3] columnwise max
//   [4] ranks taken over from another CTA, ever (statistics; not reset)
//   [8 .. 8 + kFuseMaxCtas / 32) one claim bit per rank
// A CTA is done with the words once its wait has ended (passed or not); the last of the G to
// get there zeroes words 0-3 and the claim bits, which readies them for the next launch. The
// next launch on the stream reads them only after this launch has ended (it waits for it at
// entry), so the reset needs no ordering beyond that, and no launch depends on host-side
// state: launches can be captured in a CUDA graph and replayed, and a launch whose wait gave
// up leaves the words ready for the next. Launches sharing a workspace must be ordered (one
// stream): launches on unordered streams would use the words at the same time.
#pragma once

#include "nvfp4_device.cuh"
#include "nvfp4_internal.h"

namespace nvfp4 {
namespace qk {

constexpr uint64_t kBarrierLimitNs = 2000000000ull;  // 2 s
// A CTA that has waited this long for the arrivals starts claiming unclaimed ranks. Far above
// the spread of CTA start times within one launch (a few microseconds), so that in an
// undisturbed launch every CTA does its own rank.
constexpr uint64_t kStealAfterNs = 20000ull;

constexpr int kFuseArrived = 0;
constexpr int kFuseDone = 1;
constexpr int kFuseMaxRow = 2;
constexpr int kFuseMaxCol = 3;
constexpr int kFuseSteals = kFuseStatsWord;
constexpr int kFuseClaims = 8;
static_assert(kFuseClaims + kFuseMaxCtas / 32 <= kFuseWsWords, "claim bits outside the workspace");

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

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ uint32_t ld_relaxed(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Claim rank r (one thread): returns the claim word's previous value; the claim succeeded
// when r's bit was clear in it.
__device__ __forceinline__ uint32_t fuse_claim(uint32_t* ws, int r) {
  return atomicOr(ws + kFuseClaims + (r >> 5), 1u << (r & 31));
}

// One share's arrival (one thread): fold the CTA's maxima (16-bit magnitudes) into the maxima
// words, then count `shares` ranks as arrived; the release orders the maxima before the count.
__device__ __forceinline__ void fuse_arrive(uint32_t* ws, uint32_t mr, uint32_t mc, uint32_t shares) {
  asm volatile("red.relaxed.gpu.global.max.u32 [%0], %1;" ::"l"(ws + kFuseMaxRow), "r"(mr) : "memory");
  asm volatile("red.relaxed.gpu.global.max.u32 [%0], %1;" ::"l"(ws + kFuseMaxCol), "r"(mc) : "memory");
  if (shares) asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(ws + kFuseArrived), "r"(shares) : "memory");
}

enum FuseWait { kFuseReady = 0, kFuseSteal = 1, kFuseTimedOut = 2 };

// Wait (one thread, bounded) until `target` ranks have arrived, then read the maxima. After
// kStealAfterNs (counted from t_start, when the CTA began waiting) the waiter looks for a rank
// that no CTA has claimed among the G ranks; if it wins one it returns kFuseSteal with the
// rank, to do that share's amax and come back. kFuseTimedOut after kBarrierLimitNs.
// may_steal = false: only wait (the CTA holds as many ranks as it can).
__device__ __forceinline__ FuseWait fuse_wait(uint32_t* ws, uint32_t target, int G, uint64_t t_start,
                                              bool may_steal, uint32_t& mr, uint32_t& mc,
                                              int& rank) {
  const int words = (G + 31) >> 5;
  uint64_t next_scan = t_start + kStealAfterNs;
  while (ld_acquire(ws + kFuseArrived) < target) {
    const uint64_t t = global_ns();
    if (t - t_start > kBarrierLimitNs) return kFuseTimedOut;
    if (!may_steal || t < next_scan) continue;
    next_scan = t + kStealAfterNs / 4;
    for (int i = 0; i < words; i++) {
      const int w = ((int)(blockIdx.x >> 5) + i) % words;
      const uint32_t valid = (w == words - 1 && (G & 31)) ? (1u << (G & 31)) - 1u : 0xFFFFFFFFu;
      uint32_t taken = ld_relaxed(ws + kFuseClaims + w);
      for (int tries = 0; tries < 32 && (~taken & valid); tries++) {
        const int b = __ffs(~taken & valid) - 1;
        const uint32_t before = atomicOr(ws + kFuseClaims + w, 1u << b);
        if (!(before & (1u << b))) {
          rank = 32 * w + b;
          atomicAdd(ws + kFuseSteals, 1u);
          return kFuseSteal;
        }
        taken = before | (1u << b);
      }
    }
  }
  mr = ld_acquire(ws + kFuseMaxRow);
  mc = ld_acquire(ws + kFuseMaxCol);
  return kFuseReady;
}

// A CTA done with the words (one thread; after its wait has ended, passed or not): counts
// itself and returns the count before it, to be handed to fuse_reset_if_last at the end.
__device__ __forceinline__ uint32_t fuse_done(uint32_t* ws) {
  return atomicAdd(ws + kFuseDone, 1u);
}

// The last of the G CTAs to be done with the words readies them for the next launch.
__device__ __forceinline__ void fuse_reset_if_last(uint32_t* ws, uint32_t done_before, int G) {
  if (done_before != (uint32_t)G - 1u) return;
  volatile uint32_t* v = ws;
  v[kFuseArrived] = 0u;
  v[kFuseMaxRow] = 0u;
  v[kFuseMaxCol] = 0u;
  for (int w = 0; w < (G + 31) >> 5; w++) v[kFuseClaims + w] = 0u;
  v[kFuseDone] = 0u;
}

}  // namespace qk
}  // namespace nvfp4
