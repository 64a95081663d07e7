// The quantize kernel: rowwise, columnwise (optionally after the 16-point RHT, with RTNE or
// stochastic rounding) and 16x16 2D NVFP4 quantization of BF16 tensors from ONE read of the
// input, for plain tensors and for grouped (MoE) tensors split into row segments.
//
// Page cited: "[nvfp4_training] Optimize CuteDSL kernels for NVFP4 training" (pytorch/ao pull
// request #4798). Its "linear fused" / "grouped fused" row+col kernels and its 2D weight
// kernel are the prior art; this is a design for sm_103a:
//   * one persistent CTA per SM keeps kStages 64 x 256 BF16 tiles in flight with TMA
//     (cp.async.bulk.tensor) completing on mbarriers; kGroups groups of four warps each take a
//     whole tile, one warp per 16-row slab, and refill the stage as soon as the four slabs sit
//     in registers (12 warps: three per SM sub-partition, so up to 168 registers each);
//   * each lane holds a 16-row x 8-column piece of its slab, read from shared memory once for
//     both orientations: a rowwise 1x16 block is a lane pair ("Optimization" item 7: a warp
//     covers several tokens x hidden blocks), a columnwise block is one lane's column
//     (thread-local maximum, RHT butterflies and conversion);
//   * scale reciprocals come from a per-group 128-entry table indexed by the E4M3 code, built
//     once per segment with the exact (div_rn) reciprocal ("Fast math");
//   * columnwise codes of the four slabs are staged in shared memory in the layout of a TMA
//     store's box and leave by one tensor store per tile (a 3D view of the output in which the
//     tile's 256 columns are one box), the scales as one 4-byte store per column
//     ("Optimization" item 5);
//   * a grouped tensor is tiled in the space of its columnwise outputs, where each segment's
//     rows sit padded to whole 16-row slabs, back to back: a tile is four consecutive slabs,
//     from one segment or from several, loaded as one box when they are consecutive rows of x
//     and slab by slab otherwise. No tile is partly empty except the last, and every tile's
//     columnwise codes are whole 32-byte column runs;
//   * 2D row+col: the columnwise codes are the rowwise codes transposed in registers;
//   * stochastic rounding uses one Philox4x32-10 draw per 16-element block, all four words
//     consumed by cvt.rs.satfinite.e2m1x4 ("Optimization" item 3).
// Variants: FUSED adds the amax of a plain tensor inside the launch (an amax phase over the
// same stage ring, then a wait for every CTA's arrival); AMAX_ONLY is that amax pass alone,
// per segment (fused_amax.cuh, amax_pass.cu).
// Every wait on an mbarrier gives up after a time limit; the kernel then records
// NVFP4_DEVICE_TIMEOUT and leaves after the loads it issued have landed (bounded too).
#pragma once

#include "fused_amax.cuh"
#include "nvfp4_device.cuh"
#include "nvfp4_internal.h"

namespace nvfp4 {
namespace qk {

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s: no TMA load takes this long

struct Coord {
  int32_t n0;      // first column
  int32_t colpos;  // first column of the tile in the columnwise outputs (a multiple of kTileM)
  int32_t tile;    // the tile these coordinates belong to (checked by the consumers)
  int32_t nvalid;  // slabs that hold rows of a segment (the first nvalid of the four)
  int32_t row0[kWarpsPerGroup];   // first row of each 16-row slab in x
  int32_t nrows[kWarpsPerGroup];  // rows of each slab inside its segment (0: no slab)
  int32_t seg[kWarpsPerGroup];    // segment of each slab (slab 0's where there is no slab)
};
static_assert(sizeof(Coord) == 64, "coordinate record size");

// What the column write-out of a tile needs after its coordinates' stage has been refilled.
struct OutPos {
  int32_t n0, colpos, nvalid;
};

// Byte offset of scale (r, c) in the 128 x 4 tiled layout of the block-scaled GEMMs' scale
// factors (the scale matrix zero-padded to whole 128 x 4 tiles, tiles_c tiles per tile row, 512
// bytes each in row-major tile order; inside a tile, row r % 128 = 32 i + q and column j sit at
// 16 q + 4 i + j).
__device__ __forceinline__ int64_t swz_scale_off(int64_t r, int64_t c, int64_t tiles_c) {
  return ((r >> 7) * tiles_c + (c >> 2)) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (c & 3);
}

// Columnwise code staging in the layout of the TMA store's box: column 8 y + z of the tile
// (y = 0..31, z = 0..7) at z * 1024 + y * 32, its 32 bytes the four slabs' 8 bytes in order,
// the two 16-byte halves swapped where bit 2 of y is set (the 32-byte swizzle). Lane l's
// column 8 l + z, slab sl:
__device__ __forceinline__ int col_stage_off(int l, int z, int sl) {
  return z * 1024 + l * 32 + ((((sl >> 1) ^ (l >> 2)) & 1) << 4) + ((sl & 1) << 3);
}

__device__ __forceinline__ uint32_t comp(const uint4& v, int k) {
  return k == 0 ? v.x : (k == 1 ? v.y : (k == 2 ? v.z : v.w));
}

// Packed magnitude of the two halves, merged across two rows: returns (max row a, max row b)
// as a pair of 16-bit magnitudes, each the max over the four words of its row.
__device__ __forceinline__ uint32_t row_pair_max(const uint4& a, const uint4& b) {
  const uint32_t ma = hmax_abs2(hmax_abs2(a.x, a.y), hmax_abs2(a.z, a.w));
  const uint32_t mb = hmax_abs2(hmax_abs2(b.x, b.y), hmax_abs2(b.z, b.w));
  return hmax_abs2(__byte_perm(ma, mb, 0x5410), __byte_perm(ma, mb, 0x7632)) & 0x7FFF7FFFu;
}

// max |w| over 16 packed BF16 pairs, per half, as a balanced tree; sign bits cleared.
__device__ __forceinline__ uint32_t tree_max16(const uint32_t (&w)[16]) {
  uint32_t a[8];
#pragma unroll
  for (int i = 0; i < 8; i++) a[i] = hmax_abs2(w[2 * i], w[2 * i + 1]);
  const uint32_t b0 = hmax_abs2(a[0], a[1]), b1 = hmax_abs2(a[2], a[3]);
  const uint32_t b2 = hmax_abs2(a[4], a[5]), b3 = hmax_abs2(a[6], a[7]);
  return hmax_abs2(hmax_abs2(b0, b1), hmax_abs2(b2, b3)) & 0x7FFF7FFFu;
}

// Eight scaled values -> eight codes in 32 bits, element 0 in bits 3:0. RTNE: four
// cvt.rn.satfinite.e2m1x2.f32 (first operand -> high nibble); SR: two
// cvt.rs.satfinite.e2m1x4.f32 with random words w0 (elements 0..3) and w1 (4..7), operands
// a, b, e, f = elements 3, 2, 1, 0 of each group.
template <bool SR>
__device__ __forceinline__ uint32_t e2m1x8(float t0, float t1, float t2, float t3, float t4,
                                           float t5, float t6, float t7, uint32_t w0,
                                           uint32_t w1) {
  uint32_t d;
  if (SR) {
    asm("{\n\t.reg .b16 h0, h1;\n\t"
        "cvt.rs.satfinite.e2m1x4.f32 h0, {%4, %3, %2, %1}, %9;\n\t"
        "cvt.rs.satfinite.e2m1x4.f32 h1, {%8, %7, %6, %5}, %10;\n\t"
        "mov.b32 %0, {h0, h1};\n\t}"
        : "=r"(d)
        : "f"(t0), "f"(t1), "f"(t2), "f"(t3), "f"(t4), "f"(t5), "f"(t6), "f"(t7), "r"(w0),
          "r"(w1));
  } else {
    asm("{\n\t.reg .b8 q0, q1, q2, q3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 q0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 q1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 q2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 q3, %8, %7;\n\t"
        "mov.b32 %0, {q0, q1, q2, q3};\n\t}"
        : "=r"(d)
        : "f"(t0), "f"(t1), "f"(t2), "f"(t3), "f"(t4), "f"(t5), "f"(t6), "f"(t7));
  }
  return d;
}

// Transpose of an 8 x 8 block of 4-bit codes: on entry w[i] holds row i (nibble j = column
// j), on exit w[j] holds column j (nibble i = row i). Swaps 4x4, then 2x2, then single-nibble
// blocks (byte permutes, then masks).
__device__ __forceinline__ void transpose_nibbles8(uint32_t* w) {
#pragma unroll
  for (int i = 0; i < 4; i++) {
    const uint32_t a = w[i], b = w[i + 4];
    w[i] = __byte_perm(a, b, 0x5410);
    w[i + 4] = __byte_perm(a, b, 0x7632);
  }
#pragma unroll
  for (int i = 0; i < 8; i++) {
    if ((i & 2) == 0) {
      const uint32_t a = w[i], b = w[i + 2];
      w[i] = __byte_perm(a, b, 0x6240);
      w[i + 2] = __byte_perm(a, b, 0x7351);
    }
  }
#pragma unroll
  for (int i = 0; i < 8; i += 2) {
    const uint32_t a = w[i], b = w[i + 1];
    w[i] = (a & 0x0F0F0F0Fu) | ((b << 4) & 0xF0F0F0F0u);
    w[i + 1] = ((a >> 4) & 0x0F0F0F0Fu) | (b & 0xF0F0F0F0u);
  }
}

// A warp's own scale block (kTableBlock) for segment scales q = {S_enc row, S_dec row, S_enc
// col, S_dec col}: the rowwise and columnwise reciprocal tables and the two encode scales.
// Out of line: it runs only for a slab whose segment is not its group's, and kept out of the
// tile loop's code it leaves that loop's register allocation alone.
static __device__ __noinline__ void build_scale_block(float* blk, float4 q, int lane, int fast) {
  __syncwarp();  // every lane is done with the block's previous contents
#pragma unroll 1
  for (int c = lane; c < kTableEntries; c += 32) {
    const float sv = e4m3x2_to_float2((uint16_t)c).x;
    blk[c] = fast ? element_multiplier_fast(sv, q.y) : element_multiplier(sv, q.y);
    blk[kTableEntries + c] = fast ? element_multiplier_fast(sv, q.w) : element_multiplier(sv, q.w);
  }
  if (lane == 0) {
    blk[2 * kTableEntries] = q.x;
    blk[2 * kTableEntries + 1] = q.z;
  }
  __syncwarp();
}

// Bounded wait until at least `count` loads have been issued into stage s (a monotonic
// per-stage count). Only then does the mbarrier parity of load count - 1 name its phase
// unambiguously: the previous load of the stage has been consumed, so its phase is complete.
__device__ __forceinline__ bool wait_issued(volatile int32_t* issued, int s, int count) {
  if (issued[s] >= count) return true;
  uint64_t t0;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  while (issued[s] < count) {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    if (t - t0 > kWaitLimitNs) return false;
    __nanosleep(64);
  }
  return true;
}

// FUSED: the amax is computed inside the launch (a.fused == 1; a plain tensor; fused_amax.cuh).
// A template parameter, so that each path is compiled on its own.
// AMAX_ONLY: the amax pass alone, through the same stage ring: per segment max |x| and, with
// RHT, max |bf16(RHT)| over its zero-padded 16-row column blocks, atomically maxed into
// a.amax_row / a.amax_col (zeroed by the caller); no codes. Instantiated with ROW and !COL.
// FAST_RHT: fast math with the RHT (columnwise codes from the FP32 transform, no BF16
// round-through). SWZ: both scale outputs in the GEMMs' tiled layout (a.swz_scales).
// GROUPED: a tensor split into segments (a.offsets); never FUSED or SWZ.
template <bool ROW, bool COL, bool RHT, bool TWO_D, bool SR_ROW, bool SR_COL, bool FUSED,
          bool AMAX_ONLY = false, bool FAST_RHT = false, bool SWZ = false, bool GROUPED = false>
__global__ void __launch_bounds__(kQuantThreads, 1)
    quantize_tiles_kernel(const __grid_constant__ QuantArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  // 2D with both orientations: the columnwise codes are the rowwise codes transposed
  constexpr bool kRowCol2D = ROW && COL && TWO_D;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  // Launched with programmatic dependent launch, the kernel may start before the previous
  // kernel in the stream has finished: wait for it before touching any memory, since that
  // kernel may have produced x or still use the workspace and the outputs. The next kernel
  // may start at once (it waits for this one in turn), except after a single-launch kernel,
  // which lets it start only once past its grid barrier (below).
  pdl_wait();
  if (!FUSED) pdl_allow_next();

  // grouped: per segment {first slab in the padded columnwise space, first row, end row, the
  // next segment's first slab}; [E] = {slab count, rows, rows, INT_MAX}
  int4* seg_rec = reinterpret_cast<int4*>(smem + kSmemSegRec);
  float4* seg_scale = reinterpret_cast<float4*>(smem + kSmemSegScale);
  Coord* coords = reinterpret_cast<Coord*>(smem + kSmemCoords);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kSmemBars);
  volatile int32_t* flags = reinterpret_cast<volatile int32_t*>(smem + kSmemFlags);
  volatile int32_t* issued = reinterpret_cast<volatile int32_t*>(smem + kSmemIssued);
  // grouped: per warp, the segment its last issue_slab() found (any index is a valid start)
  int32_t* seg_hint = reinterpret_cast<int32_t*>(smem + kSmemSegHint);

  const int E = a.segments;
  const int tiles_n = (int)((a.cols + kTileN - 1) / kTileN);
  const int64_t N = a.cols;

  const int stride = gridDim.x;
  int n_slabs = 0;  // grouped: slabs of all segments
  constexpr bool fused = FUSED;
  // A plain tensor is one segment: the first loads leave at once, before anything else
  // (the grouped path first needs the segment table below).
  constexpr bool plain = !GROUPED;
  static_assert(!GROUPED || (!FUSED && !SWZ), "grouped tensors: no single-launch amax, no tiled scales");
  int total = 0, n_local = 0;

  // Single-launch amax (fused_amax.cuh): the ranks this CTA computes the amax of, in order,
  // each with the first slot of its amax round. Slots number the CTA's loads through the stage
  // ring: slot k goes to stage k % kStages as that stage's load k / kStages. Rank r walks its
  // tiles r, r + G, ... from the last to the first.
  int32_t* held_rank = reinterpret_cast<int32_t*>(smem + kSmemHeld);
  int32_t* held_first = held_rank + kMaxHeld;
  // [0] ranks held, [1] the action after a wait (FuseWait), [2] the rank taken over
  volatile int32_t* fctl = reinterpret_cast<volatile int32_t*>(smem + kSmemFuseCtl);
  auto rank_tiles = [&](int r) -> int { return r < total ? (total - r + stride - 1) / stride : 0; };
  auto tile_of_slot = [&](int k) -> int {
    const int nh = fctl[0];
    for (int h = 0; h < nh; h++) {
      const int r = held_rank[h], n = rank_tiles(r), f = held_first[h];
      if (k < f + n) return r + (n - 1 - (k - f)) * stride;
    }
    return -1;
  };

  // Load tile `tile` into stage s. Tile (mt, nt) is columns nt * kTileN.. and slabs 4 mt..
  // 4 mt + 3: rows 64 mt.. of a plain tensor (one box, one arrival on the stage's mbarrier);
  // for a grouped tensor, slabs of the padded columnwise space (segment e's slabs are
  // seg_rec[e].x.., its rows 16 at a time), each loaded as a box of its own, with one arrival
  // per slab (issue_slab). The consumers read the coordinate record after their wait on the
  // stage's mbarrier, whose phase completes only after these arrivals (release; the wait
  // acquires).
  auto issue_slab = [&](int tile, int s, int k) {  // grouped: slab k of the tile
    Coord* cp = coords + s;
    const int mt = tile / tiles_n;
    const int n0 = (tile - mt * tiles_n) * kTileN;
    const int j = 4 * mt + k;
    if (k == 0) {
      cp->n0 = n0;
      cp->colpos = mt * kTileM;
      cp->tile = tile;
      cp->nvalid = min(kWarpsPerGroup, n_slabs - 4 * mt);
    }
    if (j < n_slabs) {
      // The segment of slab j: the one this warp's last call found, where it still holds j
      // (tiles are walked forward), else a binary search for the largest e whose first slab
      // is at most j (never an empty segment: the next one starts at the same slab).
      int e = seg_hint[warp];
      int4 r = seg_rec[e];
      if (AMAX_ONLY) {  // a few steps forward first (each warp walks its tiles forward)
#pragma unroll 1
        for (int step = 0; step < 4 && j >= r.w; step++) r = seg_rec[++e];
      }
      if (j < r.x || j >= r.w) {
        int lo = 0, hi = E;
        while (hi - lo > 1) {
          const int mid = (lo + hi) >> 1;
          if (seg_rec[mid].x <= j) lo = mid; else hi = mid;
        }
        e = lo;
        r = seg_rec[e];
      }
      seg_hint[warp] = e;
      const int row0 = r.y + 16 * (j - r.x);
      cp->row0[k] = row0;
      cp->nrows[k] = min(16, r.z - row0);
      cp->seg[k] = e;
      if (k == 0) issued[s] = issued[s] + 1;  // the stage's next mbarrier phase is this load's
      mbar_expect_tx(&full[s], kSlabBytes);
      tma_load_2d(smem + kSmemStages + s * kStageBytes + k * kSlabBytes, &a.tmap_slab, n0, row0,
                  &full[s]);
    } else {  // past the last slab (the last tile row only; never slab 0)
      cp->row0[k] = 0;
      cp->nrows[k] = 0;
      cp->seg[k] = -1;
      mbar_arrive(&full[s]);
    }
  };
  auto issue = [&](int tile, int s) {
    if (GROUPED) {
      for (int k = 0; k < kWarpsPerGroup; k++) issue_slab(tile, s, k);
      return;
    }
    Coord* cp = coords + s;
    const int mt = tile / tiles_n;
    const int n0 = (tile - mt * tiles_n) * kTileN;
    cp->n0 = n0;
    cp->colpos = mt * kTileM;
    cp->tile = tile;
    const int64_t rem = a.rows - (int64_t)mt * kTileM;  // rows from the tile's first on
    int nvalid = 0;
#pragma unroll
    for (int k = 0; k < kWarpsPerGroup; k++) {
      const int64_t rk = rem - 16 * k;
      cp->row0[k] = mt * kTileM + 16 * k;
      cp->nrows[k] = rk >= 16 ? 16 : (rk > 0 ? (int)rk : 0);
      cp->seg[k] = 0;
      nvalid += rk > 0 ? 1 : 0;
    }
    cp->nvalid = nvalid;
    issued[s] = issued[s] + 1;  // the stage's next mbarrier phase is this load's
    mbar_expect_tx(&full[s], kStageBytes);
    tma_load_2d(smem + kSmemStages + s * kStageBytes, &a.tmap, n0, mt * kTileM, &full[s]);
  };
  // The first kStages loads: the quantize phase's first tiles, or, with the single-launch
  // amax, the amax phase's (its slots walk the tiles from the last to the first, so that the
  // quantize phase, walking forward, starts on the kStages tiles still in shared memory).
  auto first_loads = [&]() {
    prefetch_tensormap(&a.tmap);
    if (!plain) prefetch_tensormap(&a.tmap_slab);
    for (int s = 0; s < kStages; s++) {
      mbar_init(&full[s], GROUPED ? kWarpsPerGroup : 1);  // grouped: one arrival per slab
      issued[s] = 0;
    }
    fence_barrier_init();
    for (int k = 0; k < kStages && k < n_local; k++)
      issue(fused ? tile_of_slot(k) : (int)blockIdx.x + k * stride, k);
  };

  if (plain) {
    const int tiles_m = (int)((a.rows + kTileM - 1) / kTileM);
    total = tiles_m * tiles_n;
    n_local = (int)blockIdx.x < total ? (total - (int)blockIdx.x + stride - 1) / stride : 0;
    if (tid == 0) {
      flags[0] = flags[1] = flags[2] = flags[3] = 0;
      if (fused) {
        // test hook: the last a.fuse_late CTAs hold back until every rank has arrived, so
        // that the others must take their ranks over (bounded)
        if (a.fuse_late > 0 && (int)blockIdx.x >= stride - a.fuse_late) {
          const uint64_t t0 = global_ns();
          while (ld_acquire(a.fuse_ws + kFuseArrived) < (uint32_t)(stride + a.fuse_extra) &&
                 global_ns() - t0 < kBarrierLimitNs) {
          }
        }
        fctl[0] = 1;
        held_rank[0] = blockIdx.x;  // this CTA's own rank first
        held_first[0] = 0;
      }
      first_loads();
    }
    __syncthreads();
  } else {
    // ---- segment table: starts, ends, first slabs in the padded columnwise space ----
    if (tid < 4) flags[tid] = 0;
    __syncthreads();
    for (int e = tid; e < E; e += blockDim.x) {
      const int32_t start = e == 0 ? 0 : a.offsets[e - 1];
      const int32_t end = a.offsets[e];
      if (start < 0 || end < start || (int64_t)end > a.rows) flags[3] = 1;
      seg_rec[e].y = start;
      seg_rec[e].z = end;
    }
    if (tid < kConsumerWarps) seg_hint[tid] = 0;
    __syncthreads();
    if (warp == 0) {
      int32_t slab_base = 0;
      for (int c0 = 0; c0 < E; c0 += 32) {
        const int e = c0 + lane;
        const int32_t n = (e < E && !flags[3]) ? seg_rec[e].z - seg_rec[e].y : 0;
        const int32_t p0 = (n + 15) / 16;  // the segment's slabs (its rows padded to 16)
        int32_t p = p0;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
          const int32_t pu = __shfl_up_sync(0xFFFFFFFFu, p, d);
          if (lane >= d) p += pu;
        }
        if (e < E) seg_rec[e].x = slab_base + p - p0;
        slab_base += __shfl_sync(0xFFFFFFFFu, p, 31);
      }
      if (lane == 0) {
        seg_rec[E] = make_int4(slab_base, (int32_t)a.rows, (int32_t)a.rows, 0x7FFFFFFF);
        if (COL && (int64_t)slab_base * 16 > a.col_ld) flags[3] = 1;
      }
    }
    __syncthreads();
    if (flags[3]) {
      if (blockIdx.x == 0 && tid == 0) atomicOr(a.status, 1u);  // NVFP4_DEVICE_BAD_OFFSETS
      return;
    }
    for (int e = tid; e < E; e += blockDim.x) seg_rec[e].w = seg_rec[e + 1].x;
    n_slabs = seg_rec[E].x;
    __syncthreads();
    total = ((n_slabs + kWarpsPerGroup - 1) / kWarpsPerGroup) * tiles_n;
    n_local = (int)blockIdx.x < total ? (total - (int)blockIdx.x + stride - 1) / stride : 0;
    if (tid == 0) first_loads();
    __syncthreads();
  }

  // amax pass: per-segment maxima (16-bit magnitudes) in the otherwise unused staging area
  uint32_t* seg_amax = reinterpret_cast<uint32_t*>(smem + kSmemColCodes);  // [2][kMaxSegments]
  if (AMAX_ONLY) {
    for (int e = tid; e < 2 * kMaxSegments; e += blockDim.x) seg_amax[e] = 0u;
    __syncthreads();
  }
  const int g = warp / kWarpsPerGroup;   // group
  const int rb = warp % kWarpsPerGroup;  // slab of the tile (rows 16 rb .. 16 rb + 15)
  const int gt = tid - g * 32 * kWarpsPerGroup;  // thread index inside the group

  // ---- single-launch amax: rounds of amax slots, first this CTA's own rank, then any rank it
  // takes over while waiting; fold the maxima into the workspace, count the rank as arrived,
  // wait for every rank (fused_amax.cuh) ----
  float* fused_amax = reinterpret_cast<float*>(smem + kSmemFused) + 32;  // [0] row, [1] col
  int n_slots = n_local;  // amax slots of every round (the quantize phase walks them back)
  uint32_t done_before = 0u;  // thread 0: the CTAs done with the workspace before this one
  if (fused) {
    // claim the own rank (the result is needed only at the first arrival)
    uint32_t own_before = 0u;
    if (tid == 0) own_before = fuse_claim(a.fuse_ws, blockIdx.x);
    uint32_t m = 0u, mt = 0u;
    bool ok = true;
    int first = 0, round_end = n_local;
    uint64_t t_wait = 0u;
    volatile uint32_t* red = reinterpret_cast<volatile uint32_t*>(smem + kSmemFused);
    while (true) {
      for (int k = first + (g - first % kGroups + kGroups) % kGroups; k < round_end; k += kGroups) {
        const int s = k % kStages, p = k / kStages;  // load p of stage s
        bool arrived = wait_issued(issued, s, p + 1);
        arrived = arrived && mbar_wait_bounded(&full[s], (uint32_t)p & 1u, kWaitLimitNs);
        if (!arrived || coords[s].tile != tile_of_slot(k)) ok = false;
        // rows and columns outside the tensor arrive as zeros: no masking for a maximum
        uint4 v[16];
        const uint32_t src = smem_u32(smem + kSmemStages + s * kStageBytes) +
                             (16 * rb) * (kTileN * 2) + lane * 16;
#pragma unroll
        for (int r = 0; r < 16; r++) v[r] = lds128(src + r * (kTileN * 2));
        named_bar_sync(1 + g, 32 * kWarpsPerGroup);
        if (gt == 0 && k + kStages < round_end) {
          fence_proxy_async();
          issue(tile_of_slot(k + kStages), s);
        }
        // max.xorsign.abs: the magnitude is exact, the sign bit is cleared at the end (inputs
        // are finite, so no NaN takes part)
#pragma unroll
        for (int r = 0; r < 16; r += 2)
          m = hmax_abs2(m, hmax_abs2(hmax_abs2(hmax_abs2(v[r].x, v[r].y), hmax_abs2(v[r].z, v[r].w)),
                                     hmax_abs2(hmax_abs2(v[r + 1].x, v[r + 1].y),
                                               hmax_abs2(v[r + 1].z, v[r + 1].w))));
        if (COL && RHT) {
#pragma unroll
          for (int c4 = 0; c4 < 4; c4++) {
            uint32_t w[16];
#pragma unroll
            for (int r = 0; r < 16; r++) w[r] = comp(v[r], c4);
            mt = vmax2(mt, rht16_pair_absmax(w, a.rht_flip));  // both sign-cleared
          }
        }
      }
      m &= 0x7FFF7FFFu;
      // the CTA's maxima over every round so far (cta_max's barriers also end the round: every
      // group has read its last slot)
      const uint32_t mr = cta_max(max(m & 0xFFFFu, m >> 16), red);
      const uint32_t mc = (COL && RHT) ? cta_max(max(mt & 0xFFFFu, mt >> 16), red) : mr;
      if (tid == 0) {
        // the first round is the own rank: it counts only if the claim at the start won it
        // (otherwise another CTA took it over and counts it)
        const bool own_taken = ((own_before >> (blockIdx.x & 31)) & 1u) != 0u;
        fuse_arrive(a.fuse_ws, mr, mc, (first == 0 && own_taken) ? 0u : 1u);
        if (first == 0) t_wait = global_ns();
        uint32_t pr = 0u, pc = 0u;
        int r = -1;
        const FuseWait w = fuse_wait(a.fuse_ws, (uint32_t)(stride + a.fuse_extra), stride, t_wait,
                                     fctl[0] < kMaxHeld, pr, pc, r);
        fctl[1] = w;
        if (w == kFuseSteal) {
          // take rank r over: its amax round follows in the ring (every stage is free: the
          // round's last slots were read before cta_max's barriers)
          const int h = fctl[0];
          held_rank[h] = r;
          held_first[h] = round_end;
          fctl[0] = h + 1;
          fctl[2] = r;
          fence_proxy_async();
          for (int k = round_end; k < round_end + kStages && k < round_end + rank_tiles(r); k++)
            issue(tile_of_slot(k), k % kStages);
        } else {
          if (w == kFuseTimedOut) {
            flags[3] = 1;
            atomicOr(a.status, 2u);  // NVFP4_DEVICE_TIMEOUT
          }
          done_before = fuse_done(a.fuse_ws);
          // past the wait this CTA no longer uses the workspace: the next kernel in the stream
          // may start on the SMs that finished CTAs leave
          pdl_allow_next();
          fused_amax[0] = __uint_as_float(pr << 16);
          fused_amax[1] = __uint_as_float(pc << 16);
        }
      }
      __syncthreads();
      if (fctl[1] != kFuseSteal) break;
      first = round_end;
      round_end += rank_tiles(fctl[2]);
    }
    n_slots = round_end;
    if (!ok) {
      flags[3] = 1;  // this CTA stores nothing (below); the others still need its maxima
      if (lane == 0) atomicOr(a.status, 2u);  // NVFP4_DEVICE_TIMEOUT
    }
    __syncthreads();
    if (flags[3]) flags[0] = flags[1] = flags[2] = 1;  // every group leaves without storing
  }
  // amax of segment e (rowwise / columnwise side)
  auto amax_row_of = [&](int e) -> float {
    return FUSED ? fused_amax[0] : a.amax_row[(int64_t)e * a.amax_row_stride];
  };
  auto amax_col_of = [&](int e) -> float {
    return FUSED ? fused_amax[1] : a.amax_col[(int64_t)e * a.amax_col_stride];
  };
  if (blockIdx.x == 0 && !AMAX_ONLY) {  // global scales {amax, S_dec} of every segment
    for (int e = tid; e < E; e += blockDim.x) {
      float enc, dec;
      if (ROW || TWO_D) {
        const float amax = amax_row_of(e);
        global_scale(amax, enc, dec);
        if (ROW) { a.row_gscale[2 * e] = amax; a.row_gscale[2 * e + 1] = dec; }
        if (TWO_D && COL) { a.col_gscale[2 * e] = amax; a.col_gscale[2 * e + 1] = dec; }
      }
      if (COL && !TWO_D) {
        const float amax = amax_col_of(e);
        global_scale(amax, enc, dec);
        a.col_gscale[2 * e] = amax;
        a.col_gscale[2 * e + 1] = dec;
      }
    }
  }

  // Every segment's encode and decode scales, once per CTA (the single-launch amax computes its
  // one segment's where the maxima are known, in set_segment)
  if (!FUSED && !AMAX_ONLY) {
    for (int e = tid; e < E; e += blockDim.x) {
      float4 q = make_float4(1.0f, 1.0f, 1.0f, 1.0f);
      if (ROW || TWO_D) global_scale(amax_row_of(e), q.x, q.y);
      if (COL && !TWO_D) global_scale(amax_col_of(e), q.z, q.w);
      if (TWO_D) { q.z = q.x; q.w = q.y; }
      seg_scale[e] = q;
    }
    __syncthreads();
  }

  // =========================================================================================
  // Groups of four warps, one tile at a time.
  // =========================================================================================
  const bool odd = (lane & 1) != 0;
  const int kb = lane >> 1;              // rowwise block of the tile row (lane pair)
  // the group's scale block (kTableBlock): tables [2][128], then {S_enc row, S_enc col}
  float* tab_row = reinterpret_cast<float*>(smem + kSmemTables + g * kTableBlock);
  float* tab_col = tab_row + kTableEntries;
  // columnwise staging, two buffers per group: a tile's codes and scales are staged in one
  // while the previous tile's leave from the other
  uint8_t* cc_base = smem + kSmemColCodes + g * kColStageBufs * kColCodeStage;
  uint8_t* cs_base = smem + kSmemColScales + g * kColStageBufs * kColScaleStage;
  const int64_t row_nb = N / 16;
  const int64_t col_nb = a.col_ld / 16;
  int cur_seg = -1;
  // Encode scales of segment e and the decode scales its reciprocal tables are built from.
  auto seg_scales = [&](int e, float& enc_r, float& dec_r, float& enc_c, float& dec_c) {
    if (FUSED) {
      enc_r = enc_c = dec_r = dec_c = 1.0f;
      if (ROW || TWO_D) global_scale(amax_row_of(e), enc_r, dec_r);
      if (COL && !TWO_D) global_scale(amax_col_of(e), enc_c, dec_c);
      if (TWO_D) { enc_c = enc_r; dec_c = dec_r; }
    } else {
      const float4 q = seg_scale[e];
      enc_r = q.x; dec_r = q.y; enc_c = q.z; dec_c = q.w;
    }
  };
  auto multiplier = [&](int code, float dec) -> float {
    const float sv = e4m3x2_to_float2((uint16_t)code).x;
    return a.fast ? element_multiplier_fast(sv, dec) : element_multiplier(sv, dec);
  };
  // Global scales of segment e and the group's reciprocal tables for them: one entry of each
  // table per thread of the group. Called by the whole group, between tiles (no warp of the
  // group is still reading the previous tables).
  auto set_segment = [&](int e) {
    float enc_r, dec_r, enc_c, dec_c;
    seg_scales(e, enc_r, dec_r, enc_c, dec_c);
    static_assert(kTableEntries == 32 * kWarpsPerGroup, "one table entry per group thread");
    tab_row[gt] = multiplier(gt, dec_r);
    tab_col[gt] = multiplier(gt, dec_c);
    if (gt == 0) { tab_row[2 * kTableEntries] = enc_r; tab_row[2 * kTableEntries + 1] = enc_c; }
    named_bar_sync(1 + g, 32 * kWarpsPerGroup);
    cur_seg = e;
  };
  // A grouped tile's slabs can belong to several segments; the group's scale block is its
  // first slab's, and a warp whose slab lies in another segment builds a block of its own.
  float* tab_warp = reinterpret_cast<float*>(smem + kSmemWarpTables + warp * kTableBlock);
  // Write-out of a tile's staged columnwise codes and scales by the whole group. Whole tiles'
  // codes leave by one TMA store (issued by thread 0 of the group); otherwise thread gt owns
  // the column pair 2 gt, 2 gt + 1 and a column's codes leave as one 32-byte store (or as its
  // slabs' 8-byte pieces). The scales always leave from the threads.
  auto write_out = [&](const OutPos& wc, const uint8_t* ccs, const uint8_t* css) {
    const int nrb = wc.nvalid;
    const bool whole = nrb == kWarpsPerGroup;  // all four slabs hold rows
    if (a.col_tma && whole) {
      if (gt == 0) {
        tma_store_3d(&a.tmap_colc, ccs, wc.colpos / 2, wc.n0 / 8, 0);
        bulk_commit();
      }
    }
    const int64_t col0 = (int64_t)wc.n0 + 2 * gt;   // this thread's column pair
    if (col0 < N) {
      if (!(a.col_tma && whole)) {
        const int l = gt >> 2, z0 = (2 * gt) & 7;   // lane of origin, columns z0 and z0 + 1
        const uint8_t* p0 = ccs + z0 * 1024 + l * 32;
        const uint8_t* p1 = p0 + 1024;
        const int sw = ((l >> 2) & 1) << 4;  // the 32-byte swizzle of this y
        uint4 c0a = *reinterpret_cast<const uint4*>(p0 + sw), c0b = *reinterpret_cast<const uint4*>(p0 + (16 ^ sw));
        uint4 c1a = *reinterpret_cast<const uint4*>(p1 + sw), c1b = *reinterpret_cast<const uint4*>(p1 + (16 ^ sw));
        // c?a: slabs 0, 1; c?b: slabs 2, 3
        uint8_t* dst0 = a.col_codes + col0 * (a.col_ld / 2) + wc.colpos / 2;
        uint8_t* dst1 = dst0 + a.col_ld / 2;
        const uintptr_t dbits = reinterpret_cast<uintptr_t>(dst0) | reinterpret_cast<uintptr_t>(dst1);
        if (whole && (dbits & 31) == 0) {
          stg256(dst0, c0a, c0b);
          stg256(dst1, c1a, c1b);
        } else if (whole && (dbits & 15) == 0) {
          reinterpret_cast<uint4*>(dst0)[0] = c0a;
          reinterpret_cast<uint4*>(dst0)[1] = c0b;
          reinterpret_cast<uint4*>(dst1)[0] = c1a;
          reinterpret_cast<uint4*>(dst1)[1] = c1b;
        } else {
          const uint2 q0[4] = {make_uint2(c0a.x, c0a.y), make_uint2(c0a.z, c0a.w), make_uint2(c0b.x, c0b.y), make_uint2(c0b.z, c0b.w)};
          const uint2 q1[4] = {make_uint2(c1a.x, c1a.y), make_uint2(c1a.z, c1a.w), make_uint2(c1b.x, c1b.y), make_uint2(c1b.z, c1b.w)};
#pragma unroll
          for (int r = 0; r < kWarpsPerGroup; r++) {
            if (r < nrb) {
              *reinterpret_cast<uint2*>(dst0 + 8 * r) = q0[r];
              *reinterpret_cast<uint2*>(dst1 + 8 * r) = q1[r];
            }
          }
        }
      }
      uint32_t sc0 = 0, sc1 = 0;
#pragma unroll
      for (int r = 0; r < kWarpsPerGroup; r++) {
        if (r < nrb) {
          const uint32_t pr = *reinterpret_cast<const uint16_t*>(css + r * kTileN + 2 * gt);
          sc0 |= (pr & 0xFFu) << (8 * r);
          sc1 |= (pr >> 8) << (8 * r);
        }
      }
      if (!SWZ) {
        uint8_t* sd0 = a.col_scales + col0 * col_nb + wc.colpos / 16;
        uint8_t* sd1 = sd0 + col_nb;
        if (whole && ((reinterpret_cast<uintptr_t>(sd0) | reinterpret_cast<uintptr_t>(sd1)) & 3) == 0) {
          *reinterpret_cast<uint32_t*>(sd0) = sc0;
          *reinterpret_cast<uint32_t*>(sd1) = sc1;
        } else {
          for (int r = 0; r < nrb; r++) {
            sd0[r] = (uint8_t)(sc0 >> (8 * r));
            sd1[r] = (uint8_t)(sc1 >> (8 * r));
          }
        }
      } else if (!whole) {  // the tiled layout, a partial tile: byte by byte
        for (int r = 0; r < nrb; r++) {
          a.col_scales[swz_scale_off(col0, wc.colpos / 16 + r, a.col_swz_tc)] = (uint8_t)(sc0 >> (8 * r));
          if (col0 + 1 < N)
            a.col_scales[swz_scale_off(col0 + 1, wc.colpos / 16 + r, a.col_swz_tc)] = (uint8_t)(sc1 >> (8 * r));
        }
      }
    }
    // The tiled layout, a whole tile: its 256 columns x 4 scales (colpos / 16 is a multiple of
    // four, n0 of 256) are two whole 128 x 4 tiles of 512 contiguous bytes; thread gt < 64
    // writes the 16 bytes of row q = gt % 32 of tile half gt / 32 (columns 32 i + q, i = 0..3).
    if (SWZ && whole && gt < 64) {
      const int h = gt >> 5, q = gt & 31;
      uint32_t w[4];
#pragma unroll
      for (int i = 0; i < 4; i++) {
        const int cc = 128 * h + 32 * i + q;
        w[i] = (uint32_t)css[cc] | ((uint32_t)css[kTileN + cc] << 8) |
               ((uint32_t)css[2 * kTileN + cc] << 16) | ((uint32_t)css[3 * kTileN + cc] << 24);
      }
      const int64_t row = (int64_t)wc.n0 + 128 * h;
      uint8_t* dst = a.col_scales + swz_scale_off(row, wc.colpos / 16, a.col_swz_tc) + 16 * q;
      if (row + 128 <= N) {
        *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
      } else {
#pragma unroll
        for (int i = 0; i < 4; i++)
          if (row + 32 * i + q < N) *reinterpret_cast<uint32_t*>(dst + 4 * i) = w[i];
      }
    }
  };
  OutPos prev{};          // the group's previous tile, staged in buffer buf ^ 1
  bool have_prev = false;
  int buf = 0;

  // Quantize position i: the tile of local index i; after the single-launch amax, the tile of
  // amax slot n_slots - 1 - i (the amax rounds walked back, so that the first kStages
  // positions are the tiles still in the stages).
  auto position_tile = [&](int i) -> int {
    return fused ? tile_of_slot(n_slots - 1 - i) : (int)blockIdx.x + i * stride;
  };
  if (!AMAX_ONLY && plain && n_slots > g) set_segment(0);  // overlaps the first loads (or follows the amax)

  for (int i = g; i < n_slots; i += kGroups) {
    const int tile = position_tile(i);
    // Stage and load number of position i. Plain: stage i % kStages, its load i / kStages.
    // After the single-launch amax phase (a_s loads into stage s, slot k in stage k % kStages)
    // the first kStages positions are still in the stages; position i >= kStages goes where
    // position i - kStages was.
    int s, p;
    bool resident = false;
    if (fused) {
      s = (n_slots - 1 - i) % kStages;
      const int a_s = n_slots > s ? (n_slots - 1 - s) / kStages + 1 : 0;
      p = a_s + i / kStages - 1;
      resident = i < kStages;
    } else {
      s = i % kStages;
      p = i / kStages;
    }
    // Three groups share four stages, so a group can reach tile i before the group that
    // drains the stage's previous tile has issued it. Wait until the load is issued; only
    // then does the phase parity name its phase unambiguously.
    bool arrived = resident || wait_issued(issued, s, p + 1);
    arrived = arrived && (resident || mbar_wait_bounded(&full[s], (uint32_t)p & 1u, kWaitLimitNs));
    // this warp's slab and what the group needs of the tile, read before the stage is refilled
    const Coord& cs = coords[s];
    const OutPos c = {cs.n0, cs.colpos, cs.nvalid};
    const int slab_rows = cs.nrows[rb];
    const int64_t row_g0 = cs.row0[rb];
    const int seg_w = cs.seg[rb], seg_g = cs.seg[0];
    // a slab of another segment than the tile's first: this warp's own scale block, built
    // before the tile's data take up registers (the warp is done with its previous block)
    const bool foreign =
        GROUPED && !AMAX_ONLY && arrived && cs.tile == tile && seg_w != seg_g && slab_rows > 0;
    if (foreign) build_scale_block(tab_warp, seg_scale[seg_w], lane, a.fast);
    const float* trow = foreign ? tab_warp : tab_row;  // the slab's scale block
    if (!arrived || cs.tile != tile) {
      // the data never arrived (or the stage holds another tile): record it; the loads below
      // read stale shared memory and the group leaves at its next barrier without storing
      flags[g] = 1;
      if (lane == 0) atomicOr(a.status, 2u);  // NVFP4_DEVICE_TIMEOUT
    }
    uint4 v[16];
    if (slab_rows > 0) {
      const uint32_t src = smem_u32(smem + kSmemStages + s * kStageBytes) +
                           (16 * rb) * (kTileN * 2) + lane * 16;
#pragma unroll
      for (int r = 0; r < 16; r++) v[r] = lds128(src + r * (kTileN * 2));
      if (slab_rows < 16) {  // rows past the segment's end are zero padding
#pragma unroll
        for (int r = 0; r < 16; r++)
          if (r >= slab_rows) v[r] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    // All four slabs are in registers: the stage can be refilled, the previous tile's staging
    // is complete (every warp staged it before arriving here), the buffer before it was
    // written out, and the group's abort flag is settled.
    if (COL && !AMAX_ONLY) {
      fence_proxy_async();             // this thread's staging, for the TMA store
      if (gt == 0) bulk_wait_read();   // the store that read the buffer about to be staged
    }
    named_bar_sync(1 + g, 32 * kWarpsPerGroup);
    if (flags[g]) break;
    if (GROUPED) {  // each warp loads its own slab of the stage's next tile
      if (lane == 0 && i + kStages < n_slots) {
        fence_proxy_async();
        issue_slab(position_tile(i + kStages), s, rb);
      }
    } else if (gt == 0 && i + kStages < n_slots) {
      fence_proxy_async();
      issue(position_tile(i + kStages), s);
    }

    if constexpr (AMAX_ONLY) {
      if (slab_rows > 0) {  // rows past the segment's end are zero (above)
        uint32_t t[16];
#pragma unroll
        for (int r = 0; r < 16; r++)
          t[r] = hmax_abs2(hmax_abs2(v[r].x, v[r].y), hmax_abs2(v[r].z, v[r].w));
#pragma unroll
        for (int h = 8; h >= 1; h >>= 1)
#pragma unroll
          for (int r = 0; r < h; r++) t[r] = hmax_abs2(t[r], t[r + h]);
        const uint32_t m = t[0] & 0x7FFF7FFFu;
        uint32_t mr = max(m & 0xFFFFu, m >> 16), mc = mr;
        if (RHT) {
          uint32_t mt = 0u;
#pragma unroll
          for (int k = 0; k < 4; k++) {
            uint32_t w[16];
#pragma unroll
            for (int r = 0; r < 16; r++) w[r] = comp(v[r], k);
            mt = vmax2(mt, rht16_pair_absmax(w, a.rht_flip));
          }
          mc = max(mt & 0xFFFFu, mt >> 16);
        }
        mr = __reduce_max_sync(0xFFFFFFFFu, mr);
        mc = __reduce_max_sync(0xFFFFFFFFu, mc);
        if (lane == 0) {
          atomicMax(&seg_amax[seg_w], mr);
          atomicMax(&seg_amax[kMaxSegments + seg_w], mc);
        }
      }
      continue;
    }

    if (COL && have_prev)
      write_out(prev, cc_base + (buf ^ 1) * kColCodeStage, cs_base + (buf ^ 1) * kColScaleStage);
    uint8_t* cc_stage = cc_base + buf * kColCodeStage;
    uint8_t* cs_stage = cs_base + buf * kColScaleStage;
    if (seg_g != cur_seg) set_segment(seg_g);  // uniform across the group
    const float* tcol = trow + kTableEntries;

    const bool lane_cols = (int64_t)c.n0 + lane * 8 < N;  // all 8 of the lane's columns exist
    // every row of the slab and every column of the tile exist (uniform across the warp)
    const bool full_slab = slab_rows == 16 && (int64_t)c.n0 + kTileN <= N;
    if (slab_rows > 0) {
      // ---------------- 2D: one scale per 16x16 tile (the lane pair's 16 columns) ----------------
      float tile_r = 0.0f;
      uint32_t tile_s = 0u;
      if (TWO_D) {
        uint32_t cm[4];
#pragma unroll
        for (int k = 0; k < 4; k++) {
          uint32_t w[16];
#pragma unroll
          for (int r = 0; r < 16; r++) w[r] = comp(v[r], k);
          cm[k] = tree_max16(w);
        }
        const uint32_t m = vmax2(vmax2(cm[0], cm[1]), vmax2(cm[2], cm[3]));
        uint32_t tm = max(m & 0xFFFFu, m >> 16);
        tm = max(tm, __shfl_xor_sync(0xFFFFFFFFu, tm, 1));
        tile_s = block_scales2(__uint_as_float(tm << 16), 0.0f, trow[2 * kTableEntries]) & 0xFFu;
        tile_r = trow[tile_s];
      }

      uint32_t tcode[kRowCol2D ? 16 : 1];  // 2D row+col: the slab's row codes, then transposed
      // ---------------- rowwise: 1x16 blocks, a lane pair per block ----------------
      if (ROW) {
        // Rows 4q, 4q+1 belong to the even lane of the pair, 4q+2, 4q+3 to the odd lane: the
        // owner computes their scales (and Philox draws) and shares the multipliers.
        float rr[16];
        uint32_t own_s[4];
        if (TWO_D) {
#pragma unroll
          for (int r = 0; r < 16; r++) rr[r] = tile_r;
#pragma unroll
          for (int q = 0; q < 4; q++) own_s[q] = tile_s | (tile_s << 8);
        } else {
          uint32_t P[8];
#pragma unroll
          for (int j = 0; j < 8; j++) P[j] = row_pair_max(v[2 * j], v[2 * j + 1]);
          uint32_t recv[4];
#pragma unroll
          for (int q = 0; q < 4; q++)
            recv[q] = __shfl_xor_sync(0xFFFFFFFFu, odd ? P[2 * q] : P[2 * q + 1], 1);
          float r_own[8];
          const float enc_r = trow[2 * kTableEntries];
#pragma unroll
          for (int q = 0; q < 4; q++) {
            const uint32_t bm = vmax2(odd ? P[2 * q + 1] : P[2 * q], recv[q]);
            own_s[q] = block_scales2(mag_lo(bm), mag_hi(bm), enc_r);
            r_own[2 * q] = trow[own_s[q] & 0xFFu];
            r_own[2 * q + 1] = trow[own_s[q] >> 8];
          }
#pragma unroll
          for (int q = 0; q < 4; q++) {
            const float o0 = __shfl_xor_sync(0xFFFFFFFFu, r_own[2 * q], 1);
            const float o1 = __shfl_xor_sync(0xFFFFFFFFu, r_own[2 * q + 1], 1);
            rr[4 * q] = odd ? o0 : r_own[2 * q];
            rr[4 * q + 1] = odd ? o1 : r_own[2 * q + 1];
            rr[4 * q + 2] = odd ? r_own[2 * q] : o0;
            rr[4 * q + 3] = odd ? r_own[2 * q + 1] : o1;
          }
        }
        uint32_t wr[16][2];  // random words of the lane's half of each row block
        if (SR_ROW) {
#pragma unroll
          for (int q = 0; q < 4; q++) {
            const uint64_t b0 = (uint64_t)(row_g0 + 4 * q + (odd ? 2 : 0)) * (uint64_t)row_nb +
                                (uint64_t)(c.n0 / 16 + kb);
            const uint4 D0 = block_random_rk(a.philox_key, a.rng_offset, 0u, b0);
            const uint4 D1 = block_random_rk(a.philox_key, a.rng_offset, 0u, b0 + (uint64_t)row_nb);
            const uint32_t x0 = __shfl_xor_sync(0xFFFFFFFFu, odd ? D0.x : D0.z, 1);
            const uint32_t x1 = __shfl_xor_sync(0xFFFFFFFFu, odd ? D0.y : D0.w, 1);
            const uint32_t x2 = __shfl_xor_sync(0xFFFFFFFFu, odd ? D1.x : D1.z, 1);
            const uint32_t x3 = __shfl_xor_sync(0xFFFFFFFFu, odd ? D1.y : D1.w, 1);
            wr[4 * q][0] = odd ? x0 : D0.x;      wr[4 * q][1] = odd ? x1 : D0.y;
            wr[4 * q + 1][0] = odd ? x2 : D1.x;  wr[4 * q + 1][1] = odd ? x3 : D1.y;
            wr[4 * q + 2][0] = odd ? D0.z : x0;  wr[4 * q + 2][1] = odd ? D0.w : x1;
            wr[4 * q + 3][0] = odd ? D1.z : x2;  wr[4 * q + 3][1] = odd ? D1.w : x3;
          }
        }
        auto row_code = [&](int r) -> uint32_t {
          const uint64_t rr2 = f2_pack(rr[r], rr[r]);
          const float2 t0 = f2_unpack(f2_mul(f2_from_bf16x2(v[r].x), rr2));
          const float2 t1 = f2_unpack(f2_mul(f2_from_bf16x2(v[r].y), rr2));
          const float2 t2 = f2_unpack(f2_mul(f2_from_bf16x2(v[r].z), rr2));
          const float2 t3 = f2_unpack(f2_mul(f2_from_bf16x2(v[r].w), rr2));
          return e2m1x8<SR_ROW>(t0.x, t0.y, t1.x, t1.y, t2.x, t2.y, t3.x, t3.y,
                                SR_ROW ? wr[r][0] : 0u, SR_ROW ? wr[r][1] : 0u);
        };
        uint8_t* rowp = a.row_codes + row_g0 * (N / 2) + c.n0 / 2 + lane * 4;
        // the lane's scale bytes: rows row_g0 + 4q (+ 2 on the odd lane) and the next, column
        // c.n0 / 16 + kb, row-major or in the tiled layout (rows 16 bytes apart there: no row
        // of the slab crosses a 32-row boundary)
        const int64_t rcol = c.n0 / 16 + kb, rrow = row_g0 + (odd ? 2 : 0);
        uint8_t* rsp = a.row_scales + (SWZ ? swz_scale_off(rrow, rcol, a.row_swz_tc)
                                           : rrow * row_nb + rcol);
        const int64_t rstride = SWZ ? 16 : row_nb;
        if (kRowCol2D) {
          // 2D: the columnwise codes are these codes transposed (one multiplier per 16x16
          // tile, the same in both orientations), so keep all 16 rows
#pragma unroll
          for (int r = 0; r < 16; r++) tcode[r] = row_code(r);
        }
        if (full_slab) {
#pragma unroll
          for (int r = 0; r < 16; r++)
            *reinterpret_cast<uint32_t*>(rowp + (int64_t)r * (N / 2)) = kRowCol2D ? tcode[r] : row_code(r);
#pragma unroll
          for (int q = 0; q < 4; q++) {
            rsp[(int64_t)(4 * q) * rstride] = (uint8_t)(own_s[q] & 0xFFu);
            rsp[(int64_t)(4 * q + 1) * rstride] = (uint8_t)(own_s[q] >> 8);
          }
        } else if (lane_cols) {
#pragma unroll
          for (int r = 0; r < 16; r++)
            if (r < slab_rows)
              *reinterpret_cast<uint32_t*>(rowp + (int64_t)r * (N / 2)) = kRowCol2D ? tcode[r] : row_code(r);
#pragma unroll
          for (int q = 0; q < 4; q++) {
            const int r0 = 4 * q + (odd ? 2 : 0);
            if (r0 < slab_rows) rsp[(int64_t)(4 * q) * rstride] = (uint8_t)(own_s[q] & 0xFFu);
            if (r0 + 1 < slab_rows) rsp[(int64_t)(4 * q + 1) * rstride] = (uint8_t)(own_s[q] >> 8);
          }
        }
      }

      // ---------------- columnwise: one lane-local block per column, two columns at a time --------
      if (COL && kRowCol2D) {
        // rows 0..7 and 8..15 of the lane's 8 columns: two 8 x 8 nibble transposes
        transpose_nibbles8(tcode);
        transpose_nibbles8(tcode + 8);
#pragma unroll
        for (int k = 0; k < 4; k++) {
          *reinterpret_cast<uint2*>(cc_stage + col_stage_off(lane, 2 * k, rb)) =
              make_uint2(tcode[2 * k], tcode[8 + 2 * k]);
          *reinterpret_cast<uint2*>(cc_stage + col_stage_off(lane, 2 * k + 1, rb)) =
              make_uint2(tcode[2 * k + 1], tcode[8 + 2 * k + 1]);
        }
        const uint32_t s4 = tile_s * 0x01010101u;  // the tile scale for all four column pairs
        *reinterpret_cast<uint2*>(cs_stage + rb * kTileN + lane * 8) = make_uint2(s4, s4);
      }
      if (COL && !kRowCol2D) {
        uint32_t csc[2] = {0u, 0u};
#pragma unroll
        for (int k = 0; k < 4; k++) {
          uint32_t w[16];
#pragma unroll
          for (int r = 0; r < 16; r++) w[r] = comp(v[r], k);
          uint64_t xs[16];  // fast math: the FP32 transform, not rounded (unused otherwise)
          if (FAST_RHT) rht16_pair_f32(w, a.rht_flip, xs);
          else if (RHT) rht16_pair(w, a.rht_flip);
          uint32_t s2;
          uint64_t rc2;
          if (FAST_RHT) {
            float m0 = 0.0f, m1 = 0.0f;
#pragma unroll
            for (int r = 0; r < 16; r++) {
              const float2 y = f2_unpack(xs[r]);
              m0 = fmaxf(m0, fabsf(y.x));
              m1 = fmaxf(m1, fabsf(y.y));
            }
            s2 = block_scales2(m0, m1, trow[2 * kTableEntries + 1]);
            rc2 = f2_pack(tcol[s2 & 0xFFu], tcol[s2 >> 8]);
          } else if (TWO_D) {
            s2 = tile_s | (tile_s << 8);
            rc2 = f2_pack(tile_r, tile_r);
          } else {
            const uint32_t m = tree_max16(w);
            s2 = block_scales2(mag_lo(m), mag_hi(m), trow[2 * kTableEntries + 1]);
            rc2 = f2_pack(tcol[s2 & 0xFFu], tcol[s2 >> 8]);
          }
          csc[k >> 1] |= s2 << (16 * (k & 1));
          uint4 W0 = make_uint4(0u, 0u, 0u, 0u), W1 = W0;
          if (SR_COL) {
            const uint64_t b0 = (uint64_t)(c.n0 + lane * 8 + 2 * k) * (uint64_t)col_nb +
                                (uint64_t)(c.colpos / 16 + rb);
            W0 = block_random_rk(a.philox_key, a.rng_offset, 1u, b0);
            W1 = block_random_rk(a.philox_key, a.rng_offset, 1u, b0 + (uint64_t)col_nb);
          }
          uint32_t code[2][2];  // [column of the pair][rows 0..7, 8..15]
#pragma unroll
          for (int o = 0; o < 2; o++) {
            float2 t[8];
#pragma unroll
            for (int r = 0; r < 8; r++)
              t[r] = f2_unpack(
                  f2_mul(FAST_RHT ? xs[8 * o + r] : f2_from_bf16x2(w[8 * o + r]), rc2));
            code[0][o] = e2m1x8<SR_COL>(t[0].x, t[1].x, t[2].x, t[3].x, t[4].x, t[5].x, t[6].x,
                                        t[7].x, comp(W0, 2 * o), comp(W0, 2 * o + 1));
            code[1][o] = e2m1x8<SR_COL>(t[0].y, t[1].y, t[2].y, t[3].y, t[4].y, t[5].y, t[6].y,
                                        t[7].y, comp(W1, 2 * o), comp(W1, 2 * o + 1));
          }
          *reinterpret_cast<uint2*>(cc_stage + col_stage_off(lane, 2 * k, rb)) =
              make_uint2(code[0][0], code[0][1]);
          *reinterpret_cast<uint2*>(cc_stage + col_stage_off(lane, 2 * k + 1, rb)) =
              make_uint2(code[1][0], code[1][1]);
        }
        *reinterpret_cast<uint2*>(cs_stage + rb * kTileN + lane * 8) = make_uint2(csc[0], csc[1]);
      }
    }

    prev = c;
    have_prev = true;
    buf ^= 1;
  }
  if (COL && !AMAX_ONLY && have_prev && !flags[g]) {
    fence_proxy_async();
    named_bar_sync(1 + g, 32 * kWarpsPerGroup);
    write_out(prev, cc_base + (buf ^ 1) * kColCodeStage, cs_base + (buf ^ 1) * kColScaleStage);
  }
  if (COL && !AMAX_ONLY && gt == 0) bulk_wait_all();  // the last store has left shared memory

  // Every load issued into a stage is waited for by the group that owns its tile, unless that
  // group gave up: let the last load of each stage land before the CTA leaves.
  __syncthreads();
  if (AMAX_ONLY) {  // this CTA's maxima into the per-segment results
    for (int e = tid; e < E; e += blockDim.x) {
      const uint32_t mr = seg_amax[e], mc = seg_amax[kMaxSegments + e];
      if (a.amax_row && mr)
        atomicMax(reinterpret_cast<unsigned int*>(const_cast<float*>(a.amax_row) + (int64_t)e * a.amax_row_stride), mr << 16);
      if (a.amax_col && mc)
        atomicMax(reinterpret_cast<unsigned int*>(const_cast<float*>(a.amax_col) + (int64_t)e * a.amax_col_stride), mc << 16);
    }
  }
  if (tid == 0) {
    for (int s = 0; s < kStages; s++) {
      const int loads = issued[s];
      if (loads > 0) mbar_wait_bounded(&full[s], (uint32_t)(loads - 1) & 1u, kWaitLimitNs);
    }
    if (fused) fuse_reset_if_last(a.fuse_ws, done_before, stride);
  }
}

// One variant: SWZ writes both scale outputs in the GEMMs' tiled layout (a.swz_scales).
template <bool ROW, bool COL, bool RHT, bool TWO_D, bool SR_ROW, bool SR_COL, bool FAST_RHT, bool SWZ>
cudaError_t launch_variant(const QuantArgs& args, int grid, cudaStream_t s) {
  if (args.offsets != nullptr) {  // grouped (the host rejects the single launch and SWZ there)
    return launch_pdl(quantize_tiles_kernel<ROW, COL, RHT, TWO_D, SR_ROW, SR_COL, false, false, FAST_RHT, false, true>,
                      dim3(grid), dim3(kQuantThreads), kQuantSmemBytes, s, args);
  }
  if (args.fused) {
    // No CTA waits for another to start (fused_amax.cuh), so the CTAs need not be resident at
    // once: a plain launch with programmatic dependent launch, whose CTAs may start on the SMs
    // that the previous kernel's CTAs leave and wait for that kernel at entry.
    return launch_pdl(quantize_tiles_kernel<ROW, COL, RHT, TWO_D, SR_ROW, SR_COL, true, false, FAST_RHT, SWZ>,
                      dim3(grid), dim3(kQuantThreads), kQuantSmemBytes, s, args);
  }
  return launch_pdl(quantize_tiles_kernel<ROW, COL, RHT, TWO_D, SR_ROW, SR_COL, false, false, FAST_RHT, SWZ>,
                    dim3(grid), dim3(kQuantThreads), kQuantSmemBytes, s, args);
}

template <bool ROW, bool COL, bool RHT, bool TWO_D, bool SR_ROW, bool SR_COL, bool FAST_RHT = false>
cudaError_t launch(const QuantArgs& args, int grid, cudaStream_t s) {
  return args.swz_scales
             ? launch_variant<ROW, COL, RHT, TWO_D, SR_ROW, SR_COL, FAST_RHT, true>(args, grid, s)
             : launch_variant<ROW, COL, RHT, TWO_D, SR_ROW, SR_COL, FAST_RHT, false>(args, grid, s);
}

// The amax pass (AMAX_ONLY) of a plain or grouped tensor.
template <bool RHT>
cudaError_t launch_amax_pass(const QuantArgs& args, int grid, cudaStream_t s) {
  if (args.offsets != nullptr)
    return launch_pdl(quantize_tiles_kernel<true, false, RHT, false, false, false, false, true, false, false, true>,
                      dim3(grid), dim3(kQuantThreads), kQuantSmemBytes, s, args);
  return launch_pdl(quantize_tiles_kernel<true, false, RHT, false, false, false, false, true>,
                    dim3(grid), dim3(kQuantThreads), kQuantSmemBytes, s, args);
}
template <bool RHT>
cudaError_t prepare_amax_pass() {
  cudaError_t e = cudaFuncSetAttribute(quantize_tiles_kernel<true, false, RHT, false, false, false, false, true>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kQuantSmemBytes);
  cudaError_t e2 = cudaFuncSetAttribute(
      quantize_tiles_kernel<true, false, RHT, false, false, false, false, true, false, false, true>,
      cudaFuncAttributeMaxDynamicSharedMemorySize, kQuantSmemBytes);
  return e != cudaSuccess ? e : e2;
}

template <bool ROW, bool COL, bool RHT, bool TWO_D, bool SR_ROW, bool SR_COL, bool FAST_RHT = false>
cudaError_t prepare() {
  cudaError_t e = cudaSuccess, r;
  auto set = [&](auto kernel) {
    if ((r = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  kQuantSmemBytes)) != cudaSuccess)
      e = r;
  };
  set(quantize_tiles_kernel<ROW, COL, RHT, TWO_D, SR_ROW, SR_COL, false, false, FAST_RHT, false>);
  set(quantize_tiles_kernel<ROW, COL, RHT, TWO_D, SR_ROW, SR_COL, true, false, FAST_RHT, false>);
  set(quantize_tiles_kernel<ROW, COL, RHT, TWO_D, SR_ROW, SR_COL, false, false, FAST_RHT, true>);
  set(quantize_tiles_kernel<ROW, COL, RHT, TWO_D, SR_ROW, SR_COL, true, false, FAST_RHT, true>);
  set(quantize_tiles_kernel<ROW, COL, RHT, TWO_D, SR_ROW, SR_COL, false, false, FAST_RHT, false, true>);
  return e;
}

}  // namespace qk
}  // namespace nvfp4
