// Internal declarations shared by the library's translation units (not part of the C ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace nvfp4 {

// ---- the quantize kernel's geometry ----
// A tile is kTileM rows x kTileN BF16 columns (one pipeline stage: one TMA box, or one box per
// 16-row slab where a grouped tile's slabs are not consecutive rows of x). A warp owns one
// slab of a tile; four warps (a group) share a tile; kGroups groups work on different tiles at
// once, and each group refills the stage it has just drained, so kStages tiles stay in flight.
constexpr int kTileM = 64;
constexpr int kTileN = 256;
constexpr int kStages = 4;
constexpr int kGroups = 3;
constexpr int kWarpsPerGroup = kTileM / 16;
constexpr int kConsumerWarps = kGroups * kWarpsPerGroup;
constexpr int kQuantThreads = 32 * kConsumerWarps;
constexpr int kStageBytes = kTileM * kTileN * 2;
constexpr int kSlabBytes = 16 * kTileN * 2;
constexpr int kMaxSegments = 256;
constexpr int kTableEntries = 128;  // E4M3 codes of non-negative scales
// A segment's scale block: the rowwise and columnwise reciprocal tables (f32 [2][128]), then
// {S_enc row, S_enc col} and 8 bytes of padding.
constexpr int kTableBlock = 2 * kTableEntries * 4 + 16;

// Shared-memory layout of the quantize kernel (byte offsets).
constexpr int kColCodeStage = kWarpsPerGroup * kTileN * 8;   // [4 slabs][128 chunks][16 B]
constexpr int kColScaleStage = kWarpsPerGroup * kTileN;      // [4 slabs][256 B]
constexpr int kSmemStages = 0;
constexpr int kSmemColCodes = kSmemStages + kStages * kStageBytes;
constexpr int kColStageBufs = 2;                             // per group (double-buffered)
constexpr int kSmemColScales = kSmemColCodes + kGroups * kColStageBufs * kColCodeStage;
constexpr int kSmemTables = kSmemColScales + kGroups * kColStageBufs * kColScaleStage;  // per group: a scale block
// per segment {first slab, first row, end row, next segment's first slab}, [kMaxSegments + 1]
constexpr int kSmemSegRec = kSmemTables + kGroups * kTableBlock;
// per segment {S_enc row, S_dec row, S_enc col, S_dec col}, [kMaxSegments]
constexpr int kSmemSegScale = kSmemSegRec + 16 * (kMaxSegments + 1);
constexpr int kSmemCoords = kSmemSegScale + 16 * kMaxSegments;      // [kStages][16] int32
constexpr int kSmemBars = kSmemCoords + 64 * kStages;                 // full[kStages]
constexpr int kSmemFlags = kSmemBars + 8 * kStages;                   // int32 [4]
constexpr int kSmemSegHint = kSmemFlags + 16;                         // int32 [kConsumerWarps]
constexpr int kSmemIssued = kSmemSegHint + 4 * kConsumerWarps;        // int32 [kStages]
constexpr int kSmemFused = kSmemIssued + 4 * kStages;            // uint32 [32 + 4]
// single-launch amax: the ranks this CTA does the amax of, each with its first ring slot
constexpr int kMaxHeld = 128;
constexpr int kSmemHeld = kSmemFused + 4 * 36;                   // int32 [2][kMaxHeld]
constexpr int kSmemFuseCtl = kSmemHeld + 8 * kMaxHeld;            // int32 [4]
// per warp: a scale block for a slab of another segment than its group's
constexpr int kSmemWarpTables = kSmemFuseCtl + 16;
constexpr int kQuantSmemBytes = kSmemWarpTables + kConsumerWarps * kTableBlock;
static_assert(kSmemSegRec % 16 == 0 && kSmemSegScale % 16 == 0 && kSmemCoords % 16 == 0 &&
                  kSmemBars % 8 == 0 && kSmemWarpTables % 16 == 0,
              "shared-memory record alignment");

// Workspace of the single-launch (fused amax) path, 4-byte aligned, zeroed before first use:
// the count of ranks arrived, the count of CTAs done with the words, the rowwise and
// columnwise maxima, a statistics counter and one claim bit per rank, all kept on the device
// (fused_amax.cuh). At most kFuseMaxCtas CTAs (one claim bit each).
constexpr int kFuseMaxCtas = 1024;
constexpr int kFuseWsWords = 8 + kFuseMaxCtas / 32;
constexpr int kFuseStatsWord = 4;  // ranks taken over from another CTA (statistics)

// Arguments of the quantize kernel: one BF16 tensor split into row segments (one segment for
// a plain tensor, one per expert for the grouped case).
struct QuantArgs {
  CUtensorMap tmap;                 // x as BF16 [rows][cols], box {kTileN, kTileM}
  CUtensorMap tmap_slab;            // the same, box {kTileN, 16} (grouped tensors only)
  CUtensorMap tmap_colc;            // col_codes as bytes {col_ld / 2, cols / 8, 8} (column 8y + z),
                                    // box {kTileM / 2, kTileN / 8, 8}, 32-byte swizzle
  int32_t col_tma;                  // 1: whole tiles' columnwise codes leave by TMA (tmap_colc)
  int32_t swz_scales;               // 1: both scale outputs in the 128 x 4 tiled layout
  int64_t row_swz_tc, col_swz_tc;   // tiles per tile row of that layout: ceil(scale columns / 4)
  const void* x;                    // the same tensor, for the fused amax phase
  int64_t rows, cols;
  const int32_t* offsets;           // cumulative segment ends, or nullptr: one segment
  int32_t segments;
  uint32_t sign_mask;
  uint32_t rht_flip[16];            // 0x80000000 where bit i of sign_mask is set (set_rht_flips)
  int64_t col_ld;                   // columnwise output row length (elements)
  const float* amax_row;            // amax of segment e at amax_row[e * amax_row_stride]
  const float* amax_col;
  int32_t amax_row_stride, amax_col_stride;
  uint8_t* row_codes;
  uint8_t* row_scales;
  float* row_gscale;                // [segments][2] = {amax, S_dec}
  uint8_t* col_codes;
  uint8_t* col_scales;
  float* col_gscale;
  uint64_t seed;
  uint32_t philox_key[2][10];       // Philox round keys of seed (set_philox_keys)
  uint32_t rng_offset;
  uint32_t* status;
  int32_t fused;                    // 1: compute the amax inside this launch (one segment)
  int32_t fast;                     // 1: fast-math element multipliers (rcp.approx)
  int32_t fuse_extra;               // arrivals awaited beyond the grid's: 0 (> 0 only to make
                                    // the barrier time out on purpose, in tests)
  int32_t fuse_late;                // the last fuse_late CTAs start only once every rank has
                                    // arrived (bounded): 0 (> 0 only in tests, so that the
                                    // other CTAs take their ranks over)
  uint32_t* fuse_ws;                // kFuseWsWords words, 4-byte aligned (fused_amax.cuh)
};

// Launch with programmatic dependent launch: the kernel may start before the previous kernel
// in the stream ends, so it must call pdl_wait() (nvfp4_device.cuh) before any memory access.
template <typename... KernelArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KernelArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// Round keys of Philox4x32-10 for a 64-bit seed: key (lo32, hi32) bumped by the Weyl constants
// 0x9E3779B9 and 0xBB67AE85 each round. Computed once per launch on the host, so that the
// kernels read them from their parameters instead of recomputing the schedule per draw.
inline void set_philox_keys(QuantArgs& a, uint64_t seed) {
  uint32_t k0 = (uint32_t)seed, k1 = (uint32_t)(seed >> 32);
  for (int r = 0; r < 10; r++) {
    a.philox_key[0][r] = k0;
    a.philox_key[1][r] = k1;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
}

// The RHT's sign flips as words (the sign bit of a binary32), so that the kernels take them
// from their parameters.
inline void set_rht_flips(QuantArgs& a, uint32_t sign_mask) {
  a.sign_mask = sign_mask;
  for (int i = 0; i < 16; i++) a.rht_flip[i] = ((sign_mask >> i) & 1u) ? 0x80000000u : 0u;
}

// Scale outputs in the 128 x 4 tiled layout (nvfp4_config.swizzle_scales): the tiles per tile
// row for the kernel, and the buffers zeroed first when the scale matrix does not fill whole
// tiles (the padding of that layout is zero). A NULL buffer: that side is not produced.
inline cudaError_t prepare_swizzled_scales(QuantArgs& q, uint8_t* row_scales, uint8_t* col_scales,
                                           int64_t M, int64_t N, cudaStream_t s) {
  q.swz_scales = 1;
  q.row_swz_tc = (N / 16 + 3) / 4;
  q.col_swz_tc = (M / 16 + 3) / 4;
  cudaError_t e = cudaSuccess;
  if (row_scales && (M % 128 != 0 || (N / 16) % 4 != 0))
    e = cudaMemsetAsync(row_scales, 0, (size_t)((M + 127) / 128) * q.row_swz_tc * 512, s);
  if (e == cudaSuccess && col_scales && (N % 128 != 0 || (M / 16) % 4 != 0))
    e = cudaMemsetAsync(col_scales, 0, (size_t)((N + 127) / 128) * q.col_swz_tc * 512, s);
  return e;
}

// What one quantize launch produces.
struct QuantMode {
  bool row, col, rht, two_d, sr_row, sr_col;
  bool fast;  // fast math with the RHT: the columnwise transform is not rounded through BF16
};

cudaError_t launch_quantize(const QuantMode& m, const QuantArgs& args, int grid, cudaStream_t s);
// The single-launch amax's test hooks for the next launch (fuse_extra, fuse_late), taken once.
void take_fuse_debug(QuantArgs& q);
cudaError_t prepare_quantize_kernels();
// The amax pass alone through the tile kernel (per segment; RHT amax when rht): atomic maxima
// into args.amax_row / args.amax_col, which the caller zeroes.
cudaError_t launch_amax_tiles(bool rht, const QuantArgs& args, int grid, cudaStream_t s);
cudaError_t prepare_amax_tiles();
// per-translation-unit halves of the above
cudaError_t launch_quantize_row(const QuantMode& m, const QuantArgs& a, int grid, cudaStream_t s);
cudaError_t launch_quantize_col(const QuantMode& m, const QuantArgs& a, int grid, cudaStream_t s);
cudaError_t launch_quantize_rowcol(const QuantMode& m, const QuantArgs& a, int grid, cudaStream_t s);
cudaError_t launch_quantize_rowcol_rht(const QuantMode& m, const QuantArgs& a, int grid,
                                       cudaStream_t s);
cudaError_t launch_quantize_rowcol_rht_fast(const QuantMode& m, const QuantArgs& a, int grid,
                                            cudaStream_t s);
cudaError_t launch_quantize_2d(const QuantMode& m, const QuantArgs& a, int grid, cudaStream_t s);
cudaError_t prepare_quantize_row();
cudaError_t prepare_quantize_col();
cudaError_t prepare_quantize_rowcol();
cudaError_t prepare_quantize_rowcol_rht();
cudaError_t prepare_quantize_rowcol_rht_fast();
cudaError_t prepare_quantize_2d();

}  // namespace nvfp4
