// Internal declarations shared by the library's translation units (not part of the C ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace nvfp4 {

// ---- the quantize kernel's geometry ----
// A tile is kTileM rows x kTileN BF16 columns (one TMA box, one pipeline stage). A warp owns
// one 16-row slab of a tile; four warps (a group) share a tile; kGroups groups work on
// different tiles at once, and each group refills the stage it has just drained, so kStages
// tiles stay in flight.
constexpr int kTileM = 64;
constexpr int kTileN = 256;
constexpr int kStages = 4;
constexpr int kGroups = 3;
constexpr int kWarpsPerGroup = kTileM / 16;
constexpr int kConsumerWarps = kGroups * kWarpsPerGroup;
constexpr int kQuantThreads = 32 * kConsumerWarps;
constexpr int kStageBytes = kTileM * kTileN * 2;
constexpr int kMaxSegments = 256;
constexpr int kTableEntries = 128;  // E4M3 codes of non-negative scales

// Shared-memory layout of the quantize kernel (byte offsets).
constexpr int kColCodeStage = kWarpsPerGroup * kTileN * 8;   // [4 slabs][128 chunks][16 B]
constexpr int kColScaleStage = kWarpsPerGroup * kTileN;      // [4 slabs][256 B]
constexpr int kSmemStages = 0;
constexpr int kSmemColCodes = kSmemStages + kStages * kStageBytes;
constexpr int kSmemColScales = kSmemColCodes + kGroups * kColCodeStage;
constexpr int kSmemTables = kSmemColScales + kGroups * kColScaleStage;  // per group: 2 x 128 f32
constexpr int kSmemSegStart = kSmemTables + kGroups * 2 * kTableEntries * 4;
constexpr int kSmemSegEnd = kSmemSegStart + 4 * kMaxSegments;
constexpr int kSmemSegCol0 = kSmemSegEnd + 4 * kMaxSegments;
constexpr int kSmemSegTile0 = kSmemSegCol0 + 4 * kMaxSegments;        // [kMaxSegments + 4]
constexpr int kSmemCoords = kSmemSegTile0 + 4 * (kMaxSegments + 4);   // [kStages][8] int32
constexpr int kSmemBars = kSmemCoords + 32 * kStages;                 // full[kStages]
constexpr int kSmemFlags = kSmemBars + 8 * kStages;                   // int32 [4]
constexpr int kSmemIssued = kSmemFlags + 16;                          // int32 [kStages]
constexpr int kSmemFused = kSmemIssued + 4 * kStages;            // uint32 [32 + 4]
constexpr int kQuantSmemBytes = kSmemFused + 4 * 36;

// Workspace of the single-launch (fused amax) path, 8-byte aligned: word 0 counts CTA arrivals
// (it only grows; the host knows the value each launch must reach), words 2-3 and 4-5 are the
// rowwise and columnwise maxima as (launch epoch << 16) | 16-bit magnitude. Epochs increase
// from launch to launch, so an atomic max needs no clearing in between.
constexpr int kFuseMaxCtas = 1024;
constexpr int kFuseWsWords = 6;

// Arguments of the quantize kernel: one BF16 tensor split into row segments (one segment for
// a plain tensor, one per expert for the grouped case).
struct QuantArgs {
  CUtensorMap tmap;                 // x as BF16 [rows][cols], box {kTileN, kTileM}
  const void* x;                    // the same tensor, for the fused amax phase
  int64_t rows, cols;
  const int32_t* offsets;           // cumulative segment ends, or nullptr: one segment
  int32_t segments;
  uint32_t sign_mask;
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
  uint32_t rng_offset;
  uint32_t* status;
  int32_t fused;                    // 1: compute the amax inside this launch (one segment)
  int32_t fast;                     // 1: fast-math element multipliers (rcp.approx)
  uint32_t fuse_target;             // fuse_ws[0] once every CTA of this launch has arrived
  uint64_t fuse_epoch;              // larger than any earlier launch's on fuse_ws (< 2^48)
  uint32_t* fuse_ws;                // kFuseWsWords words, 8-byte aligned
};

// What one quantize launch produces.
struct QuantMode {
  bool row, col, rht, two_d, sr_row, sr_col;
  bool fast;  // fast math with the RHT: the columnwise transform is not rounded through BF16
};

cudaError_t launch_quantize(const QuantMode& m, const QuantArgs& args, int grid, cudaStream_t s);
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
cudaError_t launch_quantize_2d(const QuantMode& m, const QuantArgs& a, int grid, cudaStream_t s);
cudaError_t prepare_quantize_row();
cudaError_t prepare_quantize_col();
cudaError_t prepare_quantize_rowcol();
cudaError_t prepare_quantize_rowcol_rht();
cudaError_t prepare_quantize_2d();

// ---- MX formats (mx_kernel.cu): 32-element blocks, E8M0 scales, no tensor scale ----
// A warp quantizes 32 x 128 units alone, kMxStages of them in flight in its own ring; a unit is
// two TMA boxes of 32 rows x 64 BF16 columns (128-byte rows, 128-byte swizzle). Its codes are
// staged in kMxOutBytes of shared memory per warp and leave by TMA stores.
constexpr int kMxUnitM = 32;
constexpr int kMxUnitN = 128;
constexpr int kMxWarps = 8;
constexpr int kMxStages = 2;
constexpr int kMxOutBytes = 8192;  // row codes, then column codes: 4 KiB each (FP8)
constexpr int kMxSmemBytes = kMxWarps * (kMxStages * (kMxUnitM * kMxUnitN * 2) + kMxOutBytes) +
                             2 * kMxWarps * kMxUnitN + kMxWarps * kMxStages * 8 + 1024;

struct MxArgs {
  CUtensorMap tmap;        // x as BF16 [rows][cols], box {64, 32}, 128-byte swizzle
  CUtensorMap tmap_row;    // row codes as bytes, box {128 (FP4: 64), 32}, swizzle span = row
  CUtensorMap tmap_col;    // column codes as bytes {M, N/4, 4}, box {32 (FP4: 16), 32, 4}
  int64_t rows, cols;
  uint8_t* row_codes;      // [rows][cols] FP8 or [rows][cols / 2] FP4
  uint8_t* row_scales;     // [rows][cols / 32] E8M0
  uint8_t* col_codes;      // [cols][rows] FP8 or [cols][rows / 2] FP4
  uint8_t* col_scales;     // [cols][rows / 32] E8M0
  uint32_t* status;
};
// fmt: 0 = E4M3, 1 = E5M2, 2 = E2M1
cudaError_t launch_mx_quantize(int fmt, bool row, bool col, const MxArgs& args, int grid,
                               cudaStream_t s);
cudaError_t prepare_mx_kernels();
cudaError_t launch_mx_dequantize(int fmt, const uint8_t* codes, const uint8_t* scales, int64_t R,
                                 int64_t C, float* out, int grid, cudaStream_t s);

// RMSNorm producer with the amax in its epilogue (producer.cu): y and an atomic max of |y|
// into *amax (zeroed by the caller); rmsnorm_rows_per_cta() rows per CTA.
cudaError_t launch_rmsnorm_amax(const void* x, const void* w, int64_t M, int64_t N, float eps,
                                float bias, void* y, float* amax, int grid, cudaStream_t s);
int rmsnorm_rows_per_cta();

cudaError_t launch_amax_flat(const void* x, int64_t n_elems, float* out0, float* out1, int grid,
                             cudaStream_t s);
cudaError_t launch_swizzle_scales(const uint8_t* scales, int64_t R, int64_t C, uint8_t* out,
                                  int grid, cudaStream_t s);
cudaError_t launch_dequantize(const uint8_t* codes, const uint8_t* scales, const float* gscale,
                              int64_t R, int64_t C, bool inverse_rht, uint32_t sign_mask,
                              bool out_bf16, void* out, int grid, cudaStream_t s);

}  // namespace nvfp4
