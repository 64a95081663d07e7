// Internal declarations shared by the library's translation units (not part of the C ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace nvfp4 {

// Tile of the quantize kernels: kTileM rows x kTileN BF16 columns, one TMA box per stage.
constexpr int kTileM = 64;
constexpr int kTileN = 256;
constexpr int kStages = 4;
constexpr int kQuantThreads = 512;
constexpr int kStageBytes = kTileM * kTileN * 2;
constexpr int kMaxSegments = 256;

// Shared-memory layout of the quantize kernels (byte offsets).
constexpr int kColCodeStage = (kTileM / 16) * kTileN * 8;    // [4 row-blocks][256 cols][8 B]
constexpr int kColScaleStage = (kTileM / 16) * kTileN;       // [4][256]
constexpr int kRowScaleStage = kTileM * (kTileN / 16);       // [64 rows][16]
constexpr int kSmemStages = 0;
constexpr int kSmemColCodes = kSmemStages + kStages * kStageBytes;
constexpr int kSmemColScales = kSmemColCodes + 2 * kColCodeStage;
constexpr int kSmemRowScales = kSmemColScales + 2 * kColScaleStage;
constexpr int kSmemTileR = kSmemRowScales + 2 * kRowScaleStage;       // float [4][16]
constexpr int kSmemTileS = kSmemTileR + 4 * 16 * 4;                   // uint8 [4][16]
constexpr int kSmemSegStart = kSmemTileS + 64;                        // int32 [kMaxSegments]
constexpr int kSmemSegEnd = kSmemSegStart + 4 * kMaxSegments;
constexpr int kSmemSegCol0 = kSmemSegEnd + 4 * kMaxSegments;
constexpr int kSmemSegTile0 = kSmemSegCol0 + 4 * kMaxSegments;        // int32 [kMaxSegments + 1]
constexpr int kSmemSegScale = kSmemSegTile0 + 4 * (kMaxSegments + 4); // float4 [kMaxSegments]
constexpr int kSmemBars = kSmemSegScale + 16 * kMaxSegments;          // uint64 [kStages]
constexpr int kSmemFlags = kSmemBars + 8 * kStages;                   // int32 [4]
constexpr int kQuantSmemBytes = kSmemFlags + 16;

// Arguments of the tile kernel: one BF16 tensor split into row segments (one segment for a
// plain tensor, one per expert for the grouped case).
struct QuantArgs {
  CUtensorMap tmap;                 // x as BF16 [rows][cols], box {kTileN, kTileM}
  int64_t rows, cols;
  const int32_t* offsets;           // cumulative segment ends, or nullptr: one segment
  int32_t segments;
  int32_t sr_row, sr_col;
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
};

// Kernel variants of the tile kernel.
enum QuantVariant : int {
  kRow = 0, kCol, kColRht, kRowCol, kRowColRht, k2dRow, k2dCol, k2dRowCol, kNumQuantVariants
};

// Arguments of the amax kernels.
struct AmaxArgs {
  const void* x;
  int64_t rows, cols;
  const int32_t* offsets;           // nullptr: one segment [0, rows)
  int32_t segments;
  uint32_t sign_mask;
  float* amax_row;                  // max |x| per segment at amax_row[e * stride_row] (or null)
  float* amax_col;                  // max |RHT(x)| (rht) or max |x| per segment (or null)
  int32_t stride_row, stride_col;
  uint32_t* status;
};

cudaError_t launch_quantize(QuantVariant v, const QuantArgs& args, int grid, cudaStream_t s);
cudaError_t launch_amax_flat(const void* x, int64_t n_elems, float* out0, float* out1, int grid,
                             cudaStream_t s);
cudaError_t launch_amax_blocks(bool rht, const AmaxArgs& args, int grid, cudaStream_t s);
cudaError_t launch_dequantize(const uint8_t* codes, const uint8_t* scales, const float* gscale,
                              int64_t R, int64_t C, float* out, int grid, cudaStream_t s);
cudaError_t prepare_quantize_kernels();

}  // namespace nvfp4
