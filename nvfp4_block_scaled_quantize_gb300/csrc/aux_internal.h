// Internal declarations of the library's kernels other than the tile kernel (not part of the
// C ABI): MX quantization, the RMSNorm producer, the flat amax, the scale swizzle and
// dequantization. Kept apart from nvfp4_internal.h, whose contents the tile kernel depends on.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace nvfp4 {

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
