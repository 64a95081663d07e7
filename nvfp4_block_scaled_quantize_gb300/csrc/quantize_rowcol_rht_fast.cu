// Instantiations of the quantize kernel (quantize_kernel.cuh): rowwise + columnwise after the RHT,
// fast math (the columnwise codes from the FP32 transform).
#include "quantize_kernel.cuh"

namespace nvfp4 {

cudaError_t launch_quantize_rowcol_rht_fast(const QuantMode& m, const QuantArgs& a, int grid,
                                            cudaStream_t s) {
  if (m.sr_row && m.sr_col) return qk::launch<true, true, true, false, true, true, true>(a, grid, s);
  if (m.sr_row) return qk::launch<true, true, true, false, true, false, true>(a, grid, s);
  if (m.sr_col) return qk::launch<true, true, true, false, false, true, true>(a, grid, s);
  return qk::launch<true, true, true, false, false, false, true>(a, grid, s);
}

cudaError_t prepare_quantize_rowcol_rht_fast() {
  cudaError_t e = cudaSuccess, r;
  if ((r = qk::prepare<true, true, true, false, true, true, true>()) != cudaSuccess) e = r;
  if ((r = qk::prepare<true, true, true, false, true, false, true>()) != cudaSuccess) e = r;
  if ((r = qk::prepare<true, true, true, false, false, true, true>()) != cudaSuccess) e = r;
  if ((r = qk::prepare<true, true, true, false, false, false, true>()) != cudaSuccess) e = r;
  return e;
}

}  // namespace nvfp4
