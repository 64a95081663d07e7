// Instantiations of the quantize kernel (quantize_kernel.cuh): rowwise + columnwise after the RHT,
// exact (the transform rounded through BF16); the fast-math variants are in
// quantize_rowcol_rht_fast.cu, so that the two compile in parallel.
#include "quantize_kernel.cuh"

namespace nvfp4 {

cudaError_t launch_quantize_rowcol_rht(const QuantMode& m, const QuantArgs& a, int grid, cudaStream_t s) {
  if (m.sr_row && m.sr_col) return qk::launch<true, true, true, false, true, true>(a, grid, s);
  if (m.sr_row) return qk::launch<true, true, true, false, true, false>(a, grid, s);
  if (m.sr_col) return qk::launch<true, true, true, false, false, true>(a, grid, s);
  return qk::launch<true, true, true, false, false, false>(a, grid, s);
}

cudaError_t prepare_quantize_rowcol_rht() {
  cudaError_t e = cudaSuccess, r;
  if ((r = qk::prepare<true, true, true, false, true, true>()) != cudaSuccess) e = r;
  if ((r = qk::prepare<true, true, true, false, true, false>()) != cudaSuccess) e = r;
  if ((r = qk::prepare<true, true, true, false, false, true>()) != cudaSuccess) e = r;
  if ((r = qk::prepare<true, true, true, false, false, false>()) != cudaSuccess) e = r;
  return e;
}

}  // namespace nvfp4
