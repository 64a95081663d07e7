// Instantiations of the quantize kernel (quantize_kernel.cuh): columnwise only, with or without
// the RHT (exact or fast math).
#include "quantize_kernel.cuh"

namespace nvfp4 {

cudaError_t launch_quantize_col(const QuantMode& m, const QuantArgs& a, int grid, cudaStream_t s) {
  if (m.rht && m.fast) {
    if (m.sr_col) return qk::launch<false, true, true, false, false, true, true>(a, grid, s);
    return qk::launch<false, true, true, false, false, false, true>(a, grid, s);
  }
  if (m.rht && m.sr_col) return qk::launch<false, true, true, false, false, true>(a, grid, s);
  if (m.rht) return qk::launch<false, true, true, false, false, false>(a, grid, s);
  if (m.sr_col) return qk::launch<false, true, false, false, false, true>(a, grid, s);
  return qk::launch<false, true, false, false, false, false>(a, grid, s);
}

cudaError_t prepare_quantize_col() {
  cudaError_t e = cudaSuccess, r;
  if ((r = qk::prepare<false, true, true, false, false, true, true>()) != cudaSuccess) e = r;
  if ((r = qk::prepare<false, true, true, false, false, false, true>()) != cudaSuccess) e = r;
  if ((r = qk::prepare<false, true, true, false, false, true>()) != cudaSuccess) e = r;
  if ((r = qk::prepare<false, true, true, false, false, false>()) != cudaSuccess) e = r;
  if ((r = qk::prepare<false, true, false, false, false, true>()) != cudaSuccess) e = r;
  if ((r = qk::prepare<false, true, false, false, false, false>()) != cudaSuccess) e = r;
  return e;
}

}  // namespace nvfp4
