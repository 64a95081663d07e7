// Instantiations of the quantize kernel (quantize_kernel.cuh): 16x16 2D blocks.
#include "quantize_kernel.cuh"

namespace nvfp4 {

cudaError_t launch_quantize_2d(const QuantMode& m, const QuantArgs& a, int grid, cudaStream_t s) {
  if (m.row && m.col) return qk::launch<true, true, false, true, false, false>(a, grid, s);
  if (m.row) return qk::launch<true, false, false, true, false, false>(a, grid, s);
  return qk::launch<false, true, false, true, false, false>(a, grid, s);
}

cudaError_t prepare_quantize_2d() {
  cudaError_t e = cudaSuccess, r;
  if ((r = qk::prepare<true, true, false, true, false, false>()) != cudaSuccess) e = r;
  if ((r = qk::prepare<true, false, false, true, false, false>()) != cudaSuccess) e = r;
  if ((r = qk::prepare<false, true, false, true, false, false>()) != cudaSuccess) e = r;
  return e;
}

}  // namespace nvfp4
