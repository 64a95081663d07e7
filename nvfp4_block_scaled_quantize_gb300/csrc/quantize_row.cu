// Instantiations of the quantize kernel (quantize_kernel.cuh): rowwise only.
#include "quantize_kernel.cuh"

namespace nvfp4 {

cudaError_t launch_quantize_row(const QuantMode& m, const QuantArgs& a, int grid, cudaStream_t s) {
  if (m.sr_row) return qk::launch<true, false, false, false, true, false>(a, grid, s);
  return qk::launch<true, false, false, false, false, false>(a, grid, s);
}

cudaError_t prepare_quantize_row() {
  cudaError_t e = cudaSuccess, r;
  if ((r = qk::prepare<true, false, false, false, true, false>()) != cudaSuccess) e = r;
  if ((r = qk::prepare<true, false, false, false, false, false>()) != cudaSuccess) e = r;
  return e;
}

}  // namespace nvfp4
