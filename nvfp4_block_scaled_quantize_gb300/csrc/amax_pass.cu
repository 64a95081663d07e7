// Instantiations of the quantize kernel (quantize_kernel.cuh) as the amax pass alone: the
// per-segment amax, and the RHT amax of the columnwise blocks, streamed through the same TMA
// stage ring (grouped tensors, and the RHT amax of plain ones).
#include "quantize_kernel.cuh"

namespace nvfp4 {

cudaError_t launch_amax_tiles(bool rht, const QuantArgs& a, int grid, cudaStream_t s) {
  return rht ? qk::launch_amax_pass<true>(a, grid, s) : qk::launch_amax_pass<false>(a, grid, s);
}

cudaError_t prepare_amax_tiles() {
  cudaError_t e = qk::prepare_amax_pass<true>();
  cudaError_t r = qk::prepare_amax_pass<false>();
  return e != cudaSuccess ? e : r;
}

}  // namespace nvfp4
