// Instantiations of the quantize kernel (quantize_kernel.cuh): rowwise + columnwise after the RHT,
// exact (transform rounded through BF16) and fast math (FP32 transform).
#include "quantize_kernel.cuh"

namespace nvfp4 {

namespace {

template <bool F>
cudaError_t launch_rowcol_rht(const QuantMode& m, const QuantArgs& a, int grid, cudaStream_t s) {
  if (m.sr_row && m.sr_col) return qk::launch<true, true, true, false, true, true, F>(a, grid, s);
  if (m.sr_row) return qk::launch<true, true, true, false, true, false, F>(a, grid, s);
  if (m.sr_col) return qk::launch<true, true, true, false, false, true, F>(a, grid, s);
  return qk::launch<true, true, true, false, false, false, F>(a, grid, s);
}

template <bool F>
cudaError_t prepare_rowcol_rht() {
  cudaError_t e = cudaSuccess, r;
  if ((r = qk::prepare<true, true, true, false, true, true, F>()) != cudaSuccess) e = r;
  if ((r = qk::prepare<true, true, true, false, true, false, F>()) != cudaSuccess) e = r;
  if ((r = qk::prepare<true, true, true, false, false, true, F>()) != cudaSuccess) e = r;
  if ((r = qk::prepare<true, true, true, false, false, false, F>()) != cudaSuccess) e = r;
  return e;
}

}  // namespace

cudaError_t launch_quantize_rowcol_rht(const QuantMode& m, const QuantArgs& a, int grid, cudaStream_t s) {
  return m.fast ? launch_rowcol_rht<true>(m, a, grid, s) : launch_rowcol_rht<false>(m, a, grid, s);
}

cudaError_t prepare_quantize_rowcol_rht() {
  const cudaError_t e = prepare_rowcol_rht<false>();
  const cudaError_t f = prepare_rowcol_rht<true>();
  return e != cudaSuccess ? e : f;
}

}  // namespace nvfp4
