// A producer with the amax in its epilogue: RMSNorm of a BF16 tensor that also folds max |y|
// into a device scalar, so that the quantize call that follows takes the amax as an input and
// skips its amax pass (one read of the tensor less).
//
// Page cited: "CuTeDSL at Perplexity", its RMS-norm kernel: y = bf16((w + bias) * (x * rms)),
// rms = rsqrt(sum(x^2) / N + eps), the sum of squares taken per thread over its 8-element
// vectors and then across the warp by a butterfly of shuffles. Here a warp owns a row: lane l
// sums the squares of vectors l, l + 32, ... in order, the butterfly (xor 16, 8, 4, 2, 1) gives
// every lane the same total, and the second sweep over the row (from L1) writes y. Every float
// step is one IEEE binary32 operation (the reciprocal square root correctly rounded), so the
// output is reproducible bit for bit.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "nvfp4_device.cuh"
#include "aux_internal.h"
#include "nvfp4_internal.h"

namespace nvfp4 {
namespace {

constexpr int kNormWarps = 8;
constexpr int kBatch = 4;  // vectors per lane loaded together

__global__ void __launch_bounds__(32 * kNormWarps) rmsnorm_amax_kernel(
    const uint4* __restrict__ x, const uint4* __restrict__ w, int64_t M, int64_t N, float eps,
    float bias, uint4* __restrict__ y, float* __restrict__ amax) {
  __shared__ uint32_t red[kNormWarps];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int64_t nv = N / 8;  // 8-element vectors per row
  uint32_t m = 0u;           // largest |y| so far, as a BF16 magnitude
  for (int64_t r = (int64_t)blockIdx.x * kNormWarps + warp; r < M;
       r += (int64_t)gridDim.x * kNormWarps) {
    const uint4* xr = x + r * nv;
    float s = 0.0f;
    // kBatch of the lane's vectors loaded at once (more loads in flight), then summed in order
    for (int64_t v0 = lane; v0 < nv; v0 += 32 * kBatch) {
      uint4 q[kBatch];
#pragma unroll
      for (int j = 0; j < kBatch; j++)
        q[j] = v0 + 32 * j < nv ? xr[v0 + 32 * j] : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int j = 0; j < kBatch; j++) {
        const uint32_t e[4] = {q[j].x, q[j].y, q[j].z, q[j].w};
#pragma unroll
        for (int i = 0; i < 4; i++) {
          const float lo = bf16_lo(e[i]), hi = bf16_hi(e[i]);
          s = __fadd_rn(s, __fmul_rn(lo, lo));  // (vectors past the row add +0: s unchanged)
          s = __fadd_rn(s, __fmul_rn(hi, hi));
        }
      }
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) s = __fadd_rn(s, __shfl_xor_sync(0xFFFFFFFFu, s, o));
    const float rms = __frsqrt_rn(__fadd_rn(__fdiv_rn(s, (float)N), eps));
    for (int64_t v0 = lane; v0 < nv; v0 += 32 * kBatch) {
      uint4 q[kBatch], qw[kBatch];
#pragma unroll
      for (int j = 0; j < kBatch; j++) {
        const bool in = v0 + 32 * j < nv;
        q[j] = in ? xr[v0 + 32 * j] : make_uint4(0u, 0u, 0u, 0u);
        qw[j] = in ? w[v0 + 32 * j] : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int j = 0; j < kBatch; j++) {
        if (v0 + 32 * j >= nv) break;
        const uint32_t e[4] = {q[j].x, q[j].y, q[j].z, q[j].w};
        const uint32_t g[4] = {qw[j].x, qw[j].y, qw[j].z, qw[j].w};
        uint32_t o[4];
#pragma unroll
        for (int i = 0; i < 4; i++) {
          const float y0 = __fmul_rn(__fadd_rn(bf16_lo(g[i]), bias), __fmul_rn(bf16_lo(e[i]), rms));
          const float y1 = __fmul_rn(__fadd_rn(bf16_hi(g[i]), bias), __fmul_rn(bf16_hi(e[i]), rms));
          const __nv_bfloat162 p = __floats2bfloat162_rn(y0, y1);
          o[i] = *reinterpret_cast<const uint32_t*>(&p);
          m = max(m, max(o[i] & 0x7FFFu, (o[i] >> 16) & 0x7FFFu));
        }
        y[r * nv + v0 + 32 * j] = make_uint4(o[0], o[1], o[2], o[3]);
      }
    }
  }
  // epilogue: the CTA's largest magnitude, one atomic max on the float's bits (non-negative
  // floats order like their bit patterns)
  m = __reduce_max_sync(0xFFFFFFFFu, m);
  if (lane == 0) red[warp] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t t = 0u;
#pragma unroll
    for (int k = 0; k < kNormWarps; k++) t = max(t, red[k]);
    atomicMax(reinterpret_cast<unsigned int*>(amax), t << 16);
  }
}

}  // namespace

cudaError_t launch_rmsnorm_amax(const void* x, const void* w, int64_t M, int64_t N, float eps,
                                float bias, void* y, float* amax, int grid, cudaStream_t s) {
  rmsnorm_amax_kernel<<<grid, 32 * kNormWarps, 0, s>>>(
      static_cast<const uint4*>(x), static_cast<const uint4*>(w), M, N, eps, bias,
      static_cast<uint4*>(y), amax);
  return cudaGetLastError();
}

int rmsnorm_rows_per_cta() { return kNormWarps; }

}  // namespace nvfp4
