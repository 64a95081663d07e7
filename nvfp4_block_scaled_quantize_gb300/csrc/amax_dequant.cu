// The flat amax kernel (plain tensors without the RHT) and dequantization. The per-segment
// and RHT amax run through the tile kernel (amax_pass.cu).
//
// Page cited: "[nvfp4_training] Optimize CuteDSL kernels for NVFP4 training" (pytorch/ao pull
// request #4798): the amax pre-pass ("Optimization" item 5: "Linear RHT amax"; "Performance":
// grouped amax) and the dequantized reconstruction its "Correctness" section measures SQNR on.
#include <cuda_bf16.h>

#include "nvfp4_device.cuh"
#include "aux_internal.h"
#include "nvfp4_internal.h"

namespace nvfp4 {

namespace {

__device__ __forceinline__ uint4 ldg_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t max4(uint4 v) {
  return vmax2(vmax2(abs2(v.x), abs2(v.y)), vmax2(abs2(v.z), abs2(v.w)));
}

// Block-wide max of a 16-bit magnitude, then one atomic per block into each output (the
// float bits of a non-negative value order like unsigned integers).
__device__ __forceinline__ void block_max_out(uint32_t v, float* out0, float* out1) {
  __shared__ uint32_t red[32];
  v = __reduce_max_sync(0xFFFFFFFFu, v);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) red[warp] = v;
  __syncthreads();
  if (warp == 0) {
    v = (lane < (int)(blockDim.x >> 5)) ? red[lane] : 0u;
    v = __reduce_max_sync(0xFFFFFFFFu, v);
    if (lane == 0 && v != 0u) {
      if (out0) atomicMax(reinterpret_cast<unsigned int*>(out0), v << 16);
      if (out1) atomicMax(reinterpret_cast<unsigned int*>(out1), v << 16);
    }
  }
}

// max |x| over a contiguous BF16 buffer of nvec 16-byte vectors. Four CTAs of 256 threads per
// SM, each thread with kFlatUnroll independent 16-byte loads in flight (128 KiB per SM).
constexpr int kFlatUnroll = 8;
__global__ void __launch_bounds__(256, 4) amax_flat_kernel(const uint4* __restrict__ x, int64_t nvec,
                                                           float* out0, float* out1) {
  pdl_wait();  // launched with programmatic dependent launch: the previous kernel may produce x
  pdl_allow_next();
  uint32_t m = 0;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nvec;
       i += kFlatUnroll * stride) {
    uint4 v[kFlatUnroll];
#pragma unroll
    for (int u = 0; u < kFlatUnroll; u++)
      v[u] = (i + u * stride < nvec) ? ldg_stream(x + i + u * stride) : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int u = 0; u < kFlatUnroll; u++) m = vmax2(m, max4(v[u]));
  }
  block_max_out(max(m & 0xFFFFu, m >> 16), out0, out1);
}

// E2M1 code -> value (exact).
__device__ __forceinline__ float e2m1_value(uint32_t nib) {
  const uint32_t c = nib & 7u;
  const float mag = (c < 2u) ? 0.5f * (float)c
                             : __uint_as_float((((c >> 1) + 126u) << 23) | ((c & 1u) << 22));
  return (nib & 8u) ? -mag : mag;
}

// out[r][c] = (e2m1(code) * e4m3(scale)) * S_dec, one 16-element block per step. RHT: then the
// inverse 16-point RHT of the block, v = d * (0.25 * FWHT16(y)) with the forward butterflies
// (stages 1, 2, 4, 8; (a, b) -> (a + b, a - b)); BF16: the results rounded to nearest-even.
template <bool RHT, bool BF16>
__global__ void __launch_bounds__(256) dequantize_kernel(const uint8_t* __restrict__ codes,
                                                         const uint8_t* __restrict__ scales,
                                                         const float* __restrict__ gscale,
                                                         int64_t R, int64_t C, uint32_t sign_mask,
                                                         void* out) {
  const float s_dec = gscale[1];
  const int64_t nbc = C / 16;
  const int64_t nblk = R * nbc;
  for (int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; b < nblk;
       b += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = b / nbc, k = b - r * nbc;
    const uint2 q = *reinterpret_cast<const uint2*>(codes + r * (C / 2) + 8 * k);
    const float s = e4m3x2_to_float2((uint16_t)scales[b]).x;
    float v[16];
#pragma unroll
    for (int i = 0; i < 16; i++) {
      const uint32_t word = (i < 8) ? q.x : q.y;
      const uint32_t nib = (word >> (4 * (i & 7))) & 0xFu;
      v[i] = __fmul_rn(__fmul_rn(e2m1_value(nib), s), s_dec);
    }
    if (RHT) {
#pragma unroll
      for (int h = 1; h < 16; h <<= 1) {
#pragma unroll
        for (int i = 0; i < 16; i++) {
          if ((i & h) == 0) {
            const float x0 = v[i], x1 = v[i + h];
            v[i] = __fadd_rn(x0, x1);
            v[i + h] = __fsub_rn(x0, x1);
          }
        }
      }
#pragma unroll
      for (int i = 0; i < 16; i++) {
        const float t = __fmul_rn(0.25f, v[i]);
        v[i] = ((sign_mask >> i) & 1u) ? -t : t;
      }
    }
    if (BF16) {
      uint32_t w[8];
#pragma unroll
      for (int i = 0; i < 8; i++) {
        const __nv_bfloat162 p2 = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
        w[i] = *reinterpret_cast<const uint32_t*>(&p2);
      }
      uint4* o = reinterpret_cast<uint4*>(static_cast<uint16_t*>(out) + r * C + 16 * k);
      o[0] = make_uint4(w[0], w[1], w[2], w[3]);
      o[1] = make_uint4(w[4], w[5], w[6], w[7]);
    } else {
      float4* o = reinterpret_cast<float4*>(static_cast<float*>(out) + r * C + 16 * k);
#pragma unroll
      for (int i = 0; i < 4; i++) o[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
    }
  }
}

// Scale bytes [R][C] -> the 128 x 4 tiled layout of the tensor-core block-scaled GEMMs: one
// thread per 16-byte chunk of the output; chunk q of tile (tr, tc) holds rows 128 tr + q +
// 32 i (i = 0..3) of columns 4 tc .. 4 tc + 3, zero past R or C.
__global__ void __launch_bounds__(256) swizzle_scales_kernel(const uint8_t* __restrict__ s,
                                                             int64_t R, int64_t C,
                                                             uint8_t* __restrict__ out) {
  const int64_t tiles_c = (C + 3) / 4;
  const int64_t nchunks = ((R + 127) / 128) * tiles_c * 32;
  const bool words = (C & 3) == 0 && (reinterpret_cast<uintptr_t>(s) & 3) == 0;
  for (int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; k < nchunks;
       k += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = k >> 5, tr = t / tiles_c, tc = t - tr * tiles_c;
    const int q = (int)(k & 31);
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; i++) {
      const int64_t r = 128 * tr + 32 * i + q;
      w[i] = 0u;
      if (r < R) {
        if (words) {
          w[i] = *reinterpret_cast<const uint32_t*>(s + r * C + 4 * tc);
        } else {
#pragma unroll
          for (int j = 0; j < 4; j++)
            if (4 * tc + j < C) w[i] |= (uint32_t)s[r * C + 4 * tc + j] << (8 * j);
        }
      }
    }
    *reinterpret_cast<uint4*>(out + 16 * k) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

}  // namespace

cudaError_t launch_swizzle_scales(const uint8_t* scales, int64_t R, int64_t C, uint8_t* out,
                                  int grid, cudaStream_t s) {
  swizzle_scales_kernel<<<grid, 256, 0, s>>>(scales, R, C, out);
  return cudaGetLastError();
}

cudaError_t launch_amax_flat(const void* x, int64_t n_elems, float* out0, float* out1, int grid,
                             cudaStream_t s) {
  return launch_pdl(amax_flat_kernel, dim3(grid), dim3(256), 0, s,
                    reinterpret_cast<const uint4*>(x), n_elems / 8, out0, out1);
}

cudaError_t launch_dequantize(const uint8_t* codes, const uint8_t* scales, const float* gscale,
                              int64_t R, int64_t C, bool inverse_rht, uint32_t sign_mask,
                              bool out_bf16, void* out, int grid, cudaStream_t s) {
  if (inverse_rht && out_bf16)
    dequantize_kernel<true, true><<<grid, 256, 0, s>>>(codes, scales, gscale, R, C, sign_mask, out);
  else if (inverse_rht)
    dequantize_kernel<true, false><<<grid, 256, 0, s>>>(codes, scales, gscale, R, C, sign_mask, out);
  else if (out_bf16)
    dequantize_kernel<false, true><<<grid, 256, 0, s>>>(codes, scales, gscale, R, C, sign_mask, out);
  else
    dequantize_kernel<false, false><<<grid, 256, 0, s>>>(codes, scales, gscale, R, C, sign_mask, out);
  return cudaGetLastError();
}

}  // namespace nvfp4
