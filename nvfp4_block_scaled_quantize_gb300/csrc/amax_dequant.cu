// Amax kernels and dequantization.
//
// Page cited: "[nvfp4_training] Optimize CuteDSL kernels for NVFP4 training" (pytorch/ao pull
// request #4798): the amax pre-pass ("Optimization" item 5: "Linear RHT amax"; "Performance":
// grouped amax) and the dequantized reconstruction its "Correctness" section measures SQNR on.
#include "nvfp4_device.cuh"
#include "nvfp4_internal.h"

namespace nvfp4 {

namespace {

__device__ __forceinline__ uint4 ldg_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

__device__ __forceinline__ uint2 ldg_stream8(const uint2* p) {
  uint2 v;
  asm volatile("ld.global.nc.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
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

// Per-segment maxima over 16-row x 4-column items. Each item's 16 rows are one columnwise
// block of its segment (zero-padded past the segment's end); with RHT the transformed block's
// maximum goes to amax_col, the plain maximum to amax_row (and to amax_col without RHT).
template <bool RHT>
__global__ void __launch_bounds__(256, 2) amax_blocks_kernel(const AmaxArgs a) {
  __shared__ int32_t seg_start[kMaxSegments], seg_end[kMaxSegments], seg_blk0[kMaxSegments + 1];
  __shared__ uint32_t seg_max_row[kMaxSegments], seg_max_col[kMaxSegments];
  __shared__ int bad;
  const int tid = threadIdx.x, lane = tid & 31;
  const int E = a.segments;
  if (tid == 0) bad = 0;
  __syncthreads();
  for (int e = tid; e < E; e += blockDim.x) {
    int32_t start = (a.offsets == nullptr || e == 0) ? 0 : a.offsets[e - 1];
    int32_t end = (a.offsets == nullptr) ? (int32_t)a.rows : a.offsets[e];
    if (start < 0 || end < start || (int64_t)end > a.rows) bad = 1;
    seg_start[e] = start;
    seg_end[e] = end;
    seg_max_row[e] = 0u;
    seg_max_col[e] = 0u;
  }
  __syncthreads();
  if (bad) {
    if (blockIdx.x == 0 && tid == 0) atomicOr(a.status, 1u);  // NVFP4_DEVICE_BAD_OFFSETS
    return;
  }
  if (tid < 32) {
    int32_t base = 0;
    for (int c0 = 0; c0 < E; c0 += 32) {
      const int e = c0 + lane;
      const int32_t nb = (e < E) ? (seg_end[e] - seg_start[e] + 15) / 16 : 0;
      int32_t v = nb;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        int32_t u = __shfl_up_sync(0xFFFFFFFFu, v, d);
        if (lane >= d) v += u;
      }
      if (e < E) seg_blk0[e] = base + v - nb;
      base += __shfl_sync(0xFFFFFFFFu, v, 31);
    }
    if (lane == 0) seg_blk0[E] = base;
  }
  __syncthreads();

  const int64_t chunks = a.cols / 4;
  const int64_t items = (int64_t)seg_blk0[E] * chunks;
  const uint2* x = reinterpret_cast<const uint2*>(a.x);
  for (int64_t it = (int64_t)blockIdx.x * blockDim.x + tid; it < items;
       it += (int64_t)gridDim.x * blockDim.x) {
    const int32_t blk = (int32_t)(it / chunks);
    const int64_t ch = it - (int64_t)blk * chunks;
    int lo = 0, hi = E;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (seg_blk0[mid] <= blk) lo = mid; else hi = mid;
    }
    const int64_t r0 = seg_start[lo] + 16 * (int64_t)(blk - seg_blk0[lo]);
    const int64_t left = seg_end[lo] - r0;
    const int valid = left < 16 ? (int)left : 16;
    uint32_t w0[16], w1[16];
#pragma unroll
    for (int i = 0; i < 16; i++) {
      const uint2 v = (i < valid) ? ldg_stream8(x + (r0 + i) * chunks + ch) : make_uint2(0, 0);
      w0[i] = v.x;
      w1[i] = v.y;
    }
    // max.xorsign.abs tree: exact magnitudes, sign bits cleared at the end (finite inputs)
    uint32_t t[16];
#pragma unroll
    for (int i = 0; i < 16; i++) t[i] = hmax_abs2(w0[i], w1[i]);
#pragma unroll
    for (int h = 8; h >= 1; h >>= 1)
#pragma unroll
      for (int i = 0; i < h; i++) t[i] = hmax_abs2(t[i], t[i + h]);
    const uint32_t m = t[0] & 0x7FFF7FFFu;
    const uint32_t mr = max(m & 0xFFFFu, m >> 16);
    uint32_t mc = mr;
    if (RHT) {
      const uint32_t mt = vmax2(rht16_pair_absmax(w0, a.sign_mask), rht16_pair_absmax(w1, a.sign_mask));
      mc = max(mt & 0xFFFFu, mt >> 16);
    }
    if (mr) atomicMax(&seg_max_row[lo], mr);
    if (mc) atomicMax(&seg_max_col[lo], mc);
  }
  __syncthreads();
  for (int e = tid; e < E; e += blockDim.x) {
    if (a.amax_row && seg_max_row[e])
      atomicMax(reinterpret_cast<unsigned int*>(a.amax_row + (int64_t)e * a.stride_row),
                seg_max_row[e] << 16);
    if (a.amax_col && seg_max_col[e])
      atomicMax(reinterpret_cast<unsigned int*>(a.amax_col + (int64_t)e * a.stride_col),
                seg_max_col[e] << 16);
  }
}

// E2M1 code -> value (exact).
__device__ __forceinline__ float e2m1_value(uint32_t nib) {
  const uint32_t c = nib & 7u;
  const float mag = (c < 2u) ? 0.5f * (float)c
                             : __uint_as_float((((c >> 1) + 126u) << 23) | ((c & 1u) << 22));
  return (nib & 8u) ? -mag : mag;
}

// out[r][c] = (e2m1(code) * e4m3(scale)) * S_dec, one 16-element block per step.
__global__ void __launch_bounds__(256) dequantize_kernel(const uint8_t* __restrict__ codes,
                                                         const uint8_t* __restrict__ scales,
                                                         const float* __restrict__ gscale,
                                                         int64_t R, int64_t C, float* out) {
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
    float4* o = reinterpret_cast<float4*>(out + r * C + 16 * k);
#pragma unroll
    for (int i = 0; i < 4; i++) o[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
  }
}

}  // namespace

cudaError_t launch_amax_flat(const void* x, int64_t n_elems, float* out0, float* out1, int grid,
                             cudaStream_t s) {
  amax_flat_kernel<<<grid, 256, 0, s>>>(reinterpret_cast<const uint4*>(x), n_elems / 8, out0, out1);
  return cudaGetLastError();
}

cudaError_t launch_amax_blocks(bool rht, const AmaxArgs& args, int grid, cudaStream_t s) {
  if (rht) amax_blocks_kernel<true><<<grid, 256, 0, s>>>(args);
  else amax_blocks_kernel<false><<<grid, 256, 0, s>>>(args);
  return cudaGetLastError();
}

cudaError_t launch_dequantize(const uint8_t* codes, const uint8_t* scales, const float* gscale,
                              int64_t R, int64_t C, float* out, int grid, cudaStream_t s) {
  dequantize_kernel<<<grid, 256, 0, s>>>(codes, scales, gscale, R, C, out);
  return cudaGetLastError();
}

}  // namespace nvfp4
