// MX quantization (MXFP8 with E4M3 or E5M2 elements, MXFP4 with E2M1 elements) of BF16
// tensors: blocks of 32 elements along a row (rowwise) or a column (columnwise, written
// transposed) share one power-of-two scale stored as E8M0, and there is no tensor-wide scale.
// The page "CuTeDSL at Perplexity" (its Blackwell paragraph) names these formats beside NVFP4
// and their 32-element block maxima; the scale rule is the OCP Microscaling Formats v1.0
// conversion: exponent = floor(log2(block max)) - emax of the element format (8 for E4M3, 15
// for E5M2, 2 for E2M1), clamped below at -127; elements are x / 2^exponent rounded to
// nearest-even with saturation (cvt.rn.satfinite).
//
// No amax pass is needed, so this is one streaming pass. Each warp works alone on 32 x 128
// units of the tensor:
//   * a per-warp ring of kMxStages units, each two 32 x 64 TMA boxes (128-byte rows) loaded
//     with the 128-byte swizzle, completing on the stage's mbarrier (bounded waits);
//   * rowwise: lane l owns row l of the unit, four 32-element blocks of 16-byte chunks; the
//     swizzle puts the eight lanes of a shared-memory phase (rows l..l+7) on eight different
//     bank groups;
//   * columnwise: lane l owns four columns (8 bytes of a row of box l / 16), read down all 32
//     rows; a block is a lane-local column;
//   * the E8M0 exponent comes from the block maximum's exponent field (BF16 magnitudes order
//     like integers), the multiplier 2^-exponent is built from bits, and x * 2^-exponent is
//     exact, so a single cvt.rn.satfinite rounds each element once;
//   * FP8 codes leave as whole 32-byte sectors (st.global.v8.b32), FP4 codes as 16 bytes.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cuda_fp16.h>

#include <cstdint>

#include "nvfp4_device.cuh"
#include "nvfp4_internal.h"

namespace nvfp4 {
namespace {

constexpr uint64_t kMxWaitLimitNs = 2000000000ull;  // 2 s: no TMA load takes this long
constexpr int kBoxBytes = kMxUnitM * 128;            // one 32 x 64 BF16 box
constexpr int kUnitBytes = 2 * kBoxBytes;

template <int FMT>
struct MxFormat;
template <>
struct MxFormat<0> { static constexpr uint32_t emax = 8; };   // E4M3, largest 448 = 1.75 * 2^8
template <>
struct MxFormat<1> { static constexpr uint32_t emax = 15; };  // E5M2, largest 57344 = 1.75 * 2^15
template <>
struct MxFormat<2> { static constexpr uint32_t emax = 2; };   // E2M1, largest 6 = 1.5 * 2^2

// E8M0 code of a block from its largest BF16 magnitude m (sign cleared): the exponent field
// of m is floor(log2(max)) + 127 for normal values and 0 for zero and subnormals, which the
// clamp at -127 (code 0) covers.
template <int FMT>
__device__ __forceinline__ uint32_t mx_scale_code(uint32_t m) {
  const uint32_t e = (m >> 7) & 0xFFu;
  return e > MxFormat<FMT>::emax ? e - MxFormat<FMT>::emax : 0u;
}

// 2^-(code - 127) = 2^(127 - code) as a binary32 (a normal number for every code <= 253).
__device__ __forceinline__ float mx_multiplier(uint32_t code) {
  return __uint_as_float((254u - code) << 23);
}

// Two scaled values -> two FP8 codes, the first in the low byte.
template <int FMT>
__device__ __forceinline__ uint32_t fp8x2(float lo, float hi) {
  uint16_t d;
  if (FMT == 0)
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
  else
    asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
  return d;
}

template <int FMT>
__device__ __forceinline__ uint32_t fp8x4(uint64_t t01, uint64_t t23) {
  const float2 a = f2_unpack(t01), b = f2_unpack(t23);
  return fp8x2<FMT>(a.x, a.y) | (fp8x2<FMT>(b.x, b.y) << 16);
}

// 16-byte global store; p must be 16-byte aligned.
__device__ __forceinline__ void stg128(void* p, const uint4& v) {
  asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

// 32 elements given as 16 packed BF16 pairs (element 2i in the low half of w[i]), times mult,
// to codes: FP8 -> 32 bytes at p (32-byte aligned), FP4 -> 16 bytes (16-byte aligned).
template <int FMT>
__device__ __forceinline__ void store_block(uint8_t* p, const uint32_t (&w)[16], float mult) {
  const uint64_t m2 = f2_pack(mult, mult);
  if (FMT == 2) {
    uint32_t o[4];
#pragma unroll
    for (int q = 0; q < 4; q++)
      o[q] = e2m1x8_rn(f2_mul(f2_from_bf16x2(w[4 * q]), m2), f2_mul(f2_from_bf16x2(w[4 * q + 1]), m2),
                       f2_mul(f2_from_bf16x2(w[4 * q + 2]), m2),
                       f2_mul(f2_from_bf16x2(w[4 * q + 3]), m2));
    stg128(p, make_uint4(o[0], o[1], o[2], o[3]));
  } else {
    uint32_t o[8];
#pragma unroll
    for (int q = 0; q < 8; q++)
      o[q] = fp8x4<FMT>(f2_mul(f2_from_bf16x2(w[2 * q]), m2), f2_mul(f2_from_bf16x2(w[2 * q + 1]), m2));
    stg256(p, make_uint4(o[0], o[1], o[2], o[3]), make_uint4(o[4], o[5], o[6], o[7]));
  }
}

template <int FMT, bool ROW, bool COL>
__global__ void __launch_bounds__(32 * kMxWarps, 1) mx_quantize_kernel(const __grid_constant__ MxArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  // the 128-byte swizzle is a function of the shared address bits 7..9: boxes start on
  // 1024-byte boundaries so that it is row & 7 inside each box
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t* const gbase = smem_raw + (base - smem_u32(smem_raw));
  uint64_t* const full = reinterpret_cast<uint64_t*>(gbase + kMxWarps * kMxStages * kUnitBytes) +
                         warp * kMxStages;
  const uint32_t wstage = base + (uint32_t)(warp * kMxStages * kUnitBytes);

  const int64_t M = a.rows, N = a.cols;
  const int units_n = (int)((N + kMxUnitN - 1) / kMxUnitN);
  const int units = (int)((M + kMxUnitM - 1) / kMxUnitM) * units_n;
  const int gw = blockIdx.x * kMxWarps + warp;
  const int W = gridDim.x * kMxWarps;
  const int n_local = gw < units ? (units - gw + W - 1) / W : 0;
  if (n_local == 0) return;

  auto issue = [&](int i, int s) {
    const int u = gw + i * W;
    const int mt = u / units_n;
    const int n0 = (u - mt * units_n) * kMxUnitN;
    uint8_t* dst = gbase + (size_t)(warp * kMxStages + s) * kUnitBytes;
    // a second box wholly right of the tensor is not loaded: nothing of it is stored
    const bool two = (int64_t)n0 + 64 < N;
    mbar_expect_tx(&full[s], two ? kUnitBytes : kBoxBytes);
    tma_load_2d(dst, &a.tmap, n0, mt * kMxUnitM, &full[s]);
    if (two) tma_load_2d(dst + kBoxBytes, &a.tmap, n0 + 64, mt * kMxUnitM, &full[s]);
  };
  if (lane == 0) {
    prefetch_tensormap(&a.tmap);
    for (int s = 0; s < kMxStages; s++) mbar_init(&full[s], 1);
    fence_barrier_init();
    for (int s = 0; s < kMxStages && s < n_local; s++) issue(s, s);
  }
  __syncwarp();

  // columnwise lane geometry: box lane / 16, byte 8 (lane % 16) of each 128-byte row
  const int cbox = lane >> 4;
  const int cg = lane & 15;
  uint32_t coff[8];  // swizzled offset of the lane's 8 bytes in a row r with r & 7 == k
#pragma unroll
  for (int k = 0; k < 8; k++) coff[k] = (uint32_t)((((cg >> 1) ^ k) << 4) | ((cg & 1) << 3));
  // rowwise: row `lane`; chunk c of the row sits at (c ^ (lane & 7)) * 16
  const uint32_t rsw = (uint32_t)(lane & 7) << 4;

  for (int i = 0; i < n_local; i++) {
    const int s = i % kMxStages;
    if (!mbar_wait_bounded(&full[s], (uint32_t)(i / kMxStages) & 1u, kMxWaitLimitNs)) {
      // record the timeout, wait (bounded) for the loads still in flight, leave
      if (lane == 0) {
        atomicOr(a.status, 2u);  // NVFP4_DEVICE_TIMEOUT
        for (int j = i; j < n_local && j < i + kMxStages; j++)
          mbar_wait_bounded(&full[j % kMxStages], (uint32_t)(j / kMxStages) & 1u, kMxWaitLimitNs);
      }
      __syncwarp();
      return;
    }
    const int u = gw + i * W;
    const int mt = u / units_n;
    const int64_t m0 = (int64_t)mt * kMxUnitM;
    const int64_t n0 = (int64_t)(u - mt * units_n) * kMxUnitN;
    const uint32_t stage = wstage + (uint32_t)(s * kUnitBytes);

    if (ROW) {
      const int64_t row = m0 + lane;
      uint32_t codes = 0u;
#pragma unroll
      for (int b = 0; b < 4; b++) {  // block b: box b / 2, chunks 4 (b % 2) .. + 3
        const uint32_t rowaddr = stage + (uint32_t)((b >> 1) * kBoxBytes + lane * 128);
        uint32_t w[16];
#pragma unroll
        for (int k = 0; k < 4; k++) {
          const uint4 q = lds128(rowaddr + ((((uint32_t)(4 * (b & 1) + k)) << 4) ^ rsw));
          w[4 * k] = q.x; w[4 * k + 1] = q.y; w[4 * k + 2] = q.z; w[4 * k + 3] = q.w;
        }
        uint32_t t[8];
#pragma unroll
        for (int k = 0; k < 8; k++) t[k] = hmax_abs2(w[2 * k], w[2 * k + 1]);
#pragma unroll
        for (int h = 4; h >= 1; h >>= 1)
#pragma unroll
          for (int k = 0; k < h; k++) t[k] = hmax_abs2(t[k], t[k + h]);
        const uint32_t m = t[0] & 0x7FFF7FFFu;
        const uint32_t code = mx_scale_code<FMT>(max(m & 0xFFFFu, m >> 16));
        codes |= code << (8 * b);
        const int64_t col = n0 + 32 * b;
        if (row < M && col < N) {
          uint8_t* p = a.row_codes + (FMT == 2 ? row * (N / 2) + col / 2 : row * N + col);
          store_block<FMT>(p, w, mx_multiplier(code));
        }
      }
      if (row < M) {
        uint8_t* sp = a.row_scales + row * (N / 32) + n0 / 32;
        const int64_t nb = (N - n0) / 32;  // blocks of this unit inside the tensor
        if (nb >= 4 && ((N / 32) & 3) == 0) {
          *reinterpret_cast<uint32_t*>(sp) = codes;
        } else {
#pragma unroll
          for (int b = 0; b < 4; b++)
            if (b < nb) sp[b] = (uint8_t)(codes >> (8 * b));
        }
      }
    }

    if (COL) {
      // lane's columns n0 + 64 cbox + 4 cg + j, j = 0..3; v[r] = their row-r elements
      const uint32_t boxaddr = stage + (uint32_t)(cbox * kBoxBytes);
      uint2 v[32];
#pragma unroll
      for (int r = 0; r < 32; r++) {
        uint2 q;
        asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];"
                     : "=r"(q.x), "=r"(q.y)
                     : "r"(boxaddr + (uint32_t)(r * 128) + coff[r & 7]));
        v[r] = q;
      }
      uint32_t mx = 0u, my = 0u;
#pragma unroll
      for (int r = 0; r < 32; r++) {
        mx = hmax_abs2(mx, v[r].x);
        my = hmax_abs2(my, v[r].y);
      }
      mx &= 0x7FFF7FFFu;
      my &= 0x7FFF7FFFu;
      const uint32_t code[4] = {mx_scale_code<FMT>(mx & 0xFFFFu), mx_scale_code<FMT>(mx >> 16),
                                mx_scale_code<FMT>(my & 0xFFFFu), mx_scale_code<FMT>(my >> 16)};
      const int64_t ncol0 = n0 + 64 * cbox + 4 * cg;
      if (ncol0 < N) {  // N % 8 == 0: the lane's four columns are all inside or all outside
#pragma unroll
        for (int j = 0; j < 4; j++) {
          // column j: the low (j even) or high half of word x (j < 2) or y
          uint32_t w[16];
#pragma unroll
          for (int r = 0; r < 32; r += 2) {
            const uint32_t a0 = j < 2 ? v[r].x : v[r].y;
            const uint32_t a1 = j < 2 ? v[r + 1].x : v[r + 1].y;
            // rows r, r + 1 of column j as one packed BF16 pair (row r in the low half)
            w[r / 2] = (j & 1) ? __byte_perm(a0, a1, 0x7632) : __byte_perm(a0, a1, 0x5410);
          }
          const int64_t n = ncol0 + j;
          uint8_t* p = a.col_codes + (FMT == 2 ? n * (M / 2) + m0 / 2 : n * M + m0);
          store_block<FMT>(p, w, mx_multiplier(code[j]));
          a.col_scales[n * (M / 32) + m0 / 32] = (uint8_t)code[j];
        }
      }
    }

    // every lane is done with the stage: refill it
    __syncwarp();
    if (lane == 0 && i + kMxStages < n_local) {
      fence_proxy_async();
      issue(i + kMxStages, s);
    }
  }
}

template <int FMT, bool ROW, bool COL>
cudaError_t launch_t(const MxArgs& args, int grid, cudaStream_t s) {
  mx_quantize_kernel<FMT, ROW, COL><<<grid, 32 * kMxWarps, kMxSmemBytes, s>>>(args);
  return cudaGetLastError();
}

template <int FMT, bool ROW, bool COL>
cudaError_t prepare_t() {
  return cudaFuncSetAttribute(mx_quantize_kernel<FMT, ROW, COL>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, kMxSmemBytes);
}

template <int FMT>
cudaError_t launch_f(bool row, bool col, const MxArgs& args, int grid, cudaStream_t s) {
  if (row && col) return launch_t<FMT, true, true>(args, grid, s);
  if (row) return launch_t<FMT, true, false>(args, grid, s);
  return launch_t<FMT, false, true>(args, grid, s);
}

template <int FMT>
cudaError_t prepare_f() {
  cudaError_t e = cudaSuccess, r;
  if ((r = prepare_t<FMT, true, true>()) != cudaSuccess) e = r;
  if ((r = prepare_t<FMT, true, false>()) != cudaSuccess) e = r;
  if ((r = prepare_t<FMT, false, true>()) != cudaSuccess) e = r;
  return e;
}

// FP8 pair (first element in the low byte) -> two floats (exact, through f16x2).
template <int FMT>
__device__ __forceinline__ float2 fp8x2_to_float2(uint16_t c) {
  uint32_t h2;
  if (FMT == 0)
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(c));
  else
    asm("cvt.rn.f16x2.e5m2x2 %0, %1;" : "=r"(h2) : "h"(c));
  return make_float2(__half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu))),
                     __half2float(__ushort_as_half((unsigned short)(h2 >> 16))));
}

// E2M1 code -> value (exact).
__device__ __forceinline__ float e2m1_to_float(uint32_t nib) {
  const uint32_t c = nib & 7u;
  const float mag = (c < 2u) ? 0.5f * (float)c
                             : __uint_as_float((((c >> 1) + 126u) << 23) | ((c & 1u) << 22));
  return (nib & 8u) ? -mag : mag;
}

// out[r][c] = element(code) * 2^(scale - 127), one 32-element block per step; the product is
// rounded once (it is exact unless it leaves binary32's range).
template <int FMT>
__global__ void __launch_bounds__(256) mx_dequantize_kernel(const uint8_t* __restrict__ codes,
                                                            const uint8_t* __restrict__ scales,
                                                            int64_t R, int64_t C, float* out) {
  const int64_t nbc = C / 32;
  const int64_t nblk = R * nbc;
  for (int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; b < nblk;
       b += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = b / nbc, k = b - r * nbc;
    const uint32_t sc = scales[b];
    const float X = sc == 0u ? __uint_as_float(0x00400000u)  // 2^-127, a subnormal
                             : (sc == 255u ? __uint_as_float(0x7FC00000u) : __uint_as_float(sc << 23));
    float v[32];
    if (FMT == 2) {
      const uint4 q = *reinterpret_cast<const uint4*>(codes + r * (C / 2) + 16 * k);
      const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int i = 0; i < 32; i++) v[i] = __fmul_rn(e2m1_to_float(w[i >> 3] >> (4 * (i & 7))), X);
    } else {
      const uint4* p = reinterpret_cast<const uint4*>(codes + r * C + 32 * k);
      const uint4 q0 = p[0], q1 = p[1];
      const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
      for (int i = 0; i < 16; i++) {
        const float2 f = fp8x2_to_float2<FMT>((uint16_t)(w[i >> 1] >> (16 * (i & 1))));
        v[2 * i] = __fmul_rn(f.x, X);
        v[2 * i + 1] = __fmul_rn(f.y, X);
      }
    }
    float4* o = reinterpret_cast<float4*>(out + r * C + 32 * k);
#pragma unroll
    for (int i = 0; i < 8; i++) o[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
  }
}

}  // namespace

cudaError_t launch_mx_dequantize(int fmt, const uint8_t* codes, const uint8_t* scales, int64_t R,
                                 int64_t C, float* out, int grid, cudaStream_t s) {
  if (fmt == 0) mx_dequantize_kernel<0><<<grid, 256, 0, s>>>(codes, scales, R, C, out);
  else if (fmt == 1) mx_dequantize_kernel<1><<<grid, 256, 0, s>>>(codes, scales, R, C, out);
  else mx_dequantize_kernel<2><<<grid, 256, 0, s>>>(codes, scales, R, C, out);
  return cudaGetLastError();
}

static_assert(kMxSmemBytes >= kMxWarps * kMxStages * kUnitBytes + kMxWarps * kMxStages * 8 + 1024,
              "MX shared memory: stages, barriers and the 1024-byte alignment slack");

cudaError_t launch_mx_quantize(int fmt, bool row, bool col, const MxArgs& args, int grid,
                               cudaStream_t s) {
  if (fmt == 0) return launch_f<0>(row, col, args, grid, s);
  if (fmt == 1) return launch_f<1>(row, col, args, grid, s);
  return launch_f<2>(row, col, args, grid, s);
}

cudaError_t prepare_mx_kernels() {
  cudaError_t e = cudaSuccess, r;
  if ((r = prepare_f<0>()) != cudaSuccess) e = r;
  if ((r = prepare_f<1>()) != cudaSuccess) e = r;
  if ((r = prepare_f<2>()) != cudaSuccess) e = r;
  return e;
}

}  // namespace nvfp4
