// Test-only probe library (not part of libnvfp4):
//   * runs single instructions, and the quantizer's x/6 routine, on chosen inputs so that the
//     tests can compare their outputs with the oracle and with IEEE division; the conversion
//     kernels are bare inline PTX, so that what they pin is the instruction itself, not the
//     library's use of it;
//   * a busy kernel that holds SMs for a bounded time, so that a test can run the
//     single-launch quantize while part of the GPU is taken by another stream's work.
//
// Page cited: "[nvfp4_training] Optimize CuteDSL kernels for NVFP4 training" (pytorch/ao pull
// request #4798), "Optimization" items 1 and 3: the packed cvt.rn.satfinite.e2m1x2.f32 and
// cvt.rs.satfinite.e2m1x4.f32 conversions are the method's rounding steps.
//
// Every kernel is a grid-stride loop bounded by its element count; host entry points
// allocate, copy, launch, copy back and free, and return the first CUDA error (0 = success).
#include <cuda_runtime.h>

#include <cstdint>

#include "nvfp4_device.cuh"

namespace {

// Element 4k+i of t -> nibble i of out[k]: operands {a, b, e, f} are elements 3, 2, 1, 0.
__global__ void cvt_rs_e2m1x4_kernel(const float* t, const uint32_t* w, uint16_t* out,
                                     int64_t n) {
  for (int64_t k = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; k < n;
       k += (int64_t)gridDim.x * blockDim.x) {
    uint16_t d;
    asm volatile("cvt.rs.satfinite.e2m1x4.f32 %0, {%1, %2, %3, %4}, %5;"
                 : "=h"(d)
                 : "f"(t[4 * k + 3]), "f"(t[4 * k + 2]), "f"(t[4 * k + 1]), "f"(t[4 * k]),
                   "r"(w[k]));
    out[k] = d;
  }
}

// a[k] -> high nibble, b[k] -> low nibble of out[k].
__global__ void cvt_rn_e2m1x2_kernel(const float* a, const float* b, uint8_t* out, int64_t n) {
  for (int64_t k = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; k < n;
       k += (int64_t)gridDim.x * blockDim.x) {
    uint16_t d;
    asm volatile("{\n\t.reg .b8 q;\n\t"
                 "cvt.rn.satfinite.e2m1x2.f32 q, %1, %2;\n\t"
                 "cvt.u16.u8 %0, q;\n\t}"
                 : "=h"(d)
                 : "f"(a[k]), "f"(b[k]));
    out[k] = (uint8_t)d;
  }
}

// Over the bit patterns [lo, hi) of non-negative finite binary32 values x: compares both lanes
// of the quantizer's div6x2 with __fdiv_rn(x, 6). counts: [0] values checked, [1] mismatches,
// [2] mismatches at BF16 values (low 16 bits zero), [3] mismatches whose IEEE quotient is
// normal, [4] mismatches not of the form x = K * 2^-149 with K < 2^24 and K = 9 (mod 12), the
// only values whose sixth is an exact tie between two subnormals with an odd lower neighbour.
// first[0]: the smallest mismatching pattern (0xFFFFFFFF when none).
__global__ void div6_check_kernel(uint32_t lo, uint32_t hi, unsigned long long* counts,
                                  uint32_t* first) {
  unsigned long long checked = 0, bad = 0, bad_bf16 = 0, bad_normal = 0, bad_other = 0;
  uint32_t first_bad = 0xFFFFFFFFu;
  const uint64_t span = (uint64_t)hi - lo;
  for (uint64_t k = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; k < span;
       k += (uint64_t)gridDim.x * blockDim.x) {
    const uint32_t bits = lo + (uint32_t)k;
    const float x = __uint_as_float(bits);
    if (!(x <= 3.402823466e38f)) continue;  // NaN or infinity
    const float ref = __fdiv_rn(x, 6.0f);
    // both lanes: x in one, a different value (x's bits reversed within the finite range) in
    // the other, so that a lane mix-up shows too
    const uint32_t other_bits = (__brev(bits) >> 1) & 0x7F7FFFFFu;
    const float other = __uint_as_float(other_bits);
    const float2 q = nvfp4::f2_unpack(nvfp4::div6x2(nvfp4::f2_pack(x, other)));
    const float2 p = nvfp4::f2_unpack(nvfp4::div6x2(nvfp4::f2_pack(other, x)));
    const bool ok = __float_as_uint(q.x) == __float_as_uint(ref) &&
                    __float_as_uint(p.y) == __float_as_uint(ref) &&
                    __float_as_uint(q.y) == __float_as_uint(p.x);
    checked++;
    if (!ok) {
      bad++;
      if ((bits & 0xFFFFu) == 0u) bad_bf16++;
      if (ref >= 1.17549435e-38f) bad_normal++;
      // below 2^-125 a binary32 is K * 2^-149 with K = its bit pattern's value as an integer
      // (subnormals) or 2^23 + mantissa (the lowest normal binade): K < 2^24 either way
      if (!(bits < (1u << 24) && bits % 12u == 9u)) bad_other++;
      first_bad = min(first_bad, bits);
    }
  }
  atomicAdd(&counts[0], checked);
  if (bad) {
    atomicAdd(&counts[1], bad);
    atomicAdd(&counts[2], bad_bf16);
    atomicAdd(&counts[3], bad_normal);
    atomicAdd(&counts[4], bad_other);
    atomicMin(&first[0], first_bad);
  }
}

// Each CTA (one warp) counts itself in *started, then spins until `ns` nanoseconds of global
// time have passed since it started: a bounded wait that keeps its SM's registers taken.
__global__ void busy_kernel(unsigned int* started, uint64_t ns) {
  uint64_t t0, t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  if (threadIdx.x == 0) atomicAdd(started, 1u);
  do {
    __nanosleep(1000);
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  } while (t - t0 < ns);
}

int grid_for(int64_t n) {
  int64_t g = (n + 255) / 256;
  if (g > 4096) g = 4096;
  return g < 1 ? 1 : (int)g;
}

}  // namespace

extern "C" int probe_cvt_rs_e2m1x4(const float* t, const uint32_t* w, int64_t n_words,
                                   uint16_t* out) {
  float* dt = nullptr;
  uint32_t* dw = nullptr;
  uint16_t* dout = nullptr;
  cudaError_t e = cudaMalloc(&dt, 16 * n_words);
  if (e == cudaSuccess) e = cudaMalloc(&dw, 4 * n_words);
  if (e == cudaSuccess) e = cudaMalloc(&dout, 2 * n_words);
  if (e == cudaSuccess) e = cudaMemcpy(dt, t, 16 * n_words, cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemcpy(dw, w, 4 * n_words, cudaMemcpyHostToDevice);
  if (e == cudaSuccess) {
    cvt_rs_e2m1x4_kernel<<<grid_for(n_words), 256>>>(dt, dw, dout, n_words);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) e = cudaMemcpy(out, dout, 2 * n_words, cudaMemcpyDeviceToHost);
  cudaFree(dt);
  cudaFree(dw);
  cudaFree(dout);
  return (int)e;
}

extern "C" int probe_cvt_rn_e2m1x2(const float* a, const float* b, int64_t n, uint8_t* out) {
  float *da = nullptr, *db = nullptr;
  uint8_t* dout = nullptr;
  cudaError_t e = cudaMalloc(&da, 4 * n);
  if (e == cudaSuccess) e = cudaMalloc(&db, 4 * n);
  if (e == cudaSuccess) e = cudaMalloc(&dout, n);
  if (e == cudaSuccess) e = cudaMemcpy(da, a, 4 * n, cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemcpy(db, b, 4 * n, cudaMemcpyHostToDevice);
  if (e == cudaSuccess) {
    cvt_rn_e2m1x2_kernel<<<grid_for(n), 256>>>(da, db, dout, n);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) e = cudaMemcpy(out, dout, n, cudaMemcpyDeviceToHost);
  cudaFree(da);
  cudaFree(db);
  cudaFree(dout);
  return (int)e;
}

// counts[5] and first[1] as div6_check_kernel; lo <= hi <= 0x80000000.
extern "C" int probe_div6(uint32_t lo, uint32_t hi, unsigned long long* counts, uint32_t* first) {
  if (lo > hi || hi > 0x80000000u) return (int)cudaErrorInvalidValue;
  unsigned long long* dc = nullptr;
  uint32_t* df = nullptr;
  cudaError_t e = cudaMalloc(&dc, 5 * sizeof(unsigned long long));
  if (e == cudaSuccess) e = cudaMalloc(&df, 4);
  if (e == cudaSuccess) e = cudaMemset(dc, 0, 5 * sizeof(unsigned long long));
  if (e == cudaSuccess) e = cudaMemset(df, 0xFF, 4);
  if (e == cudaSuccess) {
    div6_check_kernel<<<152 * 16, 256>>>(lo, hi, dc, df);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) e = cudaMemcpy(counts, dc, 5 * sizeof(unsigned long long), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemcpy(first, df, 4, cudaMemcpyDeviceToHost);
  cudaFree(dc);
  cudaFree(df);
  return (int)e;
}

// Launch busy_kernel with `ctas` one-warp CTAs on `stream` (asynchronous); *started (device,
// zeroed here) counts the CTAs that have begun. Each CTA takes 48 KiB of shared memory, so
// that a quantize CTA (about 190 KiB) cannot share an SM with it.
extern "C" int probe_busy_launch(int ctas, uint64_t ns, unsigned int* started, void* stream) {
  if (ctas < 1 || ctas > 4096 || ns > 10000000000ull) return (int)cudaErrorInvalidValue;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(started, 0, sizeof(unsigned int), s);
  if (e == cudaSuccess) {
    busy_kernel<<<ctas, 32, 48 * 1024, s>>>(started, ns);
    e = cudaGetLastError();
  }
  return (int)e;
}
