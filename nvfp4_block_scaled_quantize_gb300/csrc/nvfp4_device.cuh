// Device primitives of the NVFP4 quantizer (sm_103a): BF16 unpacking, block maxima, the
// two-level scale arithmetic, E2M1 conversion with round-to-nearest-even or stochastic
// rounding, Philox4x32-10, the 16-point Hadamard butterflies, and TMA/mbarrier plumbing.
//
// Page cited: "[nvfp4_training] Optimize CuteDSL kernels for NVFP4 training" (pytorch/ao pull
// request #4798), by section. Every float operation is an explicit IEEE round-to-nearest
// intrinsic or PTX instruction, so that no multiply-add is contracted and the results equal
// the scalar binary32 statement of the method bit for bit.
#pragma once

#include <cfloat>
#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace nvfp4 {

// ------------------------------------------------------------------------------------------
// BF16 pairs. A 32-bit word holds two BF16 values: the lower-addressed (even) element in the
// low half. BF16 is the upper half of a binary32, so widening is a shift or a mask
// ([PR4798] "Optimization" item 6).
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Magnitudes of both halves (sign bits cleared). As unsigned 16-bit integers, BF16
// magnitudes order exactly like the values they encode (finite inputs).
__device__ __forceinline__ uint32_t abs2(uint32_t w) { return w & 0x7FFF7FFFu; }
__device__ __forceinline__ uint32_t vmax2(uint32_t a, uint32_t b) { return __vmaxu2(a, b); }
// Larger of the two magnitudes of a packed pair, as a float.
__device__ __forceinline__ float pair_max(uint32_t m) {
  return __uint_as_float(max(m & 0xFFFFu, m >> 16) << 16);
}
__device__ __forceinline__ float mag_lo(uint32_t m) { return __uint_as_float(m << 16); }
__device__ __forceinline__ float mag_hi(uint32_t m) { return __uint_as_float(m & 0xFFFF0000u); }

// ------------------------------------------------------------------------------------------
// Packed binary32 pairs (f32x2). One instruction handles both lanes of a 64-bit register
// pair, each lane rounded to nearest-even exactly as the scalar instruction
// ([PR4798] "Optimization" item 1: packed mul.f32x2).
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
  return d;
}
__device__ __forceinline__ float2 f2_unpack(uint64_t d) {
  float lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(d));
  return make_float2(lo, hi);
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
// Per 16-bit half: max(|a|, |b|) of BF16 values, exact; the sign bits of the result are
// meaningless (max.xorsign.abs) and are cleared once at the end of a chain.
__device__ __forceinline__ uint32_t hmax_abs2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
// A packed BF16 pair widened to a packed binary32 pair (low half -> low lane).
__device__ __forceinline__ uint64_t f2_from_bf16x2(uint32_t w) {
  return f2_pack(bf16_lo(w), bf16_hi(w));
}
// A packed BF16 pair widened to binary32 with the sign of both halves flipped when f (0 or
// 0x80000000) is set: the low half by one multiply-add (w * 2^16 + f, the addition of bit 31
// being its flip), the high half by one three-input logic operation.
__device__ __forceinline__ uint64_t f2_from_bf16x2_flip(uint32_t w, uint32_t f) {
  return f2_pack(__uint_as_float(w * 65536u + f), __uint_as_float((w & 0xFFFF0000u) ^ f));
}

// ------------------------------------------------------------------------------------------
// Scales
// ------------------------------------------------------------------------------------------

// Per-tensor global scale: S_enc = 2688 / amax (448 * 6), 1 when amax == 0, FLT_MAX when the
// quotient overflows; S_dec = 1 / S_enc ([PR4798] "Fast math": the per-tensor
// global_decode_scale).
__device__ __forceinline__ void global_scale(float amax, float& s_enc, float& s_dec) {
  float enc = (amax == 0.0f) ? 1.0f : __fdiv_rn(2688.0f, amax);
  enc = fminf(enc, FLT_MAX);
  s_enc = enc;
  s_dec = __frcp_rn(enc);
}

// x / 6 correctly rounded for both lanes of a packed pair: the product by the rounded
// reciprocal of 6, corrected by one remainder step (Markstein's correction for a divisor known
// in advance; Brisebarre, Muller and Raina, "Accelerating correctly rounded floating-point
// division when the divisor is known in advance", IEEE Trans. Computers 53(8), 2004). The
// remainder x - 6q is exact (one fused multiply-add) and the corrected quotient equals IEEE
// division by 6 on every non-negative binary32 whose quotient is normal; a quotient in the
// subnormal range that lies exactly halfway between two subnormals can round the other way.
// No BF16 value is such a case (a BF16 subnormal is an even multiple of 2^-149, so its sixth
// is never an odd multiple of 2^-150), so the block maxima of BF16 blocks are always divided
// exactly; the fast-math FP32 transform's maxima are outside that guarantee only at quotients
// below 2^-126. A GPU test checks both statements over every non-negative finite binary32.
__device__ __forceinline__ uint64_t div6x2(uint64_t x) {
  const uint64_t c = f2_pack(0.16666667163372039794921875f, 0.16666667163372039794921875f);
  const uint64_t neg6 = f2_pack(-6.0f, -6.0f);
  const uint64_t q = f2_mul(x, c);
  const uint64_t r = f2_fma(q, neg6, x);
  return f2_fma(r, c, q);
}

// Two E4M3 block scales from two block maxima: s = E4M3_rn_satfinite((bamax / 6) * S_enc),
// with x / 6 as in div6x2. Returns the pair as a 16-bit word, `lo` in the low byte.
__device__ __forceinline__ uint16_t block_scales2(float bamax_lo, float bamax_hi, float s_enc) {
  const float2 s = f2_unpack(f2_mul(div6x2(f2_pack(bamax_lo, bamax_hi)), f2_pack(s_enc, s_enc)));
  uint16_t d;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(s.y), "f"(s.x));
  return d;
}

// E4M3 pair -> two floats (exact): .x from the low byte, .y from the high byte.
__device__ __forceinline__ float2 e4m3x2_to_float2(uint16_t s) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(s));
  return make_float2(__half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu))),
                     __half2float(__ushort_as_half((unsigned short)(h2 >> 16))));
}

// Element multiplier r = 1 / (float(s) * S_dec), correctly rounded; 0 when the product is 0;
// FLT_MAX when the reciprocal overflows ([PR4798] "Fast math": exact mode takes div_rn of
// pvscale_fp8 * global_decode_scale).
__device__ __forceinline__ float element_multiplier(float s, float s_dec) {
  float p = __fmul_rn(s, s_dec);
  float r = fminf(__frcp_rn(p), FLT_MAX);
  return (p == 0.0f) ? 0.0f : r;
}

// rht16_pair without the BF16 round-through (the fast-math variant): x[i] receives the FP32
// pair 0.25 * (H16 (d . v))_i of the two columns.
__device__ __forceinline__ void rht16_pair_f32(const uint32_t (&w)[16], const uint32_t (&flip)[16],
                                               uint64_t (&x)[16]) {
#pragma unroll
  for (int i = 0; i < 16; i++) x[i] = f2_from_bf16x2_flip(w[i], flip[i]);
#pragma unroll
  for (int h = 1; h < 16; h <<= 1) {
#pragma unroll
    for (int i = 0; i < 16; i++) {
      if ((i & h) == 0) {
        uint64_t a = x[i], b = x[i + h];
        x[i] = f2_add(a, b);
        x[i + h] = f2_sub(a, b);
      }
    }
  }
  const uint64_t quarter = f2_pack(0.25f, 0.25f);
#pragma unroll
  for (int i = 0; i < 16; i++) x[i] = f2_mul(x[i], quarter);
}

// The fast-math element multiplier: the hardware's approximate reciprocal of s * S_dec (flush
// to zero), 0 for a zero product, at most FLT_MAX ([PR4798] "Fast math": rcp.approx.ftz).
__device__ __forceinline__ float element_multiplier_fast(float s, float s_dec) {
  const float p = __fmul_rn(s, s_dec);
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(p));
  return (p == 0.0f) ? 0.0f : fminf(r, FLT_MAX);
}

// Largest |bf16(0.25 * (H16 (d . v))_i)| over the 16 outputs of each of the two columns of w
// (rht16_pair's outputs), as BF16 magnitude bits (column 0 in the low half). Scaling by 0.25
// and rounding to BF16 are both monotone, so the maximum of the rounded outputs is the rounded
// maximum of the unrounded ones: the maximum is taken in FP32 straight after the last
// butterfly stage, and only it is scaled and rounded.
__device__ __forceinline__ uint32_t rht16_pair_absmax(const uint32_t (&w)[16], const uint32_t (&flip)[16]) {
  uint64_t x[16];
#pragma unroll
  for (int i = 0; i < 16; i++) x[i] = f2_from_bf16x2_flip(w[i], flip[i]);
#pragma unroll
  for (int h = 1; h < 8; h <<= 1) {
#pragma unroll
    for (int i = 0; i < 16; i++) {
      if ((i & h) == 0) {
        uint64_t a = x[i], b = x[i + h];
        x[i] = f2_add(a, b);
        x[i + h] = f2_sub(a, b);
      }
    }
  }
  float m0 = 0.0f, m1 = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; i++) {
    const float2 s = f2_unpack(f2_add(x[i], x[i + 8]));
    const float2 d = f2_unpack(f2_sub(x[i], x[i + 8]));
    m0 = fmaxf(m0, fmaxf(fabsf(s.x), fabsf(d.x)));
    m1 = fmaxf(m1, fmaxf(fabsf(s.y), fabsf(d.y)));
  }
  const float2 q = f2_unpack(f2_mul(f2_pack(m0, m1), f2_pack(0.25f, 0.25f)));
  uint32_t packed;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(packed) : "f"(q.y), "f"(q.x));
  return packed & 0x7FFF7FFFu;
}

// ------------------------------------------------------------------------------------------
// E2M1 conversion. Codes are packed two per byte with the even element in the low nibble.
// ------------------------------------------------------------------------------------------

// Eight scaled values -> eight codes, element 0 in bits 3:0 ([PR4798] "Optimization" item 1:
// packed mul then cvt.rn.satfinite.e2m1x2.f32; that instruction puts its first operand in
// the high nibble).
__device__ __forceinline__ uint32_t e2m1x8_rn(uint64_t t01, uint64_t t23, uint64_t t45,
                                              uint64_t t67) {
  float2 a = f2_unpack(t01), b = f2_unpack(t23), c = f2_unpack(t45), d = f2_unpack(t67);
  uint32_t out;
  asm("{\n\t.reg .b8 q0, q1, q2, q3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q3, %8, %7;\n\t"
      "mov.b32 %0, {q0, q1, q2, q3};\n\t}"
      : "=r"(out)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y), "f"(d.x), "f"(d.y));
  return out;
}

// Eight scaled values -> eight codes by stochastic rounding: elements 0..3 with random word
// w0 and 4..7 with w1, each group one cvt.rs.satfinite.e2m1x4.f32 whose operands (a, b, e, f)
// are elements (3, 2, 1, 0) so that element 0 lands in the low nibble ([PR4798]
// "Optimization" item 3: the SR multiply and clamp fused into the convert).
__device__ __forceinline__ uint32_t e2m1x8_rs(uint64_t t01, uint64_t t23, uint64_t t45,
                                              uint64_t t67, uint32_t w0, uint32_t w1) {
  float2 a = f2_unpack(t01), b = f2_unpack(t23), c = f2_unpack(t45), d = f2_unpack(t67);
  uint16_t lo, hi;
  asm("cvt.rs.satfinite.e2m1x4.f32 %0, {%1, %2, %3, %4}, %5;"
      : "=h"(lo) : "f"(b.y), "f"(b.x), "f"(a.y), "f"(a.x), "r"(w0));
  asm("cvt.rs.satfinite.e2m1x4.f32 %0, {%1, %2, %3, %4}, %5;"
      : "=h"(hi) : "f"(d.y), "f"(d.x), "f"(c.y), "f"(c.x), "r"(w1));
  return (uint32_t)lo | ((uint32_t)hi << 16);
}

// Eight elements given as four packed BF16 pairs, times r, to codes. sr selects stochastic
// rounding with words (w0, w1).
__device__ __forceinline__ uint32_t quantize8(uint32_t p0, uint32_t p1, uint32_t p2, uint32_t p3,
                                              float r, bool sr, uint32_t w0, uint32_t w1) {
  uint64_t rr = f2_pack(r, r);
  uint64_t t01 = f2_mul(f2_from_bf16x2(p0), rr);
  uint64_t t23 = f2_mul(f2_from_bf16x2(p1), rr);
  uint64_t t45 = f2_mul(f2_from_bf16x2(p2), rr);
  uint64_t t67 = f2_mul(f2_from_bf16x2(p3), rr);
  return sr ? e2m1x8_rs(t01, t23, t45, t67, w0, w1) : e2m1x8_rn(t01, t23, t45, t67);
}

// One column of eight elements taken from the low (hi = false) or high halves of eight
// packed words, times r, to codes.
__device__ __forceinline__ uint32_t quantize8_column(const uint32_t* w, bool hi, float r,
                                                     bool sr, uint32_t w0, uint32_t w1) {
  uint64_t rr = f2_pack(r, r);
  uint64_t t[4];
#pragma unroll
  for (int k = 0; k < 4; k++) {
    float e0 = hi ? bf16_hi(w[2 * k]) : bf16_lo(w[2 * k]);
    float e1 = hi ? bf16_hi(w[2 * k + 1]) : bf16_lo(w[2 * k + 1]);
    t[k] = f2_mul(f2_pack(e0, e1), rr);
  }
  return sr ? e2m1x8_rs(t[0], t[1], t[2], t[3], w0, w1) : e2m1x8_rn(t[0], t[1], t[2], t[3]);
}

// Four scaled values -> four codes in 16 bits, element 0 in bits 3:0: round-to-nearest-even
// (two cvt.rn.satfinite.e2m1x2.f32) or, with SR, one cvt.rs.satfinite.e2m1x4.f32 taking
// random word w (operands a, b, e, f = elements 3, 2, 1, 0).
template <bool SR>
__device__ __forceinline__ uint32_t e2m1x4(float t0, float t1, float t2, float t3, uint32_t w) {
  uint16_t d;
  if (SR) {
    asm("cvt.rs.satfinite.e2m1x4.f32 %0, {%1, %2, %3, %4}, %5;"
        : "=h"(d) : "f"(t3), "f"(t2), "f"(t1), "f"(t0), "r"(w));
  } else {
    asm("{\n\t.reg .b8 q0, q1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 q0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 q1, %4, %3;\n\t"
        "mov.b16 %0, {q0, q1};\n\t}"
        : "=h"(d) : "f"(t0), "f"(t1), "f"(t2), "f"(t3));
  }
  return (uint32_t)d;
}

// ------------------------------------------------------------------------------------------
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3",
// SC'11). One draw per 16-element block, all four words used ([PR4798] "Optimization" item 3;
// the counter is the block's position, so results do not depend on the visit order).
// ------------------------------------------------------------------------------------------
// The round keys are precomputed on the host (k[0][r], k[1][r] for round r: the seed's halves
// bumped by the Weyl constants), so that the XORs take them straight from the kernel parameters.
__device__ __forceinline__ uint4 philox4x32_10_rk(uint4 c, const uint32_t (&k)[2][10]) {
#pragma unroll
  for (int round = 0; round < 10; round++) {
    uint64_t p0 = (uint64_t)0xD2511F53u * c.x;
    uint64_t p1 = (uint64_t)0xCD9E8D57u * c.z;
    c = make_uint4((uint32_t)(p1 >> 32) ^ c.y ^ k[0][round], (uint32_t)p1,
                   (uint32_t)(p0 >> 32) ^ c.w ^ k[1][round], (uint32_t)p0);
  }
  return c;
}
__device__ __forceinline__ uint4 block_random_rk(const uint32_t (&k)[2][10], uint32_t offset,
                                                 uint32_t tag, uint64_t b) {
  return philox4x32_10_rk(make_uint4((uint32_t)b, (uint32_t)(b >> 32), tag, offset), k);
}

// ------------------------------------------------------------------------------------------
// 16-point random Hadamard transform of two adjacent columns at once ([PR4798] "Optimization"
// items 2 and 5; "Fast math": an FP32 accumulator rounded through BF16 in exact mode).
// w[i] holds rows i of the two columns as a BF16 pair. In place: w[i] <- bf16(0.25 * (H16 (d .
// v))_i) for each column, H16 the natural-order Sylvester matrix computed by butterflies in
// stages 1, 2, 4, 8 ((a, b) -> (a + b, a - b), a the lower index), d_i = -1 where flip[i] is
// 0x80000000 (flip[i] is 0 or that word: the sign vector as the kernels' parameters hold it, so
// that the sign flips cost nothing beyond the widening to binary32).
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ void rht16_pair(uint32_t (&w)[16], const uint32_t (&flip)[16]) {
  uint64_t x[16];
#pragma unroll
  for (int i = 0; i < 16; i++) x[i] = f2_from_bf16x2_flip(w[i], flip[i]);
#pragma unroll
  for (int h = 1; h < 16; h <<= 1) {
#pragma unroll
    for (int i = 0; i < 16; i++) {
      if ((i & h) == 0) {
        uint64_t a = x[i], b = x[i + h];
        x[i] = f2_add(a, b);
        x[i + h] = f2_sub(a, b);
      }
    }
  }
  const uint64_t quarter = f2_pack(0.25f, 0.25f);
#pragma unroll
  for (int i = 0; i < 16; i++) {
    float2 y = f2_unpack(f2_mul(x[i], quarter));
    uint32_t packed;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(packed) : "f"(y.y), "f"(y.x));
    w[i] = packed;
  }
}

// ------------------------------------------------------------------------------------------
// Shared memory, mbarriers and TMA
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
// Programmatic dependent launch. A kernel launched with launch_pdl (nvfp4_internal.h) may
// start before the previous kernel in its stream has ended: it calls pdl_wait() before it
// touches memory, and pdl_allow_next() lets the next such kernel start on SMs that finish.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_allow_next() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// One 32-byte global store (a full sector); p must be 32-byte aligned.
__device__ __forceinline__ void stg256(void* p, const uint4& lo, const uint4& hi) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(lo.x),
               "r"(lo.y), "r"(lo.z), "r"(lo.w), "r"(hi.x), "r"(hi.y), "r"(hi.z), "r"(hi.w)
               : "memory");
}
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return done != 0;
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// Barrier over `count` threads (a multiple of 32) on hardware barrier `id` (1..15).
__device__ __forceinline__ void named_bar_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
// Wait for phase `parity` of `bar` to complete, giving up after `limit_ns` nanoseconds of
// global time. Returns false on a timeout.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  uint64_t t0;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    if (t - t0 > limit_ns) return false;
  }
}

// 2D tiled TMA load of the box at (x = innermost element index, y = row) into shared memory,
// completing on `bar`. Out-of-range rows and columns are filled with zeros.
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const void* tensor_map, int32_t x,
                                            int32_t y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(smem_dst)),
      "l"(tensor_map), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// 3D tiled TMA store of the box at (x, y, z) from shared memory (bulk async group); the
// parts of the box outside the tensor are not written.
__device__ __forceinline__ void tma_store_3d(const void* tensor_map, const void* smem_src, int32_t x,
                                             int32_t y, int32_t z) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];"
               ::"l"(tensor_map), "r"(smem_u32(smem_src)), "r"(x), "r"(y), "r"(z)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until the bulk stores committed by this thread have read their shared memory.
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// Wait until they have completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void prefetch_tensormap(const void* tensor_map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(tensor_map) : "memory");
}

}  // namespace nvfp4
