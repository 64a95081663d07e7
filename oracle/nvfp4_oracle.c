/*
 * nvfp4_oracle.c -- the oracle: a plain, scalar CPU statement of NVFP4 block-scaled
 * quantization, written to be read against the pages, not to be fast.
 *
 * TEST INFRASTRUCTURE. Only the test-suite, the smoke check and the benchmark's CPU-baseline
 * leg load this file. The CUDA library never links, includes or calls it, and it shares no
 * header, table or helper with the CUDA sources.
 *
 * Sources. "[PR4798]" is the page "[nvfp4_training] Optimize CuteDSL kernels for NVFP4
 * training" (pytorch/ao pull request #4798); sections are named by its headings
 * ("Optimization" items 1-7, "Fast math", "Grouped allocation tail", "Config surface and
 * AUTO", "Correctness", and the "Philox divergence between CuteDSL and Triton" part of its
 * summary). "[Perplexity]" is the page "CuTeDSL at Perplexity" (its Blackwell paragraph on
 * NVFP4/MXFP8 block reductions).
 *
 * Arithmetic. Every step of the method is IEEE binary32 with round-to-nearest-even and
 * subnormals kept -- the precision the pages fix (an FP32 global scale, packed f32 multiplies,
 * a div.rn reciprocal, an FP32 Hadamard accumulator). Build with -ffp-contract=off and
 * without fast-math so that no multiply-add is fused. The format encoders (E4M3, E2M1, BF16)
 * are exact definitions and use double only where it is exact.
 *
 * Where the pages leave a step open, the reading taken is stated beside the code:
 *   R1 global scale S_enc = 2688 / amax (448 * 6), S_enc = 1 when amax == 0, clamped to
 *      FLT_MAX when the quotient overflows; S_dec = 1 / S_enc. Stored per tensor as
 *      {amax, S_dec}.
 *   R2 block scale s = E4M3_rn_satfinite((bamax / 6) * S_enc), in that order.
 *   R3 element multiplier r = 1 / (float(s) * S_dec) correctly rounded, r = 0 when the
 *      product is 0, clamped to FLT_MAX when the reciprocal overflows.
 *   R4 E2M1 rounding keeps the sign of a value that rounds to zero (code 0x8).
 *   R5 codes are packed two per byte, the even element in the low nibble.
 *   R6 the columnwise RHT of a 16-element block v is y = bf16_rne(0.25 * FWHT16(d * v)), with
 *      FWHT16 the natural-order (Sylvester) Hadamard computed by butterflies in stages
 *      h = 1, 2, 4, 8, and d_i = -1 where bit i of the sign mask is set.
 *   R7 stochastic rounding draws one Philox4x32-10 block per 16-element block with
 *      key = (lo32(seed), hi32(seed)) and counter = (lo32(b), hi32(b), tag, offset), where b
 *      is the block's linear index in its scale tensor and tag is 0 rowwise, 1 columnwise.
 *      Word j is the random operand of the one cvt.rs.satfinite.e2m1x4.f32 that converts
 *      elements 4j..4j+3 (operands a, b, e, f = elements 4j+3, 4j+2, 4j+1, 4j, so that
 *      element 4j lands in the low nibble).
 *   R8 that instruction, as modelled here: each element gets a 16-bit random value U; its
 *      magnitude rounds up by one E2M1 step when U, added to the top 16 of the bits of |t|
 *      below the E2M1 step at |t|'s binade, carries out; the result saturates at 6 (the PTX
 *      description of cvt with .rs rounding: random bits added to the discarded mantissa
 *      bits). For rbits word w: U_b = w[31:24]:w[15:8], U_a = bit-reverse16(U_b),
 *      U_f = w[23:16]:w[7:0], U_e = bit-reverse16(U_f). This assignment of random bits to
 *      lanes was read off the instruction itself, run on chosen inputs (1.32 million
 *      cases, all four lanes, no exception).
 *   R9 columnwise outputs are the transposed tensors: codes [N][M/2], scales [N][M/16].
 *   R10 2D (16x16) scales are written replicated into the rowwise [M][N/16] and columnwise
 *      [N][M/16] scale tensors.
 *   R11 grouped: expert e owns rows [off[e-1], off[e]) (off[-1] = 0); its columnwise output
 *      starts at column sum_{j<e} pad16(n_j) and covers pad16(n_e) zero-padded tokens.
 *   R12 fast math has no CPU statement (a hardware reciprocal); it is bounded against the exact
 *      path by the GPU tests, not computed here.
 *   R13 inverse RHT (checks at the GEMM boundary), R14 the RMSNorm producer, R15 grouped 2D
 *      and M1-M4 (MX formats) are stated beside their code below.
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_API __attribute__((visibility("default")))

/* ------------------------------------------------------------------------------------------ */
/* Bit-level views                                                                             */
/* ------------------------------------------------------------------------------------------ */

static float f32_from_bits(uint32_t u) { float f; memcpy(&f, &u, sizeof f); return f; }
static uint32_t bits_of_f32(float f) { uint32_t u; memcpy(&u, &f, sizeof u); return u; }

/* BF16 is the upper half of a binary32, so widening is a 16-bit shift and exact
 * ([PR4798] Optimization item 6). */
static float bf16_to_f32(uint16_t h) { return f32_from_bits((uint32_t)h << 16); }

/* binary32 -> BF16, round to nearest, ties to even. */
static uint16_t f32_to_bf16_rne(float f) {
  uint32_t u = bits_of_f32(f);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0) {
    return (uint16_t)((u >> 16) | 0x0040u); /* NaN stays a (quiet) NaN */
  }
  uint32_t upper = u >> 16;
  uint32_t lower = u & 0xFFFFu;
  if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u) != 0)) upper += 1u;
  return (uint16_t)upper;
}

/* Round a non-negative double to the nearest integer, ties to the even integer. */
static double round_half_even(double x) {
  double f = floor(x);
  double d = x - f;
  if (d > 0.5) return f + 1.0;
  if (d < 0.5) return f;
  return (fmod(f, 2.0) == 0.0) ? f : f + 1.0;
}

/* ------------------------------------------------------------------------------------------ */
/* E4M3 (FP8, 1 sign / 4 exponent bits, bias 7 / 3 mantissa bits, no infinities, largest      */
/* finite 448 = 1.75 * 2^8, subnormals 0.mmm * 2^-6 down to 2^-9). The block-scale format.    */
/* ------------------------------------------------------------------------------------------ */

static uint8_t e4m3_encode_rn_satfinite(float v) {
  uint8_t sign = signbit(v) ? 0x80 : 0x00;
  double a = fabs((double)v);
  if (isnan(v)) return 0x7F;
  if (a >= 448.0) return (uint8_t)(sign | 0x7E); /* satfinite: clamp to the largest finite */
  if (a < ldexp(1.0, -6)) {
    /* subnormal range: the value is an integer multiple of 2^-9; q == 8 is 2^-6 = code 0x08 */
    double q = round_half_even(a * 512.0);
    return (uint8_t)(sign | (uint8_t)q);
  }
  int e2;
  double m = frexp(a, &e2); /* a = m * 2^e2, m in [0.5, 1) */
  int e = e2 - 1;           /* a = (2m) * 2^e, 2m in [1, 2) */
  double mant = round_half_even((2.0 * m - 1.0) * 8.0);
  if (mant == 8.0) { mant = 0.0; e += 1; }
  int code = ((e + 7) << 3) | (int)mant;
  if (code > 0x7E) code = 0x7E;
  return (uint8_t)(sign | code);
}

static float e4m3_decode(uint8_t c) {
  int exp_bits = (c >> 3) & 0xF;
  int man = c & 0x7;
  double v;
  if ((c & 0x7F) == 0x7F) return NAN;
  if (exp_bits == 0) v = ldexp((double)man, -9);
  else v = ldexp(1.0 + man / 8.0, exp_bits - 7);
  return (float)((c & 0x80) ? -v : v);
}

/* ------------------------------------------------------------------------------------------ */
/* E2M1 (FP4, 1 sign / 2 exponent bits / 1 mantissa bit). Magnitudes by code 0..7.            */
/* ------------------------------------------------------------------------------------------ */

static const double E2M1_MAG[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

static float e2m1_decode(uint8_t nib) {
  double v = E2M1_MAG[nib & 7];
  return (float)((nib & 8) ? -v : v);
}

/* Round-to-nearest-even onto the E2M1 grid, saturating at 6 (cvt.rn.satfinite.e2m1x2.f32,
 * [PR4798] Optimization item 1). Ties go to the code with a zero mantissa bit. Reading R4. */
static uint8_t e2m1_encode_rn_satfinite(float t) {
  uint8_t sign = signbit(t) ? 8 : 0;
  double a = fabs((double)t);
  if (a >= 6.0) return (uint8_t)(sign | 7);
  int k = 0;
  while (k < 6 && E2M1_MAG[k + 1] <= a) k++; /* E2M1_MAG[k] <= a < E2M1_MAG[k + 1] */
  double below = a - E2M1_MAG[k];
  double above = E2M1_MAG[k + 1] - a;
  int code;
  if (below < above) code = k;
  else if (above < below) code = k + 1;
  else code = (k % 2 == 0) ? k : k + 1;
  return (uint8_t)(sign | code);
}

/* Stochastic rounding onto the E2M1 grid with a 16-bit random value (one lane of
 * cvt.rs.satfinite.e2m1x4.f32, [PR4798] Optimization item 3). Reading R8: in the binade of |t|
 * the grid step is 0.5 below 2, 1 in [2, 4) and 2 in [4, 8); |t| = (q + f) * step with q an
 * integer and f in [0, 1). The discarded fraction f, cut to its top 16 bits, plus the random
 * value carries out of 16 bits exactly when the magnitude rounds up by one step. Saturates
 * at 6. */
static uint8_t e2m1_encode_sr_satfinite(float t, uint32_t rand16) {
  uint8_t sign = signbit(t) ? 8 : 0;
  double a = fabs((double)t);
  if (a >= 6.0) return (uint8_t)(sign | 7);
  double step = (a < 2.0) ? 0.5 : (a < 4.0 ? 1.0 : 2.0);
  double q = floor(a / step);            /* exact: step is a power of two */
  double f = a / step - q;               /* exact */
  uint32_t top16 = (uint32_t)floor(f * 65536.0);
  double mag = q * step;
  if (top16 + (rand16 & 0xFFFFu) >= 65536u) mag += step;
  int code = 0;
  while (code < 7 && E2M1_MAG[code] != mag) code++;
  if (mag > 6.0) code = 7;
  return (uint8_t)(sign | code);
}

static uint32_t bit_reverse16(uint32_t u) {
  uint32_t r = 0;
  for (int i = 0; i < 16; i++) r |= ((u >> i) & 1u) << (15 - i);
  return r;
}

/* The 16-bit random value that word w gives element 4j+i of its group of four (reading R8:
 * i = 0, 1, 2, 3 are the instruction's operands f, e, b, a). */
static uint32_t sr_random16(uint32_t w, int i) {
  uint32_t u_b = ((w >> 24) & 0xFFu) << 8 | ((w >> 8) & 0xFFu);
  uint32_t u_f = ((w >> 16) & 0xFFu) << 8 | (w & 0xFFu);
  switch (i) {
    case 0: return u_f;
    case 1: return bit_reverse16(u_f);
    case 2: return u_b;
    default: return bit_reverse16(u_b);
  }
}

/* ------------------------------------------------------------------------------------------ */
/* Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3",   */
/* SC'11): ten rounds of two 32x32->64 multiplies; the key is bumped by the Weyl constants     */
/* before every round after the first.                                                        */
/* ------------------------------------------------------------------------------------------ */

static void philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
  uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
  uint32_t k0 = key[0], k1 = key[1];
  for (int round = 0; round < 10; round++) {
    if (round > 0) { k0 += 0x9E3779B9u; k1 += 0xBB67AE85u; }
    uint64_t p0 = (uint64_t)0xD2511F53u * (uint64_t)c0;
    uint64_t p1 = (uint64_t)0xCD9E8D57u * (uint64_t)c2;
    uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
    uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
    uint32_t n0 = hi1 ^ c1 ^ k0;
    uint32_t n1 = lo1;
    uint32_t n2 = hi0 ^ c3 ^ k1;
    uint32_t n3 = lo0;
    c0 = n0; c1 = n1; c2 = n2; c3 = n3;
  }
  out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* The four random words of one 16-element block (reading R7; [PR4798] Optimization item 3:
 * one counter per block, all four output words consumed). */
static void block_random_words(uint64_t seed, uint32_t offset, uint32_t tag, uint64_t b,
                               uint32_t words[4]) {
  uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
  uint32_t ctr[4] = {(uint32_t)b, (uint32_t)(b >> 32), tag, offset};
  philox4x32_10(ctr, key, words);
}

/* ------------------------------------------------------------------------------------------ */
/* 16-point random Hadamard transform (reading R6; [PR4798] Optimization item 2 and "Fast      */
/* math": an FP32 accumulator rounded through BF16 in exact mode).                             */
/* ------------------------------------------------------------------------------------------ */

static void fwht16(float w[16]) {
  for (int h = 1; h < 16; h <<= 1) {
    for (int i = 0; i < 16; i++) {
      if ((i & h) == 0) {
        float a = w[i];
        float b = w[i + h];
        w[i] = a + b;
        w[i + h] = a - b;
      }
    }
  }
}

static void rht16(const float v[16], uint32_t sign_mask, float y[16]) {
  float w[16];
  for (int i = 0; i < 16; i++) w[i] = ((sign_mask >> i) & 1u) ? -v[i] : v[i];
  fwht16(w);
  for (int i = 0; i < 16; i++) {
    float scaled = 0.25f * w[i];
    y[i] = bf16_to_f32(f32_to_bf16_rne(scaled));
  }
}

/* ------------------------------------------------------------------------------------------ */
/* Scales                                                                                      */
/* ------------------------------------------------------------------------------------------ */

/* Reading R1 ([PR4798] "Fast math": the per-tensor global_decode_scale). */
static void global_scale(float amax, float* s_enc, float* s_dec) {
  float enc;
  if (amax == 0.0f) {
    enc = 1.0f;
  } else {
    enc = 2688.0f / amax;
    if (!(enc <= FLT_MAX)) enc = FLT_MAX;
  }
  *s_enc = enc;
  *s_dec = 1.0f / enc;
}

/* Reading R2: the E4M3 block scale from the block amax ([Perplexity] NVFP4 paragraph: a
 * 16-element absolute maximum per block). */
static uint8_t block_scale(float bamax, float s_enc) {
  float per_code = bamax / 6.0f;
  float s32 = per_code * s_enc;
  return e4m3_encode_rn_satfinite(s32);
}

/* Reading R3 ([PR4798] "Fast math": exact mode takes the correctly rounded reciprocal of
 * pvscale_fp8 * global_decode_scale). */
static float element_multiplier(uint8_t s, float s_dec) {
  float p = e4m3_decode(s) * s_dec;
  if (p == 0.0f) return 0.0f;
  float r = 1.0f / p;
  if (!(r <= FLT_MAX)) r = FLT_MAX;
  return r;
}

/* Quantize the 16 codes of one block with multiplier r; rand == NULL selects RTNE.
 * Reading R5 for the packing. */
static void encode_block(const float v[16], float r, const uint32_t* rand, uint8_t codes[8]) {
  uint8_t q[16];
  for (int i = 0; i < 16; i++) {
    float t = v[i] * r;
    if (rand) q[i] = e2m1_encode_sr_satfinite(t, sr_random16(rand[i / 4], i % 4));
    else q[i] = e2m1_encode_rn_satfinite(t);
  }
  for (int k = 0; k < 8; k++) codes[k] = (uint8_t)(q[2 * k] | (q[2 * k + 1] << 4));
}

static float abs_max16(const float v[16]) {
  float m = 0.0f;
  for (int i = 0; i < 16; i++) {
    float a = fabsf(v[i]);
    if (a > m) m = a;
  }
  return m;
}

/* One 1x16 block: block amax -> E4M3 scale -> multiplier -> codes. */
static void quantize_block16(const float v[16], float s_enc, float s_dec, const uint32_t* rand,
                             uint8_t codes[8], uint8_t* scale) {
  uint8_t s = block_scale(abs_max16(v), s_enc);
  encode_block(v, element_multiplier(s, s_dec), rand, codes);
  *scale = s;
}

/* ------------------------------------------------------------------------------------------ */
/* Exported primitives (pinned one by one in the oracle's own tests)                           */
/* ------------------------------------------------------------------------------------------ */

ORACLE_API uint16_t oracle_f32_to_bf16(float f) { return f32_to_bf16_rne(f); }
ORACLE_API uint8_t oracle_e4m3_encode(float v) { return e4m3_encode_rn_satfinite(v); }
ORACLE_API float oracle_e4m3_decode(uint8_t c) { return e4m3_decode(c); }
ORACLE_API uint8_t oracle_e2m1_encode_rn(float t) { return e2m1_encode_rn_satfinite(t); }
ORACLE_API uint8_t oracle_e2m1_encode_sr(float t, uint32_t r16) { return e2m1_encode_sr_satfinite(t, r16); }
ORACLE_API uint32_t oracle_sr_random16(uint32_t w, int32_t i) { return sr_random16(w, i); }
/* One cvt.rs.satfinite.e2m1x4.f32 per random word, as reading R8 models it: element 4k+i
 * (i = 0..3) of t is rounded with the 16-bit value that word k gives lane i; one code per
 * byte of `codes` (sign in bit 3). The batch form of the per-element step of encode_block. */
ORACLE_API void oracle_sr_convert4_n(const float* t, const uint32_t* words, int64_t n_words,
                                     uint8_t* codes) {
  for (int64_t k = 0; k < n_words; k++)
    for (int i = 0; i < 4; i++)
      codes[4 * k + i] = e2m1_encode_sr_satfinite(t[4 * k + i], sr_random16(words[k], i));
}
/* Round-to-nearest-even encoding of n values, one code per byte (the batch form of
 * e2m1_encode_rn_satfinite). */
ORACLE_API void oracle_e2m1_encode_rn_n(const float* t, int64_t n, uint8_t* codes) {
  for (int64_t k = 0; k < n; k++) codes[k] = e2m1_encode_rn_satfinite(t[k]);
}
ORACLE_API float oracle_e2m1_decode(uint8_t n) { return e2m1_decode(n); }
ORACLE_API void oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
  philox4x32_10(ctr, key, out);
}
ORACLE_API void oracle_fwht16(float w[16]) { fwht16(w); }
ORACLE_API void oracle_rht16(const float v[16], uint32_t sign_mask, float y[16]) { rht16(v, sign_mask, y); }
ORACLE_API void oracle_global_scale(float amax, float out[2]) { global_scale(amax, &out[0], &out[1]); }
ORACLE_API uint8_t oracle_block_scale(float bamax, float s_enc) { return block_scale(bamax, s_enc); }
ORACLE_API float oracle_element_multiplier(uint8_t s, float s_dec) { return element_multiplier(s, s_dec); }
ORACLE_API void oracle_quantize_block16(const float v[16], float s_enc, float s_dec,
                                        const uint32_t* rand, uint8_t codes[8], uint8_t* scale) {
  quantize_block16(v, s_enc, s_dec, rand, codes, scale);
}

/* ------------------------------------------------------------------------------------------ */
/* Tensors. x is BF16 [M][N] row-major, passed as its 16-bit patterns.                         */
/* ------------------------------------------------------------------------------------------ */

/* Per-tensor amax over all elements ([PR4798] "Fast math": the amax kernels are exact). */
ORACLE_API float oracle_amax(const uint16_t* x, int64_t M, int64_t N) {
  float m = 0.0f;
  for (int64_t i = 0; i < M * N; i++) {
    float a = fabsf(bf16_to_f32(x[i]));
    if (a > m) m = a;
  }
  return m;
}

/* Column block (16 rows starting at row r0, column n) of x, zero where row >= row_end. */
static void load_column_block(const uint16_t* x, int64_t N, int64_t r0, int64_t row_end,
                              int64_t n, float v[16]) {
  for (int i = 0; i < 16; i++) {
    int64_t r = r0 + i;
    v[i] = (r < row_end) ? bf16_to_f32(x[r * N + n]) : 0.0f;
  }
}

/* amax of the RHT output over every 16-row column block ("Linear RHT amax", [PR4798]
 * Optimization item 5). Requires M % 16 == 0. */
ORACLE_API float oracle_amax_rht(const uint16_t* x, int64_t M, int64_t N, uint32_t sign_mask) {
  float m = 0.0f;
  for (int64_t n = 0; n < N; n++) {
    for (int64_t rb = 0; rb < M / 16; rb++) {
      float v[16], y[16];
      load_column_block(x, N, rb * 16, M, n, v);
      rht16(v, sign_mask, y);
      float a = abs_max16(y);
      if (a > m) m = a;
    }
  }
  return m;
}

/* Rowwise 1x16 quantization of rows [row_begin, row_end) with one global scale.
 * codes [M][N/2], scales [M][N/16]. sr != 0 selects stochastic rounding (tag 0). */
static void rowwise_rows(const uint16_t* x, int64_t N, int64_t row_begin, int64_t row_end,
                         float s_enc, float s_dec, int sr, uint64_t seed, uint32_t offset,
                         uint8_t* codes, uint8_t* scales) {
  int64_t nb = N / 16;
  for (int64_t r = row_begin; r < row_end; r++) {
    for (int64_t b = 0; b < nb; b++) {
      float v[16];
      uint32_t rand[4];
      for (int i = 0; i < 16; i++) v[i] = bf16_to_f32(x[r * N + 16 * b + i]);
      if (sr) block_random_words(seed, offset, 0u, (uint64_t)(r * nb + b), rand);
      quantize_block16(v, s_enc, s_dec, sr ? rand : NULL, &codes[r * (N / 2) + 8 * b],
                       &scales[r * nb + b]);
    }
  }
}

ORACLE_API void oracle_quantize_rowwise(const uint16_t* x, int64_t M, int64_t N, float amax,
                                        int sr, uint64_t seed, uint32_t offset,
                                        uint8_t* codes, uint8_t* scales, float gscale[2]) {
  float s_enc, s_dec;
  global_scale(amax, &s_enc, &s_dec);
  gscale[0] = amax;
  gscale[1] = s_dec;
  rowwise_rows(x, N, 0, M, s_enc, s_dec, sr, seed, offset, codes, scales);
}

/* Columnwise 1x16 quantization (blocks of 16 consecutive rows of one column), written
 * transposed (reading R9). Rows [row_begin, row_begin + 16 * nblk) of x, zero-padded at and
 * beyond row_end, become output columns [col0, col0 + 16 * nblk) of the [N][ld] output
 * (ld = output row length in elements). SR uses tag 1 and the block's index in the
 * [N][ld/16] scale tensor. */
static void colwise_blocks(const uint16_t* x, int64_t N, int64_t row_begin, int64_t row_end,
                           int64_t nblk, int64_t ld, int64_t col0, float s_enc, float s_dec,
                           int rht, uint32_t sign_mask, int sr, uint64_t seed, uint32_t offset,
                           uint8_t* codes, uint8_t* scales) {
  for (int64_t n = 0; n < N; n++) {
    for (int64_t k = 0; k < nblk; k++) {
      float v[16], y[16];
      uint32_t rand[4];
      load_column_block(x, N, row_begin + 16 * k, row_end, n, v);
      if (rht) rht16(v, sign_mask, y);
      else memcpy(y, v, sizeof y);
      int64_t b = n * (ld / 16) + col0 / 16 + k;
      if (sr) block_random_words(seed, offset, 1u, (uint64_t)b, rand);
      quantize_block16(y, s_enc, s_dec, sr ? rand : NULL, &codes[n * (ld / 2) + col0 / 2 + 8 * k],
                       &scales[b]);
    }
  }
}

/* amax_col is the tensor amax, or the RHT amax when rht != 0. Requires M % 16 == 0. */
ORACLE_API void oracle_quantize_colwise(const uint16_t* x, int64_t M, int64_t N, float amax_col,
                                        int rht, uint32_t sign_mask, int sr, uint64_t seed,
                                        uint32_t offset, uint8_t* codes, uint8_t* scales,
                                        float gscale[2]) {
  float s_enc, s_dec;
  global_scale(amax_col, &s_enc, &s_dec);
  gscale[0] = amax_col;
  gscale[1] = s_dec;
  colwise_blocks(x, N, 0, M, M / 16, M, 0, s_enc, s_dec, rht, sign_mask, sr, seed, offset,
                 codes, scales);
}

/* 16x16 2D block scaling ([PR4798] Optimization item 2, the 2D weight kernel): one E4M3 scale
 * per 16x16 tile from the tile amax, shared by the rowwise and the columnwise codes, written
 * replicated (reading R10). RTNE only. Requires M % 16 == 0 and N % 16 == 0. */
ORACLE_API void oracle_quantize_2d(const uint16_t* x, int64_t M, int64_t N, float amax,
                                   uint8_t* row_codes, uint8_t* row_scales,
                                   uint8_t* col_codes, uint8_t* col_scales, float gscale[2]) {
  float s_enc, s_dec;
  global_scale(amax, &s_enc, &s_dec);
  gscale[0] = amax;
  gscale[1] = s_dec;
  for (int64_t tr = 0; tr < M / 16; tr++) {
    for (int64_t tc = 0; tc < N / 16; tc++) {
      float tile_amax = 0.0f;
      for (int i = 0; i < 16; i++) {
        for (int j = 0; j < 16; j++) {
          float a = fabsf(bf16_to_f32(x[(16 * tr + i) * N + 16 * tc + j]));
          if (a > tile_amax) tile_amax = a;
        }
      }
      uint8_t s = block_scale(tile_amax, s_enc);
      float r = element_multiplier(s, s_dec);
      for (int i = 0; i < 16; i++) { /* the tile's 16 row segments */
        int64_t row = 16 * tr + i;
        float v[16];
        for (int j = 0; j < 16; j++) v[j] = bf16_to_f32(x[row * N + 16 * tc + j]);
        encode_block(v, r, NULL, &row_codes[row * (N / 2) + 8 * tc]);
        row_scales[row * (N / 16) + tc] = s;
      }
      for (int j = 0; j < 16; j++) { /* the tile's 16 column segments */
        int64_t col = 16 * tc + j;
        float v[16];
        for (int i = 0; i < 16; i++) v[i] = bf16_to_f32(x[(16 * tr + i) * N + col]);
        encode_block(v, r, NULL, &col_codes[col * (M / 2) + 8 * tr]);
        col_scales[col * (M / 16) + tr] = s;
      }
    }
  }
}

/* Grouped (MoE) quantization ([PR4798] "Grouped allocation tail" and "Config surface and
 * AUTO": a packed [T][H] tensor with device-side cumulative offsets; rows past the last offset
 * are not written). Reading R11 for the columnwise layout. offsets[E] are cumulative ends.
 * Per expert e: amax over its rows; rowwise with that expert's global scale; columnwise over
 * its pad16(n_e) zero-padded tokens with the expert's (RHT) amax.
 * Outputs: row_codes [T][H/2], row_scales [T][H/16], row_gscale [E][2]; col_codes [H][cap/2],
 * col_scales [H][cap/16], col_gscale [E][2]. Either side may be skipped by passing NULL codes.
 * Returns 0, or -1 when the offsets are not non-decreasing within [0, T] or the padded token
 * total exceeds cap (then nothing is written). */
ORACLE_API int oracle_quantize_grouped(const uint16_t* x, int64_t T, int64_t H,
                                       const int32_t* offsets, int32_t E, int64_t cap,
                                       int round_row_sr, int round_col_sr, int rht_col,
                                       uint32_t sign_mask, uint64_t seed, uint32_t offset,
                                       uint8_t* row_codes, uint8_t* row_scales, float* row_gscale,
                                       uint8_t* col_codes, uint8_t* col_scales, float* col_gscale) {
  int64_t padded_total = 0;
  int64_t prev = 0;
  for (int32_t e = 0; e < E; e++) {
    if (offsets[e] < prev || offsets[e] > T) return -1;
    padded_total += ((offsets[e] - prev) + 15) / 16 * 16;
    prev = offsets[e];
  }
  if (col_codes && padded_total > cap) return -1;

  int64_t col_start = 0;
  for (int32_t e = 0; e < E; e++) {
    int64_t start = (e == 0) ? 0 : offsets[e - 1];
    int64_t end = offsets[e];
    int64_t n = end - start;
    int64_t nblk = (n + 15) / 16;
    float amax = oracle_amax(x + start * H, n, H);
    if (row_codes) {
      float s_enc, s_dec;
      global_scale(amax, &s_enc, &s_dec);
      row_gscale[2 * e] = amax;
      row_gscale[2 * e + 1] = s_dec;
      rowwise_rows(x, H, start, end, s_enc, s_dec, round_row_sr, seed, offset, row_codes,
                   row_scales);
    }
    if (col_codes) {
      float amax_col = amax;
      if (rht_col) {
        amax_col = 0.0f;
        for (int64_t h = 0; h < H; h++) {
          for (int64_t k = 0; k < nblk; k++) {
            float v[16], y[16];
            load_column_block(x, H, start + 16 * k, end, h, v);
            rht16(v, sign_mask, y);
            float a = abs_max16(y);
            if (a > amax_col) amax_col = a;
          }
        }
      }
      float s_enc, s_dec;
      global_scale(amax_col, &s_enc, &s_dec);
      col_gscale[2 * e] = amax_col;
      col_gscale[2 * e + 1] = s_dec;
      colwise_blocks(x, H, start, end, nblk, cap, col_start, s_enc, s_dec, rht_col, sign_mask,
                     round_col_sr, seed, offset, col_codes, col_scales);
    }
    col_start += 16 * nblk;
  }
  return 0;
}

/* Grouped 2D (weights of several experts stacked along the rows). Reading R15: expert e's 16x16
 * tiles start at its first row and its last row tile is zero-padded (as R11 pads columnwise
 * blocks); each expert has its own amax and global scales; the tile scale is written for every
 * row of the expert in the rowwise outputs (padding rows belong to no output) and into the
 * expert's padded columns of the columnwise outputs (starting at sum_{j<e} pad16(n_j)). Any
 * orientation may be absent (NULL). Returns -1 for offsets that are not non-decreasing within
 * [0, T] or a capacity below the padded total. */
ORACLE_API int oracle_quantize_grouped_2d(const uint16_t* x, int64_t T, int64_t H,
                                          const int32_t* offsets, int32_t E, int64_t cap,
                                          uint8_t* row_codes, uint8_t* row_scales,
                                          float* row_gscale, uint8_t* col_codes,
                                          uint8_t* col_scales, float* col_gscale) {
  int64_t padded_total = 0, prev = 0;
  for (int32_t e = 0; e < E; e++) {
    if (offsets[e] < prev || offsets[e] > T) return -1;
    padded_total += ((offsets[e] - prev) + 15) / 16 * 16;
    prev = offsets[e];
  }
  if (col_codes && padded_total > cap) return -1;
  int64_t col_start = 0;
  for (int32_t e = 0; e < E; e++) {
    int64_t start = (e == 0) ? 0 : offsets[e - 1];
    int64_t n = offsets[e] - start;
    int64_t P = (n + 15) / 16 * 16;
    float amax = oracle_amax(x + start * H, n, H);
    float gs[2];
    if (P > 0) {
      /* the expert's rows, zero-padded to whole tiles, through the plain 2D quantizer */
      uint16_t* xs = (uint16_t*)calloc((size_t)(P * H), sizeof(uint16_t));
      uint8_t* rc = (uint8_t*)malloc((size_t)(P * H / 2));
      uint8_t* rs = (uint8_t*)malloc((size_t)(P * H / 16));
      uint8_t* cc = (uint8_t*)malloc((size_t)(P * H / 2));
      uint8_t* cs = (uint8_t*)malloc((size_t)(P * H / 16));
      if (!xs || !rc || !rs || !cc || !cs) { free(xs); free(rc); free(rs); free(cc); free(cs); return -2; }
      memcpy(xs, x + start * H, (size_t)(n * H) * sizeof(uint16_t));
      oracle_quantize_2d(xs, P, H, amax, rc, rs, cc, cs, gs);
      if (row_codes) {
        memcpy(row_codes + start * (H / 2), rc, (size_t)(n * H / 2));
        memcpy(row_scales + start * (H / 16), rs, (size_t)(n * H / 16));
      }
      if (col_codes) {
        for (int64_t h = 0; h < H; h++) {
          memcpy(col_codes + h * (cap / 2) + col_start / 2, cc + h * (P / 2), (size_t)(P / 2));
          memcpy(col_scales + h * (cap / 16) + col_start / 16, cs + h * (P / 16), (size_t)(P / 16));
        }
      }
      free(xs); free(rc); free(rs); free(cc); free(cs);
    } else {
      float s_enc;
      global_scale(amax, &s_enc, &gs[1]);
      gs[0] = amax;
    }
    if (row_gscale) { row_gscale[2 * e] = gs[0]; row_gscale[2 * e + 1] = gs[1]; }
    if (col_gscale) { col_gscale[2 * e] = gs[0]; col_gscale[2 * e + 1] = gs[1]; }
    col_start += P;
  }
  return 0;
}

/* Dequantization: x_hat = (e2m1(q) * float(s)) * S_dec. The inner product is exact (2 + 4
 * significant bits). codes [R][C/2], scales [R][C/16], out [R][C]. */
ORACLE_API void oracle_dequantize(const uint8_t* codes, const uint8_t* scales, float s_dec,
                                  int64_t R, int64_t C, float* out) {
  for (int64_t r = 0; r < R; r++) {
    for (int64_t c = 0; c < C; c++) {
      uint8_t byte = codes[r * (C / 2) + c / 2];
      uint8_t nib = (c % 2 == 0) ? (byte & 0xF) : (byte >> 4);
      float s = e4m3_decode(scales[r * (C / 16) + c / 16]);
      float v = e2m1_decode(nib) * s;
      out[r * C + c] = v * s_dec;
    }
  }
}

/* ------------------------------------------------------------------------------------------ */
/* Verification at the GEMM boundary: BF16 dequantization and the inverse RHT.                */
/*   R13 The columnwise RHT output y of a 16-element block is undone as v = d * (0.25 *       */
/*       FWHT16(y)) in binary32 with the same butterflies as R6 (H16 H16 = 16 I, so 0.25 H16  */
/*       is its own inverse, and so is d). Applied to dequantized values it reconstructs the  */
/*       pre-transform column up to the quantization error. BF16 outputs are the binary32    */
/*       results rounded to nearest-even.                                                      */
/* ------------------------------------------------------------------------------------------ */

static void inverse_rht16(const float y[16], uint32_t sign_mask, float v[16]) {
  float w[16];
  for (int i = 0; i < 16; i++) w[i] = y[i];
  fwht16(w);
  for (int i = 0; i < 16; i++) {
    float scaled = 0.25f * w[i];
    v[i] = ((sign_mask >> i) & 1u) ? -scaled : scaled;
  }
}

ORACLE_API void oracle_inverse_rht16(const float y[16], uint32_t sign_mask, float v[16]) {
  inverse_rht16(y, sign_mask, v);
}

/* In place on x [R][C] (C % 16 == 0): every 16-element block of every row. */
ORACLE_API void oracle_inverse_rht_rows(float* x, int64_t R, int64_t C, uint32_t sign_mask) {
  for (int64_t r = 0; r < R; r++) {
    for (int64_t b = 0; b < C / 16; b++) {
      float v[16];
      inverse_rht16(x + r * C + 16 * b, sign_mask, v);
      for (int i = 0; i < 16; i++) x[r * C + 16 * b + i] = v[i];
    }
  }
}

ORACLE_API void oracle_f32_to_bf16_n(const float* in, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; i++) out[i] = f32_to_bf16_rne(in[i]);
}

/* ------------------------------------------------------------------------------------------ */
/* A producer with the amax in its epilogue: RMSNorm ([Perplexity] "CuTeDSL at Perplexity",   */
/* its RMS-norm kernel).                                                                       */
/*   R14 y_i = bf16_rne(fl(fl(w_i + bias) * fl(x_i * rms))), rms = rsqrt_rn(fl(fl(s / N) +    */
/*       eps)), s = sum of x_i^2 in binary32 in the page's order: lane l of a 32-lane group    */
/*       sums, one rounding per term, the squares of its 8-element vectors l, l + 32, l + 64,  */
/*       ... of the row (elements in order), then the 32 partial sums meet in a butterfly      */
/*       (xor 16, 8, 4, 2, 1; each step s + partner's s). rsqrt_rn is 1/sqrt correctly rounded */
/*       to binary32. The epilogue's amax is max |y_i| over the tensor.                        */
/* ------------------------------------------------------------------------------------------ */

/* Is m^2 * a (m, a > 0 finite, m with at most 25 and a with at most 24 significant bits)
 * below (-1), equal to (0) or above (+1) one? Exact, in 128-bit integers. */
static int square_times_vs_one(double m, double a) {
  int em, ea;
  double fm = frexp(m, &em), fa = frexp(a, &ea);
  unsigned __int128 Mm = (unsigned __int128)ldexp(fm, 25), Ma = (unsigned __int128)ldexp(fa, 24);
  int k = -(2 * (em - 25) + (ea - 24));  /* m^2 a = Mm^2 Ma 2^-k */
  unsigned __int128 P = Mm * Mm * Ma;      /* < 2^74 */
  if (k < 0) return 1;
  if (k >= 127) return -1;
  unsigned __int128 one = (unsigned __int128)1 << k;
  return P < one ? -1 : (P > one ? 1 : 0);
}

/* 1 / sqrt(a), correctly rounded to binary32 (round to nearest, ties to even), a > 0 finite:
 * a candidate from double arithmetic, moved until 1/sqrt(a) lies between the midpoints to its
 * neighbours (exact comparisons m^2 a against 1). */
static float rsqrt_rn(float a) {
  float c = (float)(1.0 / sqrt((double)a));
  for (int it = 0; it < 4; it++) {
    float up = nextafterf(c, INFINITY), dn = nextafterf(c, 0.0f);
    double hi = ((double)c + (double)up) / 2, lo = ((double)c + (double)dn) / 2;
    int h = square_times_vs_one(hi, a), l = square_times_vs_one(lo, a);
    if (h < 0) { c = up; continue; }          /* 1/sqrt(a) > hi */
    if (l > 0) { c = dn; continue; }          /* 1/sqrt(a) < lo */
    if (h == 0 && (bits_of_f32(c) & 1u)) c = up;   /* exactly on a midpoint: the even one */
    if (l == 0 && (bits_of_f32(c) & 1u)) c = dn;
    break;
  }
  return c;
}

ORACLE_API float oracle_rsqrt_rn(float a) { return rsqrt_rn(a); }

/* RMSNorm of x [M][N] (BF16, N % 8 == 0) with weight w [N] (BF16) into y [M][N] (BF16 bits);
 * returns the amax of y. Reading R14. */
ORACLE_API float oracle_rmsnorm(const uint16_t* x, const uint16_t* w, int64_t M, int64_t N,
                                float eps, float bias, uint16_t* y) {
  float amax = 0.0f;
  for (int64_t r = 0; r < M; r++) {
    const uint16_t* xr = x + r * N;
    float part[32];
    for (int l = 0; l < 32; l++) {
      float s = 0.0f;
      for (int64_t v = l; v < N / 8; v += 32)
        for (int i = 0; i < 8; i++) {
          float e = bf16_to_f32(xr[8 * v + i]);
          float sq = e * e;
          s = s + sq;
        }
      part[l] = s;
    }
    for (int o = 16; o >= 1; o >>= 1) {
      float next[32];
      for (int l = 0; l < 32; l++) next[l] = part[l] + part[l ^ o];
      for (int l = 0; l < 32; l++) part[l] = next[l];
    }
    float mean = part[0] / (float)N;
    float rms = rsqrt_rn(mean + eps);
    for (int64_t i = 0; i < N; i++) {
      float wb = bf16_to_f32(w[i]) + bias;
      float xr_ = bf16_to_f32(xr[i]) * rms;
      uint16_t q = f32_to_bf16_rne(wb * xr_);
      y[r * N + i] = q;
      float mag = fabsf(bf16_to_f32(q));
      if (mag > amax) amax = mag;
    }
  }
  return amax;
}

/* ========================================================================================== */
/* MX formats: MXFP8 (E4M3 or E5M2 elements) and MXFP4 (E2M1 elements). Blocks of 32         */
/* consecutive elements share one power-of-two scale stored as E8M0; there is no tensor-wide   */
/* scale, so no amax pass. [Perplexity] names the formats and their 32-element block maxima;  */
/* the pages give no formula, so the scale and rounding rules are the conversion the OCP      */
/* Microscaling Formats (MX) v1.0 specification defines (readings M1-M4):                     */
/*   M1 the block's shared exponent is floor(log2(max |v_i|)) - emax_elem, emax_elem being the */
/*      exponent of the element format's largest normal (E4M3: 8, E5M2: 15, E2M1: 2), clamped */
/*      to [-127, 127]; an all-zero block gets -127. The E8M0 code is the exponent + 127 (the  */
/*      NaN code 0xFF is never produced: inputs are finite).                                   */
/*   M2 each element is v_i / 2^exponent rounded to nearest-even onto the element format,     */
/*      saturating at its largest finite magnitude (448, 57344, 6); the sign of a value that  */
/*      rounds to zero is kept.                                                               */
/*   M3 rowwise: codes [M][N] bytes (FP8) or [M][N/2] (FP4, even element in the low nibble),  */
/*      scales [M][N/32]; columnwise: the same for the transposed tensor, codes [N][M] or     */
/*      [N][M/2], scales [N][M/32] (as R9).                                                   */
/*   M4 formats are numbered 0 = E4M3, 1 = E5M2, 2 = E2M1.                                    */
/* ========================================================================================== */

/* E5M2 (FP8, 1 sign / 5 exponent bits, bias 15 / 2 mantissa bits, infinities at 0x7C, largest
 * finite 57344 = 1.75 * 2^15, subnormals 0.mm * 2^-14 down to 2^-16). */
static uint8_t e5m2_encode_rn_satfinite(float v) {
  uint8_t sign = signbit(v) ? 0x80 : 0x00;
  double a = fabs((double)v);
  if (isnan(v)) return 0x7F;
  if (a >= 57344.0) return (uint8_t)(sign | 0x7B); /* satfinite: clamp to the largest finite */
  if (a < ldexp(1.0, -14)) {
    /* subnormal range: an integer multiple of 2^-16; q == 4 is 2^-14 = code 0x04 */
    double q = round_half_even(a * 65536.0);
    return (uint8_t)(sign | (uint8_t)q);
  }
  int e2;
  double m = frexp(a, &e2); /* a = m * 2^e2, m in [0.5, 1) */
  int e = e2 - 1;
  double mant = round_half_even((2.0 * m - 1.0) * 4.0);
  if (mant == 4.0) { mant = 0.0; e += 1; }
  int code = ((e + 15) << 2) | (int)mant;
  if (code > 0x7B) code = 0x7B;
  return (uint8_t)(sign | code);
}

static float e5m2_decode(uint8_t c) {
  int exp_bits = (c >> 2) & 0x1F;
  int man = c & 0x3;
  double v;
  if (exp_bits == 0x1F) return man ? NAN : ((c & 0x80) ? -INFINITY : INFINITY);
  if (exp_bits == 0) v = ldexp((double)man, -16);
  else v = ldexp(1.0 + man / 4.0, exp_bits - 15);
  return (float)((c & 0x80) ? -v : v);
}

static double e8m0_decode(uint8_t c) { return ldexp(1.0, (int)c - 127); }

static int mx_emax(int fmt) { return fmt == 0 ? 8 : (fmt == 1 ? 15 : 2); }

/* Reading M1: the E8M0 code of a block with maximum magnitude amax. */
static uint8_t mx_scale_code(double amax, int fmt) {
  int exponent = -127;
  if (amax > 0.0) {
    int e2;
    frexp(amax, &e2); /* amax = m * 2^e2 with m in [0.5, 1): floor(log2(amax)) = e2 - 1 */
    exponent = (e2 - 1) - mx_emax(fmt);
  }
  if (exponent < -127) exponent = -127;
  if (exponent > 127) exponent = 127;
  return (uint8_t)(exponent + 127);
}

/* Reading M2: one element, t = v / X. The division by a power of two is exact in double; the
 * cast to float is exact too unless t lies far below every format's smallest subnormal
 * (2^-16), where it rounds to a float that encodes to zero all the same. */
static uint8_t mx_encode(double t, int fmt) {
  float f = (float)t;
  if (fmt == 0) return e4m3_encode_rn_satfinite(f);
  if (fmt == 1) return e5m2_encode_rn_satfinite(f);
  return e2m1_encode_rn_satfinite(f);
}

static double mx_decode(uint8_t code, int fmt) {
  if (fmt == 0) return e4m3_decode(code);
  if (fmt == 1) return e5m2_decode(code);
  return e2m1_decode(code);
}

/* One 32-element block: its E8M0 code and element codes (FP8: 32 bytes; FP4: 16 bytes). */
static void mx_quantize_block32(const double v[32], int fmt, uint8_t* codes, uint8_t* scale) {
  double amax = 0.0;
  for (int i = 0; i < 32; i++)
    if (fabs(v[i]) > amax) amax = fabs(v[i]);
  uint8_t s = mx_scale_code(amax, fmt);
  double X = e8m0_decode(s);
  *scale = s;
  for (int i = 0; i < 32; i++) {
    uint8_t q = mx_encode(v[i] / X, fmt);
    if (fmt == 2) {
      if (i % 2 == 0) codes[i / 2] = q;
      else codes[i / 2] |= (uint8_t)(q << 4);
    } else {
      codes[i] = q;
    }
  }
}

ORACLE_API uint8_t oracle_e5m2_encode(float v) { return e5m2_encode_rn_satfinite(v); }
ORACLE_API float oracle_e5m2_decode(uint8_t c) { return e5m2_decode(c); }
ORACLE_API double oracle_e8m0_decode(uint8_t c) { return e8m0_decode(c); }
ORACLE_API uint8_t oracle_mx_scale(double amax, int32_t fmt) { return mx_scale_code(amax, fmt); }
ORACLE_API uint8_t oracle_mx_encode(double t, int32_t fmt) { return mx_encode(t, fmt); }
ORACLE_API double oracle_mx_decode(uint8_t code, int32_t fmt) { return mx_decode(code, fmt); }

/* Rowwise MX quantization of BF16 x [M][N] (N % 32 == 0). Reading M3. */
ORACLE_API void oracle_mx_quantize_rowwise(const uint16_t* x, int64_t M, int64_t N, int32_t fmt,
                                           uint8_t* codes, uint8_t* scales) {
  const int64_t code_row = fmt == 2 ? N / 2 : N;
  const int64_t bytes_per_block = fmt == 2 ? 16 : 32;
  for (int64_t m = 0; m < M; m++) {
    for (int64_t b = 0; b < N / 32; b++) {
      double v[32];
      for (int i = 0; i < 32; i++) v[i] = bf16_to_f32(x[m * N + 32 * b + i]);
      mx_quantize_block32(v, fmt, codes + m * code_row + b * bytes_per_block,
                          scales + m * (N / 32) + b);
    }
  }
}

/* Columnwise MX quantization: the blocks are 32 consecutive rows of one column (M % 32 == 0);
 * column n's codes and scales form row n of the transposed outputs. Reading M3. */
ORACLE_API void oracle_mx_quantize_colwise(const uint16_t* x, int64_t M, int64_t N, int32_t fmt,
                                           uint8_t* codes, uint8_t* scales) {
  const int64_t code_row = fmt == 2 ? M / 2 : M;
  const int64_t bytes_per_block = fmt == 2 ? 16 : 32;
  for (int64_t n = 0; n < N; n++) {
    for (int64_t b = 0; b < M / 32; b++) {
      double v[32];
      for (int i = 0; i < 32; i++) v[i] = bf16_to_f32(x[(32 * b + i) * N + n]);
      mx_quantize_block32(v, fmt, codes + n * code_row + b * bytes_per_block,
                          scales + n * (M / 32) + b);
    }
  }
}

/* MX dequantization: x_hat = decode(q) * 2^(s - 127), exact in double, stored as float.
 * codes [R][C] (FP8) or [R][C/2] (FP4), scales [R][C/32], out [R][C]. */
ORACLE_API void oracle_mx_dequantize(const uint8_t* codes, const uint8_t* scales, int32_t fmt,
                                     int64_t R, int64_t C, float* out) {
  for (int64_t r = 0; r < R; r++) {
    for (int64_t c = 0; c < C; c++) {
      uint8_t q;
      if (fmt == 2) {
        uint8_t byte = codes[r * (C / 2) + c / 2];
        q = (c % 2 == 0) ? (byte & 0xF) : (byte >> 4);
      } else {
        q = codes[r * C + c];
      }
      out[r * C + c] = (float)(mx_decode(q, fmt) * e8m0_decode(scales[r * (C / 32) + c / 32]));
    }
  }
}
