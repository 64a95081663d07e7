/*
 * nvfp4.h -- C ABI of libnvfp4: NVFP4 block-scaled quantization of BF16 tensors on one
 * NVIDIA GB300 GPU (sm_103a).
 *
 * The operation is the one described on the page "[nvfp4_training] Optimize CuteDSL kernels
 * for NVFP4 training" (pytorch/ao pull request #4798), cited below as [PR4798] with its
 * section headings, and in the NVFP4 paragraph of the page "CuTeDSL at Perplexity":
 *   - a per-tensor FP32 amax and global scale (S_enc = 2688 / amax, S_dec = 1 / S_enc; 2688 is
 *     448, the largest E4M3 value, times 6, the largest E2M1 value; S_enc = 1 when amax = 0);
 *   - one FP8-E4M3 scale per 16-element block, s = E4M3((block_amax / 6) * S_enc);
 *   - every element multiplied by r = 1 / (float(s) * S_dec) (correctly rounded; r = 0 for a
 *     zero scale) and rounded to E2M1 (FP4: 0, +-0.5, +-1, +-1.5, +-2, +-3, +-4, +-6), by
 *     round-to-nearest-even or by stochastic rounding ([PR4798] "Optimization" items 1 and 3,
 *     "Fast math": this library implements the exact mode);
 *   - codes packed two per byte, the even element in the low nibble.
 *
 * Layouts (all row-major, all buffers owned and allocated by the caller):
 *   x            BF16 [M][N]                          (2 bytes per element)
 *   row codes    uint8 [M][N/2],  row scales  uint8 (E4M3) [M][N/16]
 *   col codes    uint8 [N][M/2],  col scales  uint8 (E4M3) [N][M/16]   (the transposed tensor)
 *   gscale       float [2] = {amax, S_dec}               (grouped: float [E][2])
 * Columnwise blocks run along M (16 consecutive rows of one column); their outputs are the
 * rowwise outputs of x transposed, optionally after a 16-point random Hadamard transform.
 *
 * Execution: every call is asynchronous on the caller's stream (a cudaStream_t passed as
 * void*; NULL is the legacy default stream). The quantize, amax and MX kernels are launched
 * with programmatic dependent launch: each waits for the previous kernel in the stream before
 * it touches memory, and lets the next kernel launched that way start early, so a kernel of
 * the caller's launched after them with programmatic dependent launch must wait
 * (cudaGridDependencySynchronize) before it reads their outputs, as that mechanism requires. Pointers marked (device) must be device (or
 * managed) memory, 16-byte aligned. The return value reports argument checks and launch
 * errors only; problems the device detects (bad grouped offsets, a bounded wait that gave up)
 * are recorded in a per-device status word read by nvfp4_get_status. A call rejected by its
 * argument checks launched nothing and wrote nothing. NVFP4_ERR_CUDA reports a CUDA call or
 * launch that failed (the runtime's last-error state is cleared; a sticky error stays); kernels
 * of the call launched before it may have run, so its outputs are undefined.
 *
 * Memory: the library allocates no memory on these calls except once per device, on the
 * first call that needs it: a small workspace (status word, the single-launch amax's counts,
 * maxima words and claim bits; 16 KiB) allocated with cudaMalloc and kept until exit. Make that
 * first call outside CUDA-graph capture. Launches take no host-side state from call to call,
 * so a captured call replays correctly (the single-launch amax included). The host pipeline (end of this file) allocates its
 * device staging when it is created, and nothing when work is submitted.
 */
#ifndef NVFP4_H
#define NVFP4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum nvfp4_status {
  NVFP4_OK = 0,
  NVFP4_ERR_INVALID_ARG = 1,   /* NULL pointer where one is required, negative size, bad enum */
  NVFP4_ERR_SHAPE = 2,         /* a dimension is not a multiple of 16 where blocks need it */
  NVFP4_ERR_ALIGN = 3,         /* a pointer or row pitch is not 16-byte aligned */
  NVFP4_ERR_UNSUPPORTED = 4,   /* an option combination the method does not define */
  NVFP4_ERR_CUDA = 5,          /* a CUDA runtime call or a kernel launch failed */
  NVFP4_ERR_DEVICE_STATUS = 6, /* the device flagged its input (nvfp4_get_status) */
  NVFP4_ERR_TIMEOUT = 7        /* a bounded device-side wait gave up (nvfp4_get_status) */
} nvfp4_status;

typedef enum nvfp4_rounding {
  NVFP4_ROUND_RN = 0,          /* round to nearest, ties to even */
  NVFP4_ROUND_SR = 1           /* stochastic rounding driven by Philox4x32-10 */
} nvfp4_rounding;

/* Device status bits (nvfp4_get_status). */
#define NVFP4_DEVICE_BAD_OFFSETS 0x1u  /* grouped offsets not non-decreasing within [0, T],
                                          or padded token total above the column capacity */
#define NVFP4_DEVICE_TIMEOUT     0x2u  /* the wait for every CTA's amax or a copy wait passed
                                          its limit */

/* Options of one quantization. Zero-initialise and set what is needed. */
typedef struct nvfp4_config {
  int32_t rowwise;        /* produce rowwise codes/scales (1x16 blocks along N) */
  int32_t columnwise;     /* produce columnwise codes/scales (1x16 blocks along M, transposed) */
  int32_t block2d;        /* one scale per 16x16 tile shared by both orientations, written
                             replicated into both scale tensors ([PR4798] "Optimization"
                             item 2, the 2D weight kernel); RTNE only, no RHT */
  int32_t round_row;      /* nvfp4_rounding of the rowwise codes */
  int32_t round_col;      /* nvfp4_rounding of the columnwise codes */
  int32_t rht_col;        /* apply the 16-point random Hadamard transform to each columnwise
                             block before quantizing: y = bf16(0.25 * H16 (d * v)), H16 the
                             Sylvester Hadamard matrix, d the sign vector below ([PR4798]
                             "Optimization" items 2 and 5, "Fast math": the accumulator is
                             rounded through BF16 in exact mode) */
  uint32_t rht_sign_mask; /* bit i set: d_i = -1 (bits 16..31 must be zero) */
  uint32_t rng_offset;    /* Philox counter word 3 (advance it to draw a new stream) */
  uint64_t rng_seed;      /* Philox key = (low 32 bits, high 32 bits) */
  int32_t fused_amax;     /* when the amax inputs are NULL: 0 = amax pass + quantize pass,
                             1 = one launch: every CTA (one per SM) reduces its share of the
                             tiles, folds the maxima into the workspace with an atomic max,
                             counts the share as arrived and waits (bounded) for every share,
                             then quantizes those tiles (the re-read of x comes from L2 when x
                             fits there). No CTA waits for another to start: a CTA that has
                             waited 20 us claims any share that no CTA has started and
                             computes it itself, so the call also completes when some SMs are
                             held by other work (another stream's kernels, a reduced MPS share,
                             a green context), only more slowly. Launched with programmatic
                             dependent launch: it waits for the previous kernel in the stream
                             before it reads anything, and a kernel launched after it that way
                             may start before it ends and must wait for it before reading its
                             outputs. Fused calls share the device workspace's counts, maxima
                             and claim bits (kept on the device: the last CTA to finish with
                             them readies them for the next launch, so captured calls replay
                             correctly): on one device they must not overlap in time (issue
                             them on one stream). Plain tensors only. */
  int32_t fast_math;      /* 0 = exact (default). 1 = the fast variant of [PR4798] "Fast math":
                             the element multiplier is rcp.approx.ftz(float(s) * S_dec) instead
                             of the correctly rounded reciprocal, and the columnwise RHT output
                             is quantized from its FP32 value without the BF16 round-through.
                             Not bit-defined (the approximate reciprocal is the hardware's);
                             dequantized, it stays above 25 dB SQNR against the exact mode's
                             output; with round-to-nearest a code moves by at most one E2M1
                             step. The amax, the global scales and 2D (block2d) quantization
                             stay exact. Other values:
                             NVFP4_ERR_INVALID_ARG. */
  int32_t swizzle_scales; /* 0 = row-major scale outputs (default). 1 = both scale outputs in the
                             128 x 4 tiled layout the tensor-core block-scaled (NVFP4) GEMMs
                             read, the one nvfp4_swizzle_scales writes (see there), written by
                             the quantize kernel itself ([PR4798] "Config surface and AUTO":
                             the reference's columnwise scale store is hardwired to it): the
                             scale matrix [R][C] (rowwise R = M, C = N/16; columnwise R = N,
                             C = M/16) zero-padded to whole 128 x 4 tiles, so the buffers hold
                             ceil(R/128) * ceil(C/4) * 512 bytes. nvfp4_quantize and
                             nvfp4_quantize_noalloc only (grouped calls and the host pipeline:
                             NVFP4_ERR_UNSUPPORTED). When R or C is not a multiple of 128 or 4
                             the call first zeroes the buffers (one memset each). Other values:
                             NVFP4_ERR_INVALID_ARG. */
} nvfp4_config;

/* Stochastic rounding ([PR4798] "Optimization" item 3 and "Correctness"): one Philox4x32-10
 * draw per 16-element block with key (lo32 seed, hi32 seed) and counter (lo32 b, hi32 b, tag,
 * rng_offset), b the block's linear index in its scale tensor ([M][N/16] rowwise, [N][M/16]
 * columnwise; grouped columnwise: [H][capacity/16]), tag 0 rowwise and 1 columnwise. Word j
 * of the draw is the random operand of the cvt.rs.satfinite.e2m1x4.f32 that converts elements
 * 4j..4j+3 of the block. The stream is a pure function of (seed, offset, block position). */

/* Text for a status code (static storage). */
const char* nvfp4_status_string(nvfp4_status status);

/* Per-tensor absolute maxima ([PR4798] "Optimization" item 5: the amax and RHT-amax kernels,
 * "always exact").
 *   x        (device) BF16 [M][N], 16-byte aligned; N % 16 == 0 (M % 16 == 0 with rht_col).
 *   cfg      rht_col / rht_sign_mask select what amax_col measures.
 *   amax_row (device) float[1] or NULL: receives max |x|.
 *   amax_col (device) float[1] or NULL: receives max |y| over the RHT output y of every
 *            16-row column block when cfg->rht_col, else max |x|.
 * M == 0 or N == 0 writes 0. */
nvfp4_status nvfp4_amax(const void* x, int64_t M, int64_t N, const nvfp4_config* cfg,
                        float* amax_row, float* amax_col, void* stream);

/* Quantize one BF16 tensor, rowwise and/or columnwise, from one read of x.
 *   x                   (device) BF16 [M][N]; N % 16 == 0; M % 16 == 0 when columnwise or
 *                       block2d.
 *   amax_row, amax_col  (device) float[1] each, or NULL to compute them inside this call
 *                       (amax_col is the RHT amax when cfg->rht_col). With block2d both
 *                       orientations use amax_row.
 *   row_codes [M][N/2], row_scales [M][N/16], row_gscale [2]: (device) outputs, required when
 *                       cfg->rowwise (or block2d with rowwise), else ignored.
 *   col_codes [N][M/2], col_scales [N][M/16], col_gscale [2]: (device) outputs, required when
 *                       cfg->columnwise, else ignored.
 * Errors: NVFP4_ERR_UNSUPPORTED for block2d with RHT or SR, or neither orientation selected;
 * NVFP4_ERR_SHAPE / _ALIGN for the shape and alignment rules above. */
nvfp4_status nvfp4_quantize(const void* x, int64_t M, int64_t N, const nvfp4_config* cfg,
                            const float* amax_row, const float* amax_col,
                            uint8_t* row_codes, uint8_t* row_scales, float* row_gscale,
                            uint8_t* col_codes, uint8_t* col_scales, float* col_gscale,
                            void* stream);

/* Per-expert absolute maxima of a grouped tensor ([PR4798] "Performance": the grouped amax
 * kernel), the amax pass that nvfp4_quantize_grouped runs internally, exposed on its own.
 *   offsets, E as nvfp4_quantize_grouped; H % 16 == 0.
 *   amax_row (device) float[E] or NULL: max |x| over each expert's rows.
 *   amax_col (device) float[E] or NULL: with cfg->rht_col, max |y| over the RHT output of each
 *            expert's zero-padded 16-row column blocks; else max |x|.
 * Bad offsets set NVFP4_DEVICE_BAD_OFFSETS (nvfp4_get_status). */
nvfp4_status nvfp4_amax_grouped(const void* x, int64_t T, int64_t H, const int32_t* offsets,
                                int32_t E, const nvfp4_config* cfg, float* amax_row,
                                float* amax_col, void* stream);

/* Grouped (MoE) quantization of a packed [T][H] tensor whose rows are split among E experts
 * by device-side cumulative offsets ([PR4798] "Grouped allocation tail", "Config surface and
 * AUTO": a packed tensor plus device-side offsets; rows past offsets[E-1] are not read or
 * written).
 *   offsets      (device) int32 [E], non-decreasing, offsets[E-1] <= T; expert e owns rows
 *                [offsets[e-1], offsets[e]) with offsets[-1] = 0 (empty experts allowed).
 *   E            1 <= E <= 256.
 *   amax_row, amax_col  (device) float[E] each (per-expert amax, e.g. from
 *                nvfp4_amax_grouped or a producer's epilogue), or NULL to compute them inside
 *                this call (amax_col is the RHT amax when cfg->rht_col). With block2d both
 *                orientations use amax_row.
 *   col_capacity columns of the columnwise outputs, a multiple of 16, >= sum_e pad16(n_e)
 *                (pad16 rounds a token count up to a multiple of 16). A multiple of 32 keeps
 *                every columnwise row 16-byte aligned, so that the kernel's whole tiles leave
 *                by TMA store; an odd multiple of 16 takes per-thread stores (slower). Expert e's columnwise
 *                block starts at column sum_{j<e} pad16(n_j); its last partial 16-token block
 *                is zero-padded before the transform and stored in full.
 *   Per expert: amax over its rows and global scale for the rowwise side; RHT amax (or amax)
 *   over its zero-padded blocks for the columnwise side. Outputs:
 *   row_codes [T][H/2], row_scales [T][H/16], row_gscale [E][2];
 *   col_codes [H][col_capacity/2], col_scales [H][col_capacity/16], col_gscale [E][2].
 * block2d (stacked expert weights, the pages' grouped 2D weight quantize): each expert's 16x16
 *   tiles start at its first row, its last row tile zero-padded; one amax and global scale per
 *   expert for both orientations; no RHT or SR (NVFP4_ERR_UNSUPPORTED).
 * H % 16 == 0. fused_amax is not supported here. Offsets that break the rules above set
 * NVFP4_DEVICE_BAD_OFFSETS and the kernels write no codes. */
nvfp4_status nvfp4_quantize_grouped(const void* x, int64_t T, int64_t H,
                                    const int32_t* offsets, int32_t E, int64_t col_capacity,
                                    const nvfp4_config* cfg,
                                    const float* amax_row, const float* amax_col,
                                    uint8_t* row_codes, uint8_t* row_scales, float* row_gscale,
                                    uint8_t* col_codes, uint8_t* col_scales, float* col_gscale,
                                    void* stream);

/* Dequantize codes back to FP32: out[r][c] = (e2m1(code) * e4m3(scale[r][c/16])) * S_dec,
 * S_dec = gscale[1] (the check used by the reconstruction tests of [PR4798] "Correctness").
 *   codes (device) [R][C/2], scales (device) [R][C/16], gscale (device) float[2],
 *   out (device) float [R][C]; C % 16 == 0. Columnwise outputs dequantize with R = N, C = M. */
nvfp4_status nvfp4_dequantize(const uint8_t* codes, const uint8_t* scales, const float* gscale,
                              int64_t R, int64_t C, float* out, void* stream);

/* Dequantization for checks at the GEMM boundary ([PR4798]: columnwise operands carry the
 * 16-point RHT, "Config surface and AUTO"; the reconstruction of "Correctness"): as
 * nvfp4_dequantize, then
 *   inverse_rht = 1: every 16-element block of a row (a columnwise output: 16 consecutive
 *     tokens of one column) goes through the inverse transform v = d * (0.25 * FWHT16(y)),
 *     d_i = -1 where bit i of rht_sign_mask is set, binary32 butterflies in stages 1, 2, 4, 8
 *     (0.25 H16 is its own inverse), which returns the pre-transform column up to the
 *     quantization error;
 *   out_bf16 = 1: out is BF16 [R][C] (round to nearest-even), else float [R][C].
 * out 16-byte aligned, codes 8-byte aligned; C % 16 == 0. Errors: NVFP4_ERR_INVALID_ARG for
 * flags other than 0/1, a mask above 0xFFFF or NULL buffers; NVFP4_ERR_SHAPE; NVFP4_ERR_ALIGN. */
nvfp4_status nvfp4_dequantize_ex(const uint8_t* codes, const uint8_t* scales, const float* gscale,
                                 int64_t R, int64_t C, int32_t inverse_rht, uint32_t rht_sign_mask,
                                 int32_t out_bf16, void* out, void* stream);

/* nvfp4_quantize with fused_amax, for callers that cannot allocate device memory: code that
 * runs inside a memory allocator's own callbacks, a latency-critical path that must never
 * reach cudaMalloc (it can synchronize the whole device), or a host that gives this library a
 * fixed memory budget. The pages have no counterpart of this entry point; it exists only so
 * that such callers get the single-launch path.
 * It allocates nothing: no cudaMalloc, no cudaFree, no allocating library routine. Its scratch
 * -- a status word, the single-launch amax's counts, two maxima words and one claim bit per
 * CTA, 256 bytes in all -- is a static device array that every GPU loading this library holds
 * until exit. The caller still passes x and every output.
 *   Arguments, layouts and shape rules as nvfp4_quantize with amax_row = amax_col = NULL and
 *   cfg->fused_amax = 1 (cfg->fused_amax itself is ignored); M and N must be positive.
 *   The first call on a device looks up the array's device address and prepares the kernels
 *   (no allocation): make that first call before any stream capture.
 *   A device whose launch would need more than 1024 CTAs (one claim bit each) is refused with
 *   NVFP4_ERR_UNSUPPORTED (GB300 launches one CTA per SM, 152).
 *   Every call on a device shares the array: calls that overlap on the GPU race (issue them on
 *   one stream). The array is zero when the library loads and the last CTA of each launch to
 *   finish with the counts readies them for the next, so nothing needs clearing between calls
 *   and a captured call replays correctly. A wait that gives up is recorded in the array's own
 *   status word: read it with nvfp4_noalloc_get_status (nvfp4_get_status reads the regular
 *   workspace's). */
nvfp4_status nvfp4_quantize_noalloc(const void* x, int64_t M, int64_t N, const nvfp4_config* cfg,
                                    uint8_t* row_codes, uint8_t* row_scales, float* row_gscale,
                                    uint8_t* col_codes, uint8_t* col_scales, float* col_gscale,
                                    void* stream);

/* The status word of nvfp4_quantize_noalloc's array on the current device, without allocating
 * (the pages have no counterpart): synchronize `stream`, then read and clear the word with
 * synchronous copies from and to the array itself. *device_status receives the NVFP4_DEVICE_*
 * bits that the no-alloc calls recorded since the last read. Returns NVFP4_ERR_TIMEOUT when a
 * wait of one of those calls gave up (its outputs are then incomplete), NVFP4_OK when no bit
 * was set. Errors: NVFP4_ERR_INVALID_ARG (NULL device_status), NVFP4_ERR_CUDA. */
nvfp4_status nvfp4_noalloc_get_status(void* stream, uint32_t* device_status);

/* Scale bytes in the layout the tensor-core block-scaled (NVFP4) GEMMs read, e.g. cuBLASLt's
 * ([PR4798] "Config surface and AUTO": the reference's columnwise scale store is hardwired to
 * this swizzled layout; the layout is the 1D block-scaling-factor layout of the cuBLAS
 * documentation).
 *   scales (device) uint8 [R][C], row-major, as the quantize calls write them (rowwise:
 *          R = M, C = N/16; columnwise: R = N, C = M/16).
 *   out    (device) uint8 [ceil(R/128) * ceil(C/4) * 512], 16-byte aligned: 128 x 4 tiles of
 *          the zero-padded matrix in row-major tile order, 512 bytes each; inside a tile the
 *          scale of row r, column c is byte (r % 32) * 16 + ((r % 128) / 32) * 4 + (c % 4).
 * The codes need no change: [R][C*8] bytes, two E2M1 codes per byte, the even element in the
 * low nibble, is the packed FP4 operand those GEMMs take (the global scales S_dec of both
 * operands multiply the product). */
nvfp4_status nvfp4_swizzle_scales(const uint8_t* scales, int64_t R, int64_t C, uint8_t* out,
                                  void* stream);

/* A producer with the amax in its epilogue ([Perplexity] "CuTeDSL at Perplexity", its RMS-norm
 * kernel): y = bf16_rne((w + weight_bias) * (x * rms)), rms = rsqrt(sum(x^2) / N + eps) per row,
 * every step one IEEE binary32 operation (the reciprocal square root correctly rounded); the
 * sum of squares as that kernel takes it (lane l of a warp sums its 8-element vectors l, l + 32,
 * ... in order, then a butterfly of shuffles, xor 16 .. 1). The epilogue writes amax =
 * max |y| over the tensor, so that nvfp4_quantize(y, amax_row = amax, ...) needs no amax pass.
 *   x (device) BF16 [M][N], weight (device) BF16 [N], y (device) BF16 [M][N]: 16-byte aligned,
 *   N % 8 == 0; amax (device) float[1], zeroed on `stream` before the kernel.
 * Errors: NVFP4_ERR_INVALID_ARG (NULL buffers, negative sizes, non-finite eps or bias),
 * NVFP4_ERR_SHAPE, NVFP4_ERR_ALIGN, NVFP4_ERR_CUDA. */
nvfp4_status nvfp4_rmsnorm_amax(const void* x, const void* weight, int64_t M, int64_t N,
                                float eps, float weight_bias, void* y, float* amax, void* stream);

/* nvfp4_rmsnorm_amax, then nvfp4_quantize of y with that amax (N % 16 == 0): two launches
 * instead of norm, amax pass and quantize. With rht_col the columnwise amax (that of the
 * transformed columns) still comes from an amax pass over y. Outputs and errors as
 * nvfp4_quantize. */
nvfp4_status nvfp4_rmsnorm_quantize(const void* x, const void* weight, int64_t M, int64_t N,
                                    float eps, float weight_bias, const nvfp4_config* cfg,
                                    void* y, float* amax, uint8_t* row_codes, uint8_t* row_scales,
                                    float* row_gscale, uint8_t* col_codes, uint8_t* col_scales,
                                    float* col_gscale, void* stream);

/* MX formats ([Perplexity] "CuTeDSL at Perplexity", its Blackwell paragraph: MXFP8 and MXFP4
 * beside NVFP4, with block maxima over 32 elements). Blocks of 32 consecutive elements share a
 * power-of-two scale stored as E8M0 (value 2^(code - 127)); there is no tensor-wide scale.
 * The scale and rounding rules are the OCP Microscaling Formats v1.0 conversion: exponent =
 * floor(log2(block max)) - emax, emax = 8 (E4M3), 15 (E5M2), 2 (E2M1), at least -127 (an
 * all-zero block gets code 0); elements are x / 2^exponent rounded to nearest-even, saturating
 * at the format's largest magnitude (448, 57344, 6). Inputs must be finite. */
typedef enum {
  NVFP4_MX_E4M3 = 0, /* MXFP8, E4M3 elements, one byte each */
  NVFP4_MX_E5M2 = 1, /* MXFP8, E5M2 elements, one byte each */
  NVFP4_MX_E2M1 = 2  /* MXFP4, E2M1 elements, two per byte, the even element in the low nibble */
} nvfp4_mx_format;

/* MX quantization of a BF16 [M][N] row-major device tensor in one pass (no amax).
 *   rowwise    (N % 32 == 0): row_codes [M][N] (FP8) or [M][N/2] (FP4), row_scales [M][N/32].
 *   columnwise (M % 32 == 0, N % 8 == 0): the transposed tensor's, col_codes [N][M] or
 *              [N][M/2], col_scales [N][M/32] (blocks are 32 consecutive rows of a column).
 * Alignment: x 16 bytes; code buffers 32 bytes (FP8) or 16 bytes (FP4); row_scales 4 bytes.
 * Buffers of an orientation not selected may be NULL. Asynchronous on `stream`; an empty
 * tensor returns NVFP4_OK without a launch. Errors: NVFP4_ERR_INVALID_ARG (format, NULL
 * buffers, negative sizes), NVFP4_ERR_UNSUPPORTED (neither orientation), NVFP4_ERR_SHAPE,
 * NVFP4_ERR_ALIGN, NVFP4_ERR_CUDA; a device-side wait that gives up sets NVFP4_DEVICE_TIMEOUT. */
nvfp4_status nvfp4_mx_quantize(const void* x, int64_t M, int64_t N, int32_t format,
                               int32_t rowwise, int32_t columnwise, uint8_t* row_codes,
                               uint8_t* row_scales, uint8_t* col_codes, uint8_t* col_scales,
                               void* stream);

/* out[r][c] = element(code) * 2^(scale - 127) in binary32 (one rounding of the exact product)
 * for codes [R][C] (FP8) or [R][C/2] (FP4) and scales [R][C/32]; C % 32 == 0; codes and out
 * 16-byte aligned. */
nvfp4_status nvfp4_mx_dequantize(const uint8_t* codes, const uint8_t* scales, int32_t format,
                                 int64_t R, int64_t C, float* out, void* stream);

/* The per-device workspace: the status word the kernels report to, and the counts, maxima and
 * claim bits of the single-launch amax. By default the library allocates it with cudaMalloc
 * (once per device, on the first call that needs it, zeroed) and never frees it. */
#define NVFP4_WORKSPACE_BYTES 16384

/* Use caller-owned device memory as the current device's workspace instead, e.g. memory from
 * the caller's own allocator, set up before stream capture so that no later call allocates.
 *   workspace (device) at least NVFP4_WORKSPACE_BYTES, 256-byte aligned; NULL returns to the
 *   library's own workspace. The library zeroes it (synchronously: the call waits for the
 *   device) and uses it for every later call on this device; the caller keeps it alive while
 *   any call may use it, and calls this only when no work of the library is in flight on the
 *   device.
 * Errors: NVFP4_ERR_INVALID_ARG (bytes below NVFP4_WORKSPACE_BYTES), NVFP4_ERR_ALIGN,
 * NVFP4_ERR_CUDA. */
nvfp4_status nvfp4_set_workspace(void* workspace, size_t bytes);

/* Synchronize `stream`, then read and clear the current device's status word into
 * *device_status (NVFP4_DEVICE_* bits). Returns NVFP4_ERR_DEVICE_STATUS or NVFP4_ERR_TIMEOUT
 * when bits were set, NVFP4_OK otherwise. */
nvfp4_status nvfp4_get_status(void* stream, uint32_t* device_status);

/* Test hook for the bounded wait of the single-launch amax: the next call that takes the
 * single-launch path (nvfp4_quantize or nvfp4_quantize_noalloc, on any device) waits for
 * `extra` arrivals more than its grid has shares. With extra > 0 no launch can reach that
 * count, so every CTA gives up after its bounded wait (about 2 s), stores nothing, sets
 * NVFP4_DEVICE_TIMEOUT and exits; the last CTA to finish still readies the counts for the next
 * launch, so the next call runs normally. The hook is consumed by that one call (0 clears it).
 * Not for production use. Errors: NVFP4_ERR_INVALID_ARG (extra outside 0 .. 1024). */
nvfp4_status nvfp4_debug_fused_extra_arrivals(int32_t extra);

/* Test hook for the take-over of shares: in the next single-launch call (as above), the last
 * `count` CTAs of the grid hold back before they claim their own shares until every share has
 * arrived (bounded, about 2 s), as if their SMs were busy with other work. The other CTAs then
 * take those shares over after their 20 us wait, and the held-back CTAs find their shares
 * taken. The outputs are those of a normal call. Consumed by that one call (0 clears it). Not
 * for production use. Errors: NVFP4_ERR_INVALID_ARG (count outside 0 .. 1024). */
nvfp4_status nvfp4_debug_fused_late_ctas(int32_t count);

/* Synchronize `stream`, then read and clear the count of shares that single-launch calls on
 * the current device's workspace have taken over from CTAs that had not claimed them yet
 * (statistics for tests; nvfp4_quantize_noalloc's calls are not counted). Errors:
 * NVFP4_ERR_INVALID_ARG (NULL count), NVFP4_ERR_CUDA. */
nvfp4_status nvfp4_debug_fused_takeovers(void* stream, uint32_t* count);

/* Test hook for launch failures: with on = 1, the next nvfp4_quantize or nvfp4_quantize_grouped
 * call (on any device) launches its quantize kernel with an empty grid, which the runtime
 * rejects before anything reaches the GPU; the call returns NVFP4_ERR_CUDA and the next call
 * runs normally. on = 0 clears it. Not for production use.
 * Errors: NVFP4_ERR_INVALID_ARG (on not 0 or 1). */
nvfp4_status nvfp4_debug_fail_next_launch(int32_t on);

/* Host pipeline: quantization of tensors that live in host memory, with the copies of
 * consecutive submissions overlapped (the input of one on the host-to-device link while the
 * outputs of the previous one use the device-to-host direction). Runtime plumbing around
 * nvfp4_quantize; the pages have no counterpart.
 * A pipeline owns `depth` (1 to 4) slots of device staging (x and every output of one tensor
 * of the shape given at creation), three CUDA streams (copy in, compute, copy out) and events.
 * Submission i uses slot i % depth: copy x in once the slot's previous input has been read,
 * quantize (nvfp4_quantize on the compute stream, with fused_amax as configured) once the
 * copy landed and the slot's previous outputs have been copied out, copy the outputs out.
 * Host buffers should be page-locked (cudaHostAlloc / torch pin_memory): pageable memory
 * works, without overlap. Host outputs are written in submission order; the caller must not
 * touch a submission's host buffers until a join has been waited for. One host thread drives
 * a pipeline at a time. All submissions run on the device that was current at creation. */
typedef struct nvfp4_host_pipeline nvfp4_host_pipeline;

/* Create a pipeline for BF16 [M][N] tensors quantized with *cfg (copied; the rounding seed
 * and offset stay fixed for every submission). Allocates the staging with cudaMalloc.
 * Shape and option rules as nvfp4_quantize, with M, N > 0. *out receives the handle. */
nvfp4_status nvfp4_host_pipeline_create(int64_t M, int64_t N, const nvfp4_config* cfg,
                                        int32_t depth, nvfp4_host_pipeline** out);

/* Enqueue one tensor: x_host (host) BF16 [M][N]; outputs (host) as nvfp4_quantize's, NULL for
 * an orientation the configuration does not produce. The work starts after everything already
 * enqueued on `stream` (the caller's stream at submission time). Returns without waiting. */
nvfp4_status nvfp4_host_pipeline_submit(nvfp4_host_pipeline* p, const void* x_host,
                                        uint8_t* row_codes, uint8_t* row_scales,
                                        float* row_gscale, uint8_t* col_codes,
                                        uint8_t* col_scales, float* col_gscale, void* stream);

/* The same for grouped tensors: BF16 [T][H] with E experts (1 <= E <= 256), quantized by
 * nvfp4_quantize_grouped with *cfg (fused_amax 0: NVFP4_ERR_UNSUPPORTED otherwise) and
 * col_capacity columns of columnwise outputs (a multiple of 16 when cfg->columnwise); each
 * slot also stages the submission's E offsets. Shape rules as nvfp4_quantize_grouped. */
nvfp4_status nvfp4_host_pipeline_create_grouped(int64_t T, int64_t H, int32_t E,
                                                int64_t col_capacity, const nvfp4_config* cfg,
                                                int32_t depth, nvfp4_host_pipeline** out);

/* Enqueue one grouped tensor: x_host (host) BF16 [T][H], offsets_host (host) int32 [E] (the
 * expert ends, rules as nvfp4_quantize_grouped's; copied in with x), outputs (host) as
 * nvfp4_quantize_grouped's. A pipeline created by nvfp4_host_pipeline_create takes only
 * nvfp4_host_pipeline_submit, one created by nvfp4_host_pipeline_create_grouped only this
 * call (NVFP4_ERR_INVALID_ARG otherwise). */
nvfp4_status nvfp4_host_pipeline_submit_grouped(nvfp4_host_pipeline* p, const void* x_host,
                                                const int32_t* offsets_host,
                                                uint8_t* row_codes, uint8_t* row_scales,
                                                float* row_gscale, uint8_t* col_codes,
                                                uint8_t* col_scales, float* col_gscale,
                                                void* stream);

/* Make `stream` wait (on the device) until every submitted tensor's outputs are in host
 * memory. Synchronize `stream` (or an event recorded after this call) before reading them. */
nvfp4_status nvfp4_host_pipeline_join(nvfp4_host_pipeline* p, void* stream);

/* Wait for all submitted work, then free the staging, streams and events. NULL is a no-op. */
nvfp4_status nvfp4_host_pipeline_destroy(nvfp4_host_pipeline* p);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4_H */
