// MX quantization (MXFP8 with E4M3 or E5M2 elements, MXFP4 with E2M1 elements) of BF16
// tensors: blocks of 32 elements along a row (rowwise) or a column (columnwise, written
// transposed) share one power-of-two scale stored as E8M0, and there is no tensor-wide scale.
// The page "CuTeDSL at Perplexity" (its Blackwell paragraph) names these formats beside NVFP4
// and their 32-element block maxima; the scale rule is the OCP Microscaling Formats v1.0
// conversion: exponent = floor(log2(block max)) - emax of the element format (8 for E4M3, 15
// for E5M2, 2 for E2M1), clamped below at -127; elements are x / 2^exponent rounded to
// nearest-even with saturation (cvt.rn.satfinite).
//
// No amax pass is needed, so this is one streaming pass over 32 x 128 units:
//   * a CTA round is eight vertically adjacent units (256 rows x 128 columns), warp w taking
//     the w-th; each warp keeps its next kMxStages units in flight in its own ring (two 32 x 64
//     TMA boxes per unit, 128-byte rows, 128-byte swizzle, bounded mbarrier waits);
//   * rowwise: lane l owns row l of the unit, four 32-element blocks of 16-byte chunks; the
//     swizzle puts the eight lanes of a shared-memory phase (rows l..l+7) on eight different
//     bank groups;
//   * columnwise: lane l owns four columns (8 bytes of a row of box l / 16), read down all 32
//     rows; a block is a lane-local column;
//   * the E8M0 exponent comes from the block maximum's exponent field (BF16 magnitudes order
//     like integers), the multiplier 2^-exponent is built from bits, and x * 2^-exponent is
//     exact, so a single cvt.rn.satfinite rounds each element once;
//   * codes are staged in shared memory in the swizzled layouts of the output boxes and leave
//     by TMA stores (row codes as 32 whole lines per unit; column codes through a 3D view of
//     the transposed output that keeps the staging writes free of bank conflicts);
//   * column scales: the CTA's eight units give each column eight consecutive scale bytes,
//     gathered in shared memory and written as one 8-byte word per column per round.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cuda_fp16.h>

#include <cstdint>

#include "nvfp4_device.cuh"
#include "aux_internal.h"
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

// 32 elements given as 16 packed BF16 pairs (element 2i in the low half of w[i]), times mult,
// to codes: FP8 -> o[0..7] (32 bytes), FP4 -> o[0..3] (16 bytes), element 0 first.
template <int FMT>
__device__ __forceinline__ void block_codes(const uint32_t (&w)[16], float mult, uint32_t (&o)[8]) {
  const uint64_t m2 = f2_pack(mult, mult);
  if (FMT == 2) {
#pragma unroll
    for (int q = 0; q < 4; q++)
      o[q] = e2m1x8_rn(f2_mul(f2_from_bf16x2(w[4 * q]), m2), f2_mul(f2_from_bf16x2(w[4 * q + 1]), m2),
                       f2_mul(f2_from_bf16x2(w[4 * q + 2]), m2),
                       f2_mul(f2_from_bf16x2(w[4 * q + 3]), m2));
  } else {
#pragma unroll
    for (int q = 0; q < 8; q++)
      o[q] = fp8x4<FMT>(f2_mul(f2_from_bf16x2(w[2 * q]), m2), f2_mul(f2_from_bf16x2(w[2 * q + 1]), m2));
  }
}

// Offset of byte `off` of a 1024-byte-aligned staging buffer of ROWB-byte rows under the TMA
// swizzle whose span is the row (128, 64 or 32 bytes: the 16-byte chunk index bits 4..6, 4..5
// or 4 XOR address bits 7..9, 7..8 or 7); 16-byte rows are not swizzled.
template <int ROWB>
__device__ __forceinline__ uint32_t swz(uint32_t off) {
  constexpr uint32_t mask = ROWB == 128 ? 0x70u : (ROWB == 64 ? 0x30u : (ROWB == 32 ? 0x10u : 0u));
  return off ^ ((off >> 3) & mask);
}

__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
               : "memory");
}

// A block's codes into staging of ROWB-byte rows: 32 bytes (FP8, two swizzled chunks) or 16
// bytes (FP4) at logical offset off (a multiple of the block's code bytes).
template <int FMT, int ROWB>
__device__ __forceinline__ void stage_block(uint32_t stbase, uint32_t off, const uint32_t (&o)[8]) {
  sts128(stbase + swz<ROWB>(off), o[0], o[1], o[2], o[3]);
  if (FMT != 2) sts128(stbase + swz<ROWB>(off + 16), o[4], o[5], o[6], o[7]);
}

// 2D tiled TMA store of a shared-memory box to (x, y) of the tensor, in the current bulk group;
// the parts of the box outside the tensor are not written.
__device__ __forceinline__ void tma_store_2d(const void* tensor_map, uint32_t smem_src, int32_t x,
                                             int32_t y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];"
               ::"l"(tensor_map), "r"(smem_src), "r"(x), "r"(y)
               : "memory");
}
// The same for a 3D box at (x, y, z).
__device__ __forceinline__ void tma_store_3d(const void* tensor_map, uint32_t smem_src, int32_t x,
                                             int32_t y, int32_t z) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];"
               ::"l"(tensor_map), "r"(smem_src), "r"(x), "r"(y), "r"(z)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// The shared memory of every committed store has been read (it may be written again).
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Every committed store is complete.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

template <int FMT, bool ROW, bool COL>
__global__ void __launch_bounds__(32 * kMxWarps, 1) mx_quantize_kernel(const __grid_constant__ MxArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  pdl_wait();  // launched with programmatic dependent launch: the previous kernel may produce x
  pdl_allow_next();
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  // the 128-byte swizzle is a function of the shared address bits 7..9: every box and staging
  // buffer starts on a 1024-byte boundary, so that it is row & 7 inside each box
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t* const gbase = smem_raw + (base - smem_u32(smem_raw));
  constexpr int kWarpBytes = kMxStages * kUnitBytes + kMxOutBytes;
  // per CTA, after the warps' areas: column-scale staging [2][kMxWarps][128], then mbarriers
  const uint32_t csst = base + (uint32_t)(kMxWarps * kWarpBytes);
  uint64_t* const full =
      reinterpret_cast<uint64_t*>(gbase + kMxWarps * kWarpBytes + 2 * kMxWarps * kMxUnitN) +
      warp * kMxStages;
  const uint32_t wstage = base + (uint32_t)(warp * kWarpBytes);
  // output staging: row codes [32][128 or 64 B], then column codes [4][32][32 or 16 B]
  constexpr uint32_t kRowOut = FMT == 2 ? 2048u : 4096u;
  const uint32_t rowst = wstage + (uint32_t)(kMxStages * kUnitBytes);
  const uint32_t colst = rowst + kRowOut;

  // A round of the CTA is a group of kMxWarps vertically adjacent units (kMxWarps x 32 rows,
  // 128 columns), warp w taking the w-th; the groups go round-robin over the CTAs, the 128-column
  // strips fastest. Warps past the tensor's last unit row have nothing to do in that round.
  const int64_t M = a.rows, N = a.cols;
  const int units_n = (int)((N + kMxUnitN - 1) / kMxUnitN);
  const int units_m = (int)((M + kMxUnitM - 1) / kMxUnitM);
  const int groups = ((units_m + kMxWarps - 1) / kMxWarps) * units_n;
  const int rounds = (int)blockIdx.x < groups ? (groups - (int)blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
  auto unit_of = [&](int i, int& mt, int& nt) {  // this warp's unit in round i; false: none
    const int gidx = blockIdx.x + i * gridDim.x;
    const int gq = gidx / units_n;
    nt = gidx - gq * units_n;
    mt = gq * kMxWarps + warp;
    return mt < units_m;
  };

  auto issue = [&](int mt, int nt, int s) {
    const int n0 = nt * kMxUnitN;
    uint8_t* dst = gbase + (size_t)warp * kWarpBytes + (size_t)s * kUnitBytes;
    // a second box wholly right of the tensor is not loaded: nothing of it is stored
    const bool two = (int64_t)n0 + 64 < N;
    mbar_expect_tx(&full[s], two ? kUnitBytes : kBoxBytes);
    tma_load_2d(dst, &a.tmap, n0, mt * kMxUnitM, &full[s]);
    if (two) tma_load_2d(dst + kBoxBytes, &a.tmap, n0 + 64, mt * kMxUnitM, &full[s]);
  };
  if (lane == 0) {
    prefetch_tensormap(&a.tmap);
    if (ROW) prefetch_tensormap(&a.tmap_row);
    if (COL) prefetch_tensormap(&a.tmap_col);
    for (int s = 0; s < kMxStages; s++) mbar_init(&full[s], 1);
    fence_barrier_init();
  }
  uint32_t pending = 0u;  // bit s: a load into stage s is in flight (the same in every lane)
  for (int i = 0; i < kMxStages && i < rounds; i++) {
    int mt, nt;
    if (unit_of(i, mt, nt)) {
      if (lane == 0) issue(mt, nt, i);
      pending |= 1u << i;
    }
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

  uint32_t phase = 0u;      // bit s: parity of the next load to complete in stage s
  bool ok = true;           // false after a wait gave up: no more loads, waits or codes
  bool staged = false;      // this warp has TMA stores in flight that read its staging
  for (int i = 0; i < rounds; i++) {
    const int s = i % kMxStages;
    int mt, nt;
    const bool mine = unit_of(i, mt, nt);
    if (mine && ok) {
      // the phase is complete once any lane has seen it complete
      ok = __any_sync(0xFFFFFFFFu, mbar_wait_bounded(&full[s], (phase >> s) & 1u, kMxWaitLimitNs));
      if (ok) {
        phase ^= 1u << s;
        pending &= ~(1u << s);
      } else if (lane == 0) {
        atomicOr(a.status, 2u);  // NVFP4_DEVICE_TIMEOUT
      }
    }
    const int64_t m0 = (int64_t)mt * kMxUnitM;
    const int64_t n0 = (int64_t)nt * kMxUnitN;
    const uint32_t stage = wstage + (uint32_t)(s * kUnitBytes);
    const uint32_t cs_buf = csst + (uint32_t)((i & 1) * kMxWarps * kMxUnitN);
    if (mine && ok) {
      // the previous unit's stores must have read the staging before it is written again:
      // wait just before the first write, after this unit's first loads and arithmetic
      bool staging_free = !staged;
      auto wait_staging = [&]() {
        if (!staging_free) {
          if (lane == 0) bulk_wait_read_all();
          __syncwarp();
          staging_free = true;
        }
      };

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
          uint32_t o[8];
          block_codes<FMT>(w, mx_multiplier(code), o);
          if (b == 0) wait_staging();
          // row `lane` of the row-code box, block b
          stage_block<FMT, FMT == 2 ? 64 : 128>(
              rowst, (uint32_t)(FMT == 2 ? lane * 64 + 16 * b : lane * 128 + 32 * b), o);
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
        // lane's columns lc0 + j, j = 0..3, of the unit; v[r] = their row-r elements
        const int lc0 = 64 * cbox + 4 * cg;
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
          uint32_t o[8];
          block_codes<FMT>(w, mx_multiplier(code[j]), o);
          if (j == 0) wait_staging();
          // column lc0 + j = 4 g + j is row j * 32 + g of the column-code box [4][32][row]: the
          // eight lanes of a shared-memory phase then write eight different bank groups
          const int g = 16 * cbox + cg;
          stage_block<FMT, FMT == 2 ? 16 : 32>(colst, (uint32_t)((j * 32 + g) * (FMT == 2 ? 16 : 32)), o);
        }
        // the four scales, for the CTA's write-out: [warp][unit column]
        asm volatile("st.shared.u32 [%0], %1;" ::"r"(cs_buf + (uint32_t)(warp * kMxUnitN + lc0)),
                     "r"(code[0] | (code[1] << 8) | (code[2] << 16) | (code[3] << 24))
                     : "memory");
      }

      // every lane has staged its codes: store them (the TMA clips the parts of the boxes
      // outside the tensor)
      __syncwarp();
      if (lane == 0) {
        fence_proxy_async();
        if (ROW) tma_store_2d(&a.tmap_row, rowst, (int32_t)(FMT == 2 ? n0 / 2 : n0), (int32_t)m0);
        if (COL)
          tma_store_3d(&a.tmap_col, colst, (int32_t)(FMT == 2 ? m0 / 2 : m0), (int32_t)(n0 / 4), 0);
        bulk_commit();
      }
      staged = true;
    }

    // refill the stage with this warp's unit kMxStages rounds ahead
    if (ok && i + kMxStages < rounds) {
      int mt2, nt2;
      if (unit_of(i + kMxStages, mt2, nt2)) {
        if (lane == 0) {
          fence_proxy_async();
          issue(mt2, nt2, s);
        }
        pending |= 1u << s;
      }
    }

    if (COL) {
      // column scales: every warp's four bytes per lane are in cs_buf; warp i % kMxWarps writes
      // the group's kMxWarps consecutive scales of each column as one 8-byte word
      named_bar_sync(1, 32 * kMxWarps);
      if (warp == i % kMxWarps) {
        const int gidx = blockIdx.x + i * gridDim.x;
        const int gq = gidx / units_n;
        const int64_t gn0 = (int64_t)(gidx - gq * units_n) * kMxUnitN;
        const int vm = min(kMxWarps, units_m - gq * kMxWarps);  // units of the group in the tensor
        uint32_t x[kMxWarps];
#pragma unroll
        for (int w = 0; w < kMxWarps; w++) x[w] = lds32(cs_buf + (uint32_t)(w * kMxUnitN + 4 * lane));
        static_assert(kMxWarps == 8, "the transpose below packs eight warps' bytes");
        uint32_t lo[4], hi[4];
        {
          const uint32_t t01 = __byte_perm(x[0], x[1], 0x5140), t23 = __byte_perm(x[2], x[3], 0x5140);
          const uint32_t u01 = __byte_perm(x[0], x[1], 0x7362), u23 = __byte_perm(x[2], x[3], 0x7362);
          lo[0] = __byte_perm(t01, t23, 0x5410); lo[1] = __byte_perm(t01, t23, 0x7632);
          lo[2] = __byte_perm(u01, u23, 0x5410); lo[3] = __byte_perm(u01, u23, 0x7632);
          const uint32_t t45 = __byte_perm(x[4], x[5], 0x5140), t67 = __byte_perm(x[6], x[7], 0x5140);
          const uint32_t u45 = __byte_perm(x[4], x[5], 0x7362), u67 = __byte_perm(x[6], x[7], 0x7362);
          hi[0] = __byte_perm(t45, t67, 0x5410); hi[1] = __byte_perm(t45, t67, 0x7632);
          hi[2] = __byte_perm(u45, u67, 0x5410); hi[3] = __byte_perm(u45, u67, 0x7632);
        }
        const bool whole = vm == kMxWarps && ((M / 32) % kMxWarps) == 0 &&
                           (reinterpret_cast<uintptr_t>(a.col_scales) & 7) == 0;
#pragma unroll
        for (int k = 0; k < 4; k++) {
          const int64_t n = gn0 + 4 * lane + k;
          if (n < N) {
            uint8_t* sp = a.col_scales + n * (M / 32) + (int64_t)gq * kMxWarps;
            if (whole) {
              *reinterpret_cast<uint2*>(sp) = make_uint2(lo[k], hi[k]);
            } else {
              for (int w = 0; w < vm; w++)
                sp[w] = (uint8_t)((w < 4 ? lo[k] >> (8 * w) : hi[k] >> (8 * (w - 4))) & 0xFFu);
            }
          }
        }
      }
    }
  }
  // leave only after the stores have read the staging and, after a timeout, after the loads
  // still in flight have landed (bounded)
  if (lane == 0) {
    bulk_wait_all();
    for (int s = 0; s < kMxStages; s++)
      if ((pending >> s) & 1u) mbar_wait_bounded(&full[s], (phase >> s) & 1u, kMxWaitLimitNs);
  }
  __syncwarp();
}

template <int FMT, bool ROW, bool COL>
cudaError_t launch_t(const MxArgs& args, int grid, cudaStream_t s) {
  return launch_pdl(mx_quantize_kernel<FMT, ROW, COL>, dim3(grid), dim3(32 * kMxWarps),
                    kMxSmemBytes, s, args);
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

static_assert(kMxSmemBytes >= kMxWarps * (kMxStages * kUnitBytes + kMxOutBytes) +
                                  2 * kMxWarps * kMxUnitN + kMxWarps * kMxStages * 8 + 1024,
              "MX shared memory: stages, output and scale staging, barriers, alignment slack");
static_assert(kMxOutBytes >= 2 * 4096 && kMxOutBytes % 1024 == 0, "MX output staging");

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
