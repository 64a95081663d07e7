// The tile kernel: rowwise, columnwise (optionally after the 16-point RHT, with RTNE or
// stochastic rounding) and 16x16 2D NVFP4 quantization of BF16 tensors from ONE read of the
// input, for plain tensors and for grouped (MoE) tensors split into row segments.
//
// Page cited: "[nvfp4_training] Optimize CuteDSL kernels for NVFP4 training" (pytorch/ao pull
// request #4798). Its kernels -- "linear fused" and "grouped fused" row+col quantize, the 2D
// weight kernel -- are the prior art; this is a design for sm_103a:
//   * one persistent CTA per SM (512 threads) walks the tile list; a 4-stage ring of
//     64 x 256 BF16 tiles is filled by TMA (cp.async.bulk.tensor) on mbarriers, so three tiles
//     (96 KiB) are in flight per SM while the fourth is consumed;
//   * the rowwise pass reads 16-byte chunks of two rows per warp step; a lane pair shares one
//     1x16 block, splitting the scale work and the Philox draw between the pair
//     ("Optimization" items 2, 3 and 7);
//   * the columnwise pass gives each thread a 16-row x 2-column strip (one 32-bit shared load
//     per row, conflict-free), so the column block maximum, the RHT butterflies and the
//     conversion are thread-local;
//   * columnwise codes and scales are staged in shared memory and leave as whole 8/16-byte
//     runs per column ("Optimization" item 5: word-wide scale stores);
//   * all arithmetic follows the exact mode ("Fast math"): IEEE div/rcp, f32x2 products,
//     cvt.rn/cvt.rs.satfinite conversions.
#include "nvfp4_device.cuh"
#include "nvfp4_internal.h"

namespace nvfp4 {

namespace {

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s: a TMA load never takes this long

__device__ __forceinline__ void st_global_u32(uint8_t* p, uint32_t v) {
  *reinterpret_cast<uint32_t*>(p) = v;
}
__device__ __forceinline__ void st_global_u64(uint8_t* p, uint64_t v) {
  *reinterpret_cast<uint64_t*>(p) = v;
}

// Store n bytes from shared memory (n <= 16) with the widest accesses the destination's
// alignment allows.
__device__ __forceinline__ void store_bytes(uint8_t* dst, const uint8_t* src, int n) {
  uintptr_t a = reinterpret_cast<uintptr_t>(dst);
  if (n == 16 && (a & 15) == 0) {
    *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(src);
  } else if ((a & 3) == 0 && (n & 3) == 0) {
    for (int i = 0; i < n; i += 4)
      *reinterpret_cast<uint32_t*>(dst + i) = *reinterpret_cast<const uint32_t*>(src + i);
  } else {
    for (int i = 0; i < n; i++) dst[i] = src[i];
  }
}

struct TileCoord {
  int seg;
  int32_t row0;    // first row of the tile in x
  int32_t nrows;   // rows of the tile inside its segment (<= kTileM)
  int32_t n0;      // first column
  int32_t mt;      // tile index inside its segment along M
};

__device__ __forceinline__ TileCoord locate_tile(int tile, int segments, int tiles_n,
                                                 const int32_t* seg_tile0,
                                                 const int32_t* seg_start,
                                                 const int32_t* seg_end) {
  // largest e with seg_tile0[e] <= tile (empty segments share their successor's start)
  int lo = 0, hi = segments;  // seg_tile0[segments] = total > tile
  while (hi - lo > 1) {
    int mid = (lo + hi) >> 1;
    if (seg_tile0[mid] <= tile) lo = mid; else hi = mid;
  }
  TileCoord c;
  c.seg = lo;
  int local = tile - seg_tile0[lo];
  c.mt = local / tiles_n;
  c.n0 = (local - c.mt * tiles_n) * kTileN;
  c.row0 = seg_start[lo] + c.mt * kTileM;
  c.nrows = min(kTileM, seg_end[lo] - c.row0);
  return c;
}

template <bool ROW, bool COL, bool RHT, bool TWO_D>
__global__ void __launch_bounds__(kQuantThreads, 1)
    quantize_tiles_kernel(const __grid_constant__ QuantArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;

  int32_t* seg_start = reinterpret_cast<int32_t*>(smem + kSmemSegStart);
  int32_t* seg_end = reinterpret_cast<int32_t*>(smem + kSmemSegEnd);
  int32_t* seg_col0 = reinterpret_cast<int32_t*>(smem + kSmemSegCol0);
  int32_t* seg_tile0 = reinterpret_cast<int32_t*>(smem + kSmemSegTile0);
  float4* seg_scale = reinterpret_cast<float4*>(smem + kSmemSegScale);
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + kSmemBars);
  volatile int32_t* flags = reinterpret_cast<volatile int32_t*>(smem + kSmemFlags);
  float* tile_r = reinterpret_cast<float*>(smem + kSmemTileR);
  uint8_t* tile_s = smem + kSmemTileS;

  const int E = a.segments;
  const int tiles_n = (int)((a.cols + kTileN - 1) / kTileN);

  // ---- segment table: starts, ends, padded column starts, tile prefix sums ----
  if (tid == 0) { flags[0] = 0; flags[1] = 0; }
  __syncthreads();
  for (int e = tid; e < E; e += blockDim.x) {
    int32_t start = (a.offsets == nullptr || e == 0) ? 0 : a.offsets[e - 1];
    int32_t end = (a.offsets == nullptr) ? (int32_t)a.rows : a.offsets[e];
    if (start < 0 || end < start || (int64_t)end > a.rows) flags[1] = 1;
    seg_start[e] = start;
    seg_end[e] = end;
  }
  __syncthreads();
  if (warp == 0) {
    // serial over chunks of 32 segments, warp-inclusive scans inside a chunk
    int32_t tile_base = 0, col_base = 0;
    for (int c0 = 0; c0 < E; c0 += 32) {
      int e = c0 + lane;
      int32_t n = (e < E && !flags[1]) ? seg_end[e] - seg_start[e] : 0;
      int32_t t = ((n + kTileM - 1) / kTileM) * tiles_n;
      int32_t p = ((n + 15) / 16) * 16;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        int32_t tu = __shfl_up_sync(0xFFFFFFFFu, t, d);
        int32_t pu = __shfl_up_sync(0xFFFFFFFFu, p, d);
        if (lane >= d) { t += tu; p += pu; }
      }
      int32_t t_excl = t - (((n + kTileM - 1) / kTileM) * tiles_n);
      int32_t p_excl = p - ((n + 15) / 16) * 16;
      if (e < E) {
        seg_tile0[e] = tile_base + t_excl;
        seg_col0[e] = col_base + p_excl;
      }
      tile_base += __shfl_sync(0xFFFFFFFFu, t, 31);
      col_base += __shfl_sync(0xFFFFFFFFu, p, 31);
    }
    if (lane == 0) {
      seg_tile0[E] = tile_base;
      if (COL && (int64_t)col_base > a.col_ld) flags[1] = 1;
    }
  }
  __syncthreads();
  if (flags[1]) {
    if (blockIdx.x == 0 && tid == 0) atomicOr(a.status, 1u);  // NVFP4_DEVICE_BAD_OFFSETS
    return;
  }
  // per-segment global scales {S_enc_row, S_dec_row, S_enc_col, S_dec_col}
  for (int e = tid; e < E; e += blockDim.x) {
    float4 sc = make_float4(1.f, 1.f, 1.f, 1.f);
    if (ROW || TWO_D) {
      float amax = a.amax_row[(int64_t)e * a.amax_row_stride];
      global_scale(amax, sc.x, sc.y);
      if (blockIdx.x == 0) {
        if (ROW) { a.row_gscale[2 * e] = amax; a.row_gscale[2 * e + 1] = sc.y; }
        if (TWO_D && COL) { a.col_gscale[2 * e] = amax; a.col_gscale[2 * e + 1] = sc.y; }
      }
    }
    if (COL && !TWO_D) {
      float amax = a.amax_col[(int64_t)e * a.amax_col_stride];
      global_scale(amax, sc.z, sc.w);
      if (blockIdx.x == 0) { a.col_gscale[2 * e] = amax; a.col_gscale[2 * e + 1] = sc.w; }
    }
    if (TWO_D) { sc.z = sc.x; sc.w = sc.y; }
    seg_scale[e] = sc;
  }

  const int total = seg_tile0[E];
  const int stride = gridDim.x;
  if (tid == 0) {
    for (int s = 0; s < kStages; s++) mbar_init(&full_bar[s], 1);
    fence_barrier_init();
    prefetch_tensormap(&a.tmap);
  }
  __syncthreads();
  // prologue: fill the ring
  if (tid == 0) {
    for (int s = 0; s < kStages; s++) {
      int t = blockIdx.x + s * stride;
      if (t >= total) break;
      TileCoord c = locate_tile(t, E, tiles_n, seg_tile0, seg_start, seg_end);
      mbar_expect_tx(&full_bar[s], kStageBytes);
      tma_load_2d(smem + kSmemStages + s * kStageBytes, &a.tmap, c.n0, c.row0, &full_bar[s]);
    }
  }

  const int64_t N = a.cols;
  const int64_t row_nb = N / 16;           // rowwise scale-tensor row length
  const int64_t col_nb = a.col_ld / 16;    // columnwise scale-tensor row length
  int it = 0;
  for (int tile = blockIdx.x; tile < total; tile += stride, it++) {
    const int s = it % kStages;
    const uint32_t parity = (uint32_t)(it / kStages) & 1u;
    const int buf = it & 1;
    const TileCoord c = locate_tile(tile, E, tiles_n, seg_tile0, seg_start, seg_end);
    const float4 sc = seg_scale[c.seg];
    const uint32_t stage = smem_u32(smem + kSmemStages + s * kStageBytes);
    const int nrb = (c.nrows + 15) >> 4;    // row blocks of the tile (last one zero-padded)

    if (!mbar_wait_bounded(&full_bar[s], parity, kWaitLimitNs)) {
      // The tile's data never arrived. The passes below still run (on stale shared memory,
      // every address stays inside the tile), and all threads leave together after the
      // end-of-tile barrier.
      flags[0] = 1;
      atomicOr(a.status, 2u);  // NVFP4_DEVICE_TIMEOUT
    }

    // ---- 2D: one scale per 16x16 tile, from the tile amax ----
    uint32_t strip[16];  // column strip of the 2D and columnwise passes (16 rows x 2 columns)
    const int cp = tid & 127;  // column pair of the strip
    const int rb = tid >> 7;   // row block of the strip
    if (TWO_D) {
#pragma unroll
      for (int i = 0; i < 16; i++) strip[i] = lds32(stage + (rb * 16 + i) * (kTileN * 2) + cp * 4);
      uint32_t m = 0;
#pragma unroll
      for (int i = 0; i < 16; i++) m = vmax2(m, abs2(strip[i]));
      uint32_t tm = max(m & 0xFFFFu, m >> 16);
      tm = max(tm, __shfl_xor_sync(0xFFFFFFFFu, tm, 1));
      tm = max(tm, __shfl_xor_sync(0xFFFFFFFFu, tm, 2));
      tm = max(tm, __shfl_xor_sync(0xFFFFFFFFu, tm, 4));
      if ((lane & 7) == 0) {
        uint16_t s2 = block_scales2(__uint_as_float(tm << 16), 0.0f, sc.x);
        float2 sf = e4m3x2_to_float2(s2);
        tile_s[rb * 16 + (cp >> 3)] = (uint8_t)(s2 & 0xFFu);
        tile_r[rb * 16 + (cp >> 3)] = element_multiplier(sf.x, sc.y);
      }
      __syncthreads();
    }

    // ---- rowwise: 1x16 blocks along N ----
    if (ROW) {
      uint8_t* rs_stage = smem + kSmemRowScales + buf * kRowScaleStage;
      const bool even = (lane & 1) == 0;
      const int k = lane >> 1;                  // block of the tile row
      const bool col_ok = (int64_t)c.n0 + lane * 8 < N;
#pragma unroll
      for (int pr = 0; pr < 2; pr++) {
        const int j = warp * 4 + pr * 2;        // rows j, j + 1 of the tile
        const uint4 va = lds128(stage + j * (kTileN * 2) + lane * 16);
        const uint4 vb = lds128(stage + (j + 1) * (kTileN * 2) + lane * 16);
        float r_j, r_j1;
        uint8_t s_mine;                         // scale of (row j, even lane) / (row j+1, odd)
        if (TWO_D) {
          r_j = r_j1 = tile_r[(j >> 4) * 16 + k];
          s_mine = tile_s[(j >> 4) * 16 + k];
        } else {
          uint32_t ma = vmax2(vmax2(abs2(va.x), abs2(va.y)), vmax2(abs2(va.z), abs2(va.w)));
          uint32_t mb = vmax2(vmax2(abs2(vb.x), abs2(vb.y)), vmax2(abs2(vb.z), abs2(vb.w)));
          uint32_t fa = max(ma & 0xFFFFu, ma >> 16);
          uint32_t fb = max(mb & 0xFFFFu, mb >> 16);
          uint32_t recv = __shfl_xor_sync(0xFFFFFFFFu, even ? fb : fa, 1);
          uint32_t bm = even ? max(fa, recv) : max(fb, recv);
          uint16_t s2 = block_scales2(__uint_as_float(bm << 16), 0.0f, sc.x);
          s_mine = (uint8_t)(s2 & 0xFFu);
          float r = element_multiplier(e4m3x2_to_float2(s2).x, sc.y);
          float r_other = __shfl_xor_sync(0xFFFFFFFFu, r, 1);
          r_j = even ? r : r_other;
          r_j1 = even ? r_other : r;
        }
        uint32_t wa0 = 0, wa1 = 0, wb0 = 0, wb1 = 0;
        if (a.sr_row) {
          // even lane draws block (row j, k), odd lane block (row j+1, k); each lane then
          // needs the two words of its half of both blocks
          const uint64_t b = (uint64_t)(c.row0 + j + (even ? 0 : 1)) * row_nb +
                             (uint64_t)(c.n0 / 16 + k);
          const uint4 R = block_random(a.seed, a.rng_offset, 0u, b);
          uint32_t y0 = __shfl_xor_sync(0xFFFFFFFFu, even ? R.z : R.x, 1);
          uint32_t y1 = __shfl_xor_sync(0xFFFFFFFFu, even ? R.w : R.y, 1);
          if (even) { wa0 = R.x; wa1 = R.y; wb0 = y0; wb1 = y1; }
          else { wa0 = y0; wa1 = y1; wb0 = R.z; wb1 = R.w; }
        }
        const uint32_t ca = quantize8(va.x, va.y, va.z, va.w, r_j, a.sr_row, wa0, wa1);
        const uint32_t cb = quantize8(vb.x, vb.y, vb.z, vb.w, r_j1, a.sr_row, wb0, wb1);
        if (col_ok) {
          uint8_t* base = a.row_codes + (int64_t)c.n0 / 2 + lane * 4;
          if (j < c.nrows) st_global_u32(base + (int64_t)(c.row0 + j) * (N / 2), ca);
          if (j + 1 < c.nrows) st_global_u32(base + (int64_t)(c.row0 + j + 1) * (N / 2), cb);
        }
        rs_stage[(j + (even ? 0 : 1)) * 16 + k] = s_mine;
      }
    }

    // ---- columnwise: 1x16 blocks along M, written transposed ----
    if (COL) {
      if (!TWO_D) {
#pragma unroll
        for (int i = 0; i < 16; i++)
          strip[i] = lds32(stage + (rb * 16 + i) * (kTileN * 2) + cp * 4);
      }
      if (c.nrows < kTileM) {  // rows past the segment's end are zero padding
#pragma unroll
        for (int i = 0; i < 16; i++)
          if (rb * 16 + i >= c.nrows) strip[i] = 0u;
      }
      if (RHT) rht16_pair(strip, a.sign_mask);
      float r0, r1;
      uint16_t s2;
      if (TWO_D) {
        const uint8_t sv = tile_s[rb * 16 + (cp >> 3)];
        s2 = (uint16_t)(sv | (sv << 8));
        r0 = r1 = tile_r[rb * 16 + (cp >> 3)];
      } else {
        uint32_t m = 0;
#pragma unroll
        for (int i = 0; i < 16; i++) m = vmax2(m, abs2(strip[i]));
        s2 = block_scales2(mag_lo(m), mag_hi(m), sc.z);
        float2 sf = e4m3x2_to_float2(s2);
        r0 = element_multiplier(sf.x, sc.w);
        r1 = element_multiplier(sf.y, sc.w);
      }
      uint4 R0 = make_uint4(0, 0, 0, 0), R1 = make_uint4(0, 0, 0, 0);
      if (a.sr_col) {
        const uint64_t b0 = (uint64_t)(c.n0 + 2 * cp) * (uint64_t)col_nb +
                            (uint64_t)(seg_col0[c.seg] / 16 + c.mt * (kTileM / 16) + rb);
        R0 = block_random(a.seed, a.rng_offset, 1u, b0);
        R1 = block_random(a.seed, a.rng_offset, 1u, b0 + (uint64_t)col_nb);
      }
      uint4 q;
      q.x = quantize8_column(strip, false, r0, a.sr_col, R0.x, R0.y);
      q.y = quantize8_column(strip + 8, false, r0, a.sr_col, R0.z, R0.w);
      q.z = quantize8_column(strip, true, r1, a.sr_col, R1.x, R1.y);
      q.w = quantize8_column(strip + 8, true, r1, a.sr_col, R1.z, R1.w);
      uint8_t* cc = smem + kSmemColCodes + buf * kColCodeStage;
      *reinterpret_cast<uint4*>(cc + rb * (kTileN * 8) + cp * 16) = q;
      uint8_t* cs = smem + kSmemColScales + buf * kColScaleStage;
      *reinterpret_cast<uint16_t*>(cs + rb * kTileN + cp * 2) = s2;
    }

    __syncthreads();  // stage s fully read; staging buffers complete
    if (flags[0]) break;
    if (tid == 0) {
      const int next = tile + kStages * stride;
      if (next < total) {
        fence_proxy_async();
        TileCoord nc = locate_tile(next, E, tiles_n, seg_tile0, seg_start, seg_end);
        mbar_expect_tx(&full_bar[s], kStageBytes);
        tma_load_2d(smem + kSmemStages + s * kStageBytes, &a.tmap, nc.n0, nc.row0, &full_bar[s]);
      }
    }

    // ---- write-out of the staged columnwise codes/scales and rowwise scales ----
    if (COL) {
      const uint8_t* cc = smem + kSmemColCodes + buf * kColCodeStage;
      const int cl = tid >> 1, h = tid & 1;       // column of the tile, half (row blocks 2h, 2h+1)
      const int64_t col = (int64_t)c.n0 + cl;
      const int64_t colpos = (int64_t)seg_col0[c.seg] + (int64_t)c.mt * kTileM;  // in elements
      if (col < N && 2 * h < nrb) {
        uint8_t* dst = a.col_codes + col * (a.col_ld / 2) + colpos / 2 + 16 * h;
        const uint64_t v0 = *reinterpret_cast<const uint64_t*>(cc + (2 * h) * (kTileN * 8) + cl * 8);
        if (2 * h + 1 < nrb) {
          const uint64_t v1 =
              *reinterpret_cast<const uint64_t*>(cc + (2 * h + 1) * (kTileN * 8) + cl * 8);
          if ((reinterpret_cast<uintptr_t>(dst) & 15) == 0) {
            *reinterpret_cast<uint4*>(dst) =
                make_uint4((uint32_t)v0, (uint32_t)(v0 >> 32), (uint32_t)v1, (uint32_t)(v1 >> 32));
          } else {
            st_global_u64(dst, v0);
            st_global_u64(dst + 8, v1);
          }
        } else {
          st_global_u64(dst, v0);
        }
      }
      if (tid < kTileN) {
        const int64_t colx = (int64_t)c.n0 + tid;
        if (colx < N) {
          const uint8_t* cs = smem + kSmemColScales + buf * kColScaleStage;
          uint8_t* dst = a.col_scales + colx * col_nb + colpos / 16;
          if (nrb == 4 && (reinterpret_cast<uintptr_t>(dst) & 3) == 0) {
            uint32_t v = (uint32_t)cs[tid] | ((uint32_t)cs[kTileN + tid] << 8) |
                         ((uint32_t)cs[2 * kTileN + tid] << 16) | ((uint32_t)cs[3 * kTileN + tid] << 24);
            st_global_u32(dst, v);
          } else {
            for (int q = 0; q < nrb; q++) dst[q] = cs[q * kTileN + tid];
          }
        }
      }
    }
    if (ROW && tid >= 256 && tid < 256 + kTileM) {
      const int row = tid - 256;
      if (row < c.nrows) {
        const int64_t left = (N - c.n0) / 16;
        const int nb = left < 16 ? (int)left : 16;
        uint8_t* dst = a.row_scales + (int64_t)(c.row0 + row) * row_nb + c.n0 / 16;
        store_bytes(dst, smem + kSmemRowScales + buf * kRowScaleStage + row * 16, nb);
      }
    }
  }

  if (flags[0] && tid == 0) {
    // a wait gave up: let every load still in flight land before the CTA leaves
    for (int q = 0; q < kStages; q++) {
      const int t = blockIdx.x + (it + q) * stride;
      if (t >= total) break;
      const int s = (it + q) % kStages;
      mbar_wait_bounded(&full_bar[s], (uint32_t)((it + q) / kStages) & 1u, kWaitLimitNs);
    }
  }
}

template <bool ROW, bool COL, bool RHT, bool TWO_D>
cudaError_t launch_variant(const QuantArgs& args, int grid, cudaStream_t s) {
  quantize_tiles_kernel<ROW, COL, RHT, TWO_D><<<grid, kQuantThreads, kQuantSmemBytes, s>>>(args);
  return cudaGetLastError();
}

template <bool ROW, bool COL, bool RHT, bool TWO_D>
cudaError_t set_smem() {
  return cudaFuncSetAttribute(quantize_tiles_kernel<ROW, COL, RHT, TWO_D>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, kQuantSmemBytes);
}

}  // namespace

cudaError_t prepare_quantize_kernels() {
  cudaError_t e = cudaSuccess;
  cudaError_t r;
  if ((r = set_smem<true, false, false, false>()) != cudaSuccess) e = r;
  if ((r = set_smem<false, true, false, false>()) != cudaSuccess) e = r;
  if ((r = set_smem<false, true, true, false>()) != cudaSuccess) e = r;
  if ((r = set_smem<true, true, false, false>()) != cudaSuccess) e = r;
  if ((r = set_smem<true, true, true, false>()) != cudaSuccess) e = r;
  if ((r = set_smem<true, false, false, true>()) != cudaSuccess) e = r;
  if ((r = set_smem<false, true, false, true>()) != cudaSuccess) e = r;
  if ((r = set_smem<true, true, false, true>()) != cudaSuccess) e = r;
  return e;
}

cudaError_t launch_quantize(QuantVariant v, const QuantArgs& args, int grid, cudaStream_t s) {
  switch (v) {
    case kRow: return launch_variant<true, false, false, false>(args, grid, s);
    case kCol: return launch_variant<false, true, false, false>(args, grid, s);
    case kColRht: return launch_variant<false, true, true, false>(args, grid, s);
    case kRowCol: return launch_variant<true, true, false, false>(args, grid, s);
    case kRowColRht: return launch_variant<true, true, true, false>(args, grid, s);
    case k2dRow: return launch_variant<true, false, false, true>(args, grid, s);
    case k2dCol: return launch_variant<false, true, false, true>(args, grid, s);
    case k2dRowCol: return launch_variant<true, true, false, true>(args, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace nvfp4
