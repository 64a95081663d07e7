// C ABI of libnvfp4 (declared in include/nvfp4.h): argument checks, the per-device workspace,
// TMA descriptors, and the launch sequence of each entry point.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <atomic>
#include <mutex>

#include "nvfp4.h"
#include "nvfp4_device.cuh"
#include "aux_internal.h"
#include "nvfp4_internal.h"

#define NVFP4_EXPORT extern "C" __attribute__((visibility("default")))

namespace nvfp4 {
namespace {

constexpr int kMaxDevices = 64;
constexpr size_t kWorkspaceBytes = NVFP4_WORKSPACE_BYTES;
constexpr int kFuseWsOffset = 16;  // words: [0] status, [16 .. 16 + kFuseWsWords) fused barrier
static_assert((kFuseWsOffset + kFuseWsWords) * 4 <= (int)kWorkspaceBytes, "workspace too small");

struct DeviceState {
  bool ready = false;
  int sm_count = 0;
  uint32_t* workspace = nullptr;  // [0] status word; the library's own or the caller's
  uint32_t* own = nullptr;        // the library's own workspace, allocated on first need
};

std::mutex g_mutex;
DeviceState g_devices[kMaxDevices];
// Arrivals the next single-launch amax awaits beyond its grid (nvfp4_debug_fused_extra_arrivals)
std::atomic<int32_t> g_fuse_extra{0};
// CTAs of the next single-launch amax that hold back until every rank has arrived
// (nvfp4_debug_fused_late_ctas)
std::atomic<int32_t> g_fuse_late{0};
// Set: the next quantize call launches an empty grid, which the runtime rejects
// (nvfp4_debug_fail_next_launch)
std::atomic<int32_t> g_fail_next{0};
int launch_grid(int grid) { return g_fail_next.exchange(0) ? 0 : grid; }

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

// Everything of a device's state but its workspace (under g_mutex).
nvfp4_status init_device(DeviceState& st, int dev) {
  if (st.ready) return NVFP4_OK;
  if (cudaDeviceGetAttribute(&st.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return NVFP4_ERR_CUDA;
  if (prepare_quantize_kernels() != cudaSuccess) return NVFP4_ERR_CUDA;
  if (g_encode == nullptr) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr)
      return NVFP4_ERR_CUDA;
    g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  }
  st.ready = true;
  return NVFP4_OK;
}

nvfp4_status device_state(DeviceState** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return NVFP4_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState& st = g_devices[dev];
  nvfp4_status r = init_device(st, dev);
  if (r != NVFP4_OK) return r;
  if (st.workspace == nullptr) {  // no caller workspace: the library's own, zeroed once
    if (st.own == nullptr) {
      void* ws = nullptr;
      if (cudaMalloc(&ws, kWorkspaceBytes) != cudaSuccess) return NVFP4_ERR_CUDA;
      if (cudaMemset(ws, 0, kWorkspaceBytes) != cudaSuccess) return NVFP4_ERR_CUDA;
      st.own = static_cast<uint32_t*>(ws);
    }
    st.workspace = st.own;
  }
  *out = &st;
  return NVFP4_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// TMA descriptor of a BF16 [rows][cols] row-major tensor, box {kTileN, box_rows} (a tile, or
// one 16-row slab of it); reads outside the tensor return zeros.
nvfp4_status make_tensor_map(CUtensorMap* map, const void* x, int64_t rows, int64_t cols,
                             int box_rows = kTileM) {
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {(cuuint32_t)kTileN, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(x), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? NVFP4_OK : NVFP4_ERR_CUDA;
}

// TMA descriptor of the columnwise codes [cols][col_ld / 2] bytes as a 3D tensor
// {col_ld / 2, cols / 8, 8} (column 8y + z), box {kTileM / 2, kTileN / 8, 8} with the 32-byte
// swizzle: one quantize tile's codes. Returns false (thread stores are used) when the row pitch
// is not a multiple of 16 bytes or cols not of 8.
bool make_col_codes_map(CUtensorMap* map, uint8_t* col_codes, int64_t cols, int64_t col_ld) {
  const int64_t pitch = col_ld / 2;
  if (col_codes == nullptr || pitch % 16 != 0 || cols % 8 != 0 || cols == 0 || pitch == 0) return false;
  cuuint64_t dims[3] = {(cuuint64_t)pitch, (cuuint64_t)(cols / 8), 8};
  cuuint64_t strides[2] = {(cuuint64_t)(8 * pitch), (cuuint64_t)pitch};
  cuuint32_t box[3] = {(cuuint32_t)(kTileM / 2), (cuuint32_t)(kTileN / 8), 8};
  cuuint32_t estr[3] = {1, 1, 1};
  return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, col_codes, dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_32B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

nvfp4_status check_config(const nvfp4_config* cfg) {
  if (cfg == nullptr) return NVFP4_ERR_INVALID_ARG;
  if (cfg->fast_math != 0 && cfg->fast_math != 1) return NVFP4_ERR_INVALID_ARG;
  if (cfg->swizzle_scales != 0 && cfg->swizzle_scales != 1) return NVFP4_ERR_INVALID_ARG;
  if ((cfg->round_row != NVFP4_ROUND_RN && cfg->round_row != NVFP4_ROUND_SR) ||
      (cfg->round_col != NVFP4_ROUND_RN && cfg->round_col != NVFP4_ROUND_SR))
    return NVFP4_ERR_INVALID_ARG;
  if (cfg->rht_sign_mask > 0xFFFFu) return NVFP4_ERR_INVALID_ARG;
  return NVFP4_OK;
}

// Writes {amax, S_dec} (amax = 0 when `amax` is null) into gscale[e][2] for e < n.
__global__ void gscale_fill_kernel(const float* amax, float* gscale, int n) {
  for (int e = threadIdx.x; e < n; e += blockDim.x) {
    float a = amax ? amax[0] : 0.0f;
    float enc, dec;
    global_scale(a, enc, dec);
    gscale[2 * e] = a;
    gscale[2 * e + 1] = dec;
  }
}

}  // namespace

void take_fuse_debug(QuantArgs& q) {
  q.fuse_extra = g_fuse_extra.exchange(0);
  q.fuse_late = g_fuse_late.exchange(0);
}

cudaError_t launch_quantize(const QuantMode& m, const QuantArgs& args, int grid, cudaStream_t s) {
  if (m.two_d) return launch_quantize_2d(m, args, grid, s);
  if (m.row && m.col && m.rht)
    return m.fast ? launch_quantize_rowcol_rht_fast(m, args, grid, s)
                  : launch_quantize_rowcol_rht(m, args, grid, s);
  if (m.row && m.col) return launch_quantize_rowcol(m, args, grid, s);
  if (m.row) return launch_quantize_row(m, args, grid, s);
  return launch_quantize_col(m, args, grid, s);
}

cudaError_t prepare_quantize_kernels() {
  cudaError_t e = cudaSuccess, r;
  if ((r = prepare_quantize_row()) != cudaSuccess) e = r;
  if ((r = prepare_quantize_col()) != cudaSuccess) e = r;
  if ((r = prepare_quantize_rowcol()) != cudaSuccess) e = r;
  if ((r = prepare_quantize_rowcol_rht()) != cudaSuccess) e = r;
  if ((r = prepare_quantize_rowcol_rht_fast()) != cudaSuccess) e = r;
  if ((r = prepare_quantize_2d()) != cudaSuccess) e = r;
  if ((r = prepare_amax_tiles()) != cudaSuccess) e = r;
  if ((r = prepare_mx_kernels()) != cudaSuccess) e = r;
  return e;
}

namespace {

// A failed launch or call is reported as NVFP4_ERR_CUDA; the runtime's last-error state is
// cleared so that the caller's next, unrelated error check does not see it (a sticky error
// stays sticky).
nvfp4_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return NVFP4_OK;
  (void)cudaGetLastError();
  return NVFP4_ERR_CUDA;
}

// One wave of the flat amax kernel (four 256-thread CTAs per SM), fewer for small tensors.
int amax_flat_grid(const DeviceState* st, int64_t nvec) {
  int64_t g = (nvec + 2047) / 2048;
  const int64_t cap = (int64_t)st->sm_count * 4;
  if (g > cap) g = cap;
  return g < 1 ? 1 : (int)g;
}

int amax_grid(const DeviceState* st, int64_t work_items, int per_block) {
  int64_t g = (work_items + per_block - 1) / per_block;
  int64_t cap = (int64_t)st->sm_count * 8;
  if (g > cap) g = cap;
  return g < 1 ? 1 : (int)g;
}

// The amax pass through the tile kernel: per segment (offsets, or one segment when null)
// max |x| into amax_row[e * stride] and max |x| or the RHT amax into amax_col[e * stride],
// both zeroed by the caller.
nvfp4_status amax_tiles(const DeviceState* ds, const void* x, int64_t rows, int64_t cols,
                        const int32_t* offsets, int32_t segments, uint32_t sign_mask, bool rht,
                        float* amax_row, float* amax_col, int32_t stride, cudaStream_t s) {
  QuantArgs q;
  std::memset(&q, 0, sizeof q);
  nvfp4_status st = make_tensor_map(&q.tmap, x, rows, cols);
  if (st != NVFP4_OK) return st;
  if (offsets && (st = make_tensor_map(&q.tmap_slab, x, rows, cols, 16)) != NVFP4_OK) return st;
  q.x = x; q.rows = rows; q.cols = cols; q.offsets = offsets; q.segments = segments;
  set_rht_flips(q, sign_mask);
  q.amax_row = amax_row; q.amax_col = amax_col;
  q.amax_row_stride = stride; q.amax_col_stride = stride;
  q.status = ds->workspace;
  const int64_t tiles =
      ((rows + kTileM - 1) / kTileM + (offsets ? segments : 0)) * ((cols + kTileN - 1) / kTileN);
  const int grid = (int)(tiles < ds->sm_count ? tiles : ds->sm_count);
  return cuda_status(launch_amax_tiles(rht, q, grid, s));
}

}  // namespace
}  // namespace nvfp4

using namespace nvfp4;

NVFP4_EXPORT const char* nvfp4_status_string(nvfp4_status s) {
  switch (s) {
    case NVFP4_OK: return "ok";
    case NVFP4_ERR_INVALID_ARG: return "invalid argument";
    case NVFP4_ERR_SHAPE: return "shape not a multiple of 16 where blocks need it";
    case NVFP4_ERR_ALIGN: return "pointer or row pitch not 16-byte aligned";
    case NVFP4_ERR_UNSUPPORTED: return "unsupported option combination";
    case NVFP4_ERR_CUDA: return "CUDA error";
    case NVFP4_ERR_DEVICE_STATUS: return "device flagged its input (bad grouped offsets)";
    case NVFP4_ERR_TIMEOUT: return "a bounded device wait gave up";
  }
  return "unknown status";
}

NVFP4_EXPORT nvfp4_status nvfp4_amax(const void* x, int64_t M, int64_t N, const nvfp4_config* cfg,
                                     float* amax_row, float* amax_col, void* stream) {
  nvfp4_status st = check_config(cfg);
  if (st != NVFP4_OK) return st;
  if (M < 0 || N < 0 || (amax_row == nullptr && amax_col == nullptr)) return NVFP4_ERR_INVALID_ARG;
  if (N % 16 != 0 || (cfg->rht_col && amax_col && M % 16 != 0)) return NVFP4_ERR_SHAPE;
  if (M > INT32_MAX || N > INT32_MAX) return NVFP4_ERR_SHAPE;
  if ((M * N > 0 && (x == nullptr || !aligned(x, 16))) || (amax_row && !aligned(amax_row, 4)) ||
      (amax_col && !aligned(amax_col, 4)))
    return NVFP4_ERR_ALIGN;
  DeviceState* ds = nullptr;
  if ((st = device_state(&ds)) != NVFP4_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (amax_row && cudaMemsetAsync(amax_row, 0, 4, s) != cudaSuccess) return NVFP4_ERR_CUDA;
  if (amax_col && cudaMemsetAsync(amax_col, 0, 4, s) != cudaSuccess) return NVFP4_ERR_CUDA;
  if (M * N == 0) return NVFP4_OK;
  if (cfg->rht_col && amax_col)
    return amax_tiles(ds, x, M, N, nullptr, 1, cfg->rht_sign_mask, true, amax_row, amax_col, 1, s);
  return cuda_status(launch_amax_flat(x, M * N, amax_row, amax_col, amax_flat_grid(ds, M * N / 8), s));
}

NVFP4_EXPORT nvfp4_status nvfp4_amax_grouped(const void* x, int64_t T, int64_t H,
                                             const int32_t* offsets, int32_t E,
                                             const nvfp4_config* cfg, float* amax_row,
                                             float* amax_col, void* stream) {
  nvfp4_status st = check_config(cfg);
  if (st != NVFP4_OK) return st;
  if (T < 0 || H < 0 || E < 1 || E > kMaxSegments || offsets == nullptr ||
      (amax_row == nullptr && amax_col == nullptr))
    return NVFP4_ERR_INVALID_ARG;
  if (H % 16 != 0) return NVFP4_ERR_SHAPE;
  if (T > INT32_MAX - kTileM || H > INT32_MAX - kTileN) return NVFP4_ERR_SHAPE;
  if ((T * H > 0 && (x == nullptr || !aligned(x, 16))) || !aligned(offsets, 4) ||
      (amax_row && !aligned(amax_row, 4)) || (amax_col && !aligned(amax_col, 4)))
    return NVFP4_ERR_ALIGN;
  DeviceState* ds = nullptr;
  if ((st = device_state(&ds)) != NVFP4_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (amax_row && cudaMemsetAsync(amax_row, 0, 4 * (size_t)E, s) != cudaSuccess) return NVFP4_ERR_CUDA;
  if (amax_col && cudaMemsetAsync(amax_col, 0, 4 * (size_t)E, s) != cudaSuccess) return NVFP4_ERR_CUDA;
  if (T * H == 0) return NVFP4_OK;
  return amax_tiles(ds, x, T, H, offsets, E, cfg->rht_sign_mask, cfg->rht_col != 0 && amax_col,
                    amax_row, amax_col, 1, s);
}

NVFP4_EXPORT nvfp4_status nvfp4_quantize(const void* x, int64_t M, int64_t N,
                                         const nvfp4_config* cfg, const float* amax_row,
                                         const float* amax_col, uint8_t* row_codes,
                                         uint8_t* row_scales, float* row_gscale,
                                         uint8_t* col_codes, uint8_t* col_scales,
                                         float* col_gscale, void* stream) {
  nvfp4_status st = check_config(cfg);
  if (st != NVFP4_OK) return st;
  const bool two_d = cfg->block2d != 0;
  const bool row = cfg->rowwise != 0;
  const bool col = cfg->columnwise != 0;
  const bool rht = cfg->rht_col != 0 && col;
  if (!row && !col) return NVFP4_ERR_UNSUPPORTED;
  if (two_d && (cfg->rht_col || cfg->round_row == NVFP4_ROUND_SR || cfg->round_col == NVFP4_ROUND_SR))
    return NVFP4_ERR_UNSUPPORTED;
  if (M < 0 || N < 0) return NVFP4_ERR_INVALID_ARG;
  if (N % 16 != 0 || ((col || two_d) && M % 16 != 0)) return NVFP4_ERR_SHAPE;
  if (M > INT32_MAX - kTileM || N > INT32_MAX - kTileN) return NVFP4_ERR_SHAPE;
  const bool empty = M * N == 0;  // empty tensors: only the global scales are written
  if (row && (row_gscale == nullptr || (!empty && (row_codes == nullptr || row_scales == nullptr))))
    return NVFP4_ERR_INVALID_ARG;
  if (col && (col_gscale == nullptr || (!empty && (col_codes == nullptr || col_scales == nullptr))))
    return NVFP4_ERR_INVALID_ARG;
  if ((!empty && (x == nullptr || !aligned(x, 16))) ||
      (row && (!aligned(row_codes, 16) || !aligned(row_scales, 16) || !aligned(row_gscale, 4))) ||
      (col && (!aligned(col_codes, 16) || !aligned(col_scales, 16) || !aligned(col_gscale, 4))) ||
      (amax_row && !aligned(amax_row, 4)) || (amax_col && !aligned(amax_col, 4)))
    return NVFP4_ERR_ALIGN;
  DeviceState* ds = nullptr;
  if ((st = device_state(&ds)) != NVFP4_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  if (M * N == 0) {
    if (row) gscale_fill_kernel<<<1, 32, 0, s>>>(amax_row, row_gscale, 1);
    if (col) gscale_fill_kernel<<<1, 32, 0, s>>>(two_d ? amax_row : amax_col, col_gscale, 1);
    return cuda_status(cudaGetLastError());
  }

  // amax pass (two-pass pipeline) for whatever the caller did not supply; the maxima land in
  // the gscale outputs' amax slots, which the tile kernel reads.
  const bool need_row_amax = (row || two_d) && amax_row == nullptr;
  const bool need_col_amax = col && !two_d && amax_col == nullptr;
  // fused_amax: the missing maxima are computed inside the quantize launch (grid barrier)
  const bool fused = cfg->fused_amax != 0 && (need_row_amax || need_col_amax) &&
                     (amax_row == nullptr || !(row || two_d)) &&
                     (amax_col == nullptr || !(col && !two_d));
  float* row_amax_slot = row ? row_gscale : col_gscale;  // 2D column-only keeps it in col_gscale
  if (!fused && (need_row_amax || need_col_amax)) {
    if (need_row_amax && cudaMemsetAsync(row_amax_slot, 0, 8, s) != cudaSuccess) return NVFP4_ERR_CUDA;
    if (need_col_amax && cudaMemsetAsync(col_gscale, 0, 8, s) != cudaSuccess) return NVFP4_ERR_CUDA;
    if (need_col_amax && rht) {
      if ((st = amax_tiles(ds, x, M, N, nullptr, 1, cfg->rht_sign_mask, true,
                           need_row_amax ? row_amax_slot : nullptr, col_gscale, 2, s)) != NVFP4_OK)
        return st;
    } else {
      if (launch_amax_flat(x, M * N, need_row_amax ? row_amax_slot : nullptr,
                           need_col_amax ? col_gscale : nullptr, amax_flat_grid(ds, M * N / 8),
                           s) != cudaSuccess)
        return NVFP4_ERR_CUDA;
    }
  }

  QuantArgs q;
  std::memset(&q, 0, sizeof q);
  if ((st = make_tensor_map(&q.tmap, x, M, N)) != NVFP4_OK) return st;
  q.rows = M; q.cols = N; q.offsets = nullptr; q.segments = 1;
  const int sr_row = cfg->round_row == NVFP4_ROUND_SR, sr_col = cfg->round_col == NVFP4_ROUND_SR;
  set_rht_flips(q, cfg->rht_sign_mask); q.col_ld = M;
  q.amax_row = amax_row ? amax_row : row_amax_slot;
  q.amax_col = amax_col ? amax_col : col_gscale;
  q.amax_row_stride = 2; q.amax_col_stride = 2;
  q.row_codes = row_codes; q.row_scales = row_scales; q.row_gscale = row_gscale;
  q.col_codes = col_codes; q.col_scales = col_scales; q.col_gscale = col_gscale;
  q.col_tma = col && make_col_codes_map(&q.tmap_colc, col_codes, q.cols, q.col_ld) ? 1 : 0;
  q.seed = cfg->rng_seed; set_philox_keys(q, cfg->rng_seed); q.rng_offset = cfg->rng_offset; q.status = ds->workspace;
  q.x = x;
  q.fused = fused ? 1 : 0;
  q.fast = (cfg->fast_math && !two_d) ? 1 : 0;  // weights (2D blocks) have no fast variant
  q.fuse_ws = ds->workspace + kFuseWsOffset;
  if (cfg->swizzle_scales) {
    const bool row_scales_out = row, col_scales_out = col;
    if (prepare_swizzled_scales(q, row_scales_out ? row_scales : nullptr,
                                col_scales_out ? col_scales : nullptr, M, N, s) != cudaSuccess)
      return cuda_status(cudaErrorUnknown);
  }
  const int64_t tiles = ((M + kTileM - 1) / kTileM) * ((N + kTileN - 1) / kTileN);
  const int grid = (int)(tiles < ds->sm_count ? tiles : ds->sm_count);
  const QuantMode mode{row, col, rht, two_d, sr_row != 0, sr_col != 0, q.fast && rht};
  // the single-launch amax keeps its counts on the device (the last CTA to finish with them
  // readies them for the next launch), so the launch depends on no host state and can be
  // captured in a CUDA graph
  if (fused) take_fuse_debug(q);
  return cuda_status(launch_quantize(mode, q, launch_grid(grid), s));
}

NVFP4_EXPORT nvfp4_status nvfp4_quantize_grouped(const void* x, int64_t T, int64_t H,
                                                 const int32_t* offsets, int32_t E,
                                                 int64_t col_capacity, const nvfp4_config* cfg,
                                                 const float* amax_row, const float* amax_col,
                                                 uint8_t* row_codes, uint8_t* row_scales,
                                                 float* row_gscale, uint8_t* col_codes,
                                                 uint8_t* col_scales, float* col_gscale,
                                                 void* stream) {
  nvfp4_status st = check_config(cfg);
  if (st != NVFP4_OK) return st;
  const bool row = cfg->rowwise != 0;
  const bool col = cfg->columnwise != 0;
  const bool rht = cfg->rht_col != 0 && col;
  if (!row && !col) return NVFP4_ERR_UNSUPPORTED;
  const bool two_d = cfg->block2d != 0;
  if (cfg->fused_amax || cfg->swizzle_scales) return NVFP4_ERR_UNSUPPORTED;
  if (two_d && (cfg->rht_col || cfg->round_row == NVFP4_ROUND_SR || cfg->round_col == NVFP4_ROUND_SR))
    return NVFP4_ERR_UNSUPPORTED;
  if (T < 0 || H < 0 || E < 1 || E > kMaxSegments || offsets == nullptr) return NVFP4_ERR_INVALID_ARG;
  if (H % 16 != 0 || (col && (col_capacity < 0 || col_capacity % 16 != 0))) return NVFP4_ERR_SHAPE;
  if (T > INT32_MAX - kTileM || H > INT32_MAX - kTileN || col_capacity > INT32_MAX)
    return NVFP4_ERR_SHAPE;
  const bool empty = T * H == 0;  // empty tensors: only the global scales are written
  if (row && (row_gscale == nullptr || (!empty && (row_codes == nullptr || row_scales == nullptr))))
    return NVFP4_ERR_INVALID_ARG;
  if (col && (col_gscale == nullptr || (!empty && (col_codes == nullptr || col_scales == nullptr))))
    return NVFP4_ERR_INVALID_ARG;
  if ((!empty && (x == nullptr || !aligned(x, 16))) || !aligned(offsets, 4) ||
      (row && (!aligned(row_codes, 16) || !aligned(row_scales, 16) || !aligned(row_gscale, 4))) ||
      (col && (!aligned(col_codes, 16) || !aligned(col_scales, 16) || !aligned(col_gscale, 4))) ||
      (amax_row && !aligned(amax_row, 4)) || (amax_col && !aligned(amax_col, 4)))
    return NVFP4_ERR_ALIGN;
  DeviceState* ds = nullptr;
  if ((st = device_state(&ds)) != NVFP4_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  if (T * H == 0) {
    if (row) gscale_fill_kernel<<<1, 256, 0, s>>>(nullptr, row_gscale, E);
    if (col) gscale_fill_kernel<<<1, 256, 0, s>>>(nullptr, col_gscale, E);
    return cuda_status(cudaGetLastError());
  }
  // per-expert amax (and RHT amax) of what the caller did not supply, from one read, into the
  // gscale outputs' amax slots. 2D reads the one per-expert amax from the rowwise side (kept in
  // col_gscale when only columnwise).
  const bool need_row = (row || two_d) && amax_row == nullptr;
  const bool need_col = col && !two_d && amax_col == nullptr;
  float* row_slot = row ? row_gscale : col_gscale;
  if (need_row || need_col) {
    if (need_row && cudaMemsetAsync(row_slot, 0, 8 * (size_t)E, s) != cudaSuccess) return NVFP4_ERR_CUDA;
    if (need_col && cudaMemsetAsync(col_gscale, 0, 8 * (size_t)E, s) != cudaSuccess) return NVFP4_ERR_CUDA;
    if ((st = amax_tiles(ds, x, T, H, offsets, E, cfg->rht_sign_mask, need_col && rht,
                         need_row ? row_slot : nullptr, need_col ? col_gscale : nullptr, 2, s)) !=
        NVFP4_OK)
      return st;
  }

  QuantArgs q;
  std::memset(&q, 0, sizeof q);
  if ((st = make_tensor_map(&q.tmap, x, T, H)) != NVFP4_OK) return st;
  if ((st = make_tensor_map(&q.tmap_slab, x, T, H, 16)) != NVFP4_OK) return st;
  q.rows = T; q.cols = H; q.offsets = offsets; q.segments = E;
  const int sr_row = cfg->round_row == NVFP4_ROUND_SR, sr_col = cfg->round_col == NVFP4_ROUND_SR;
  set_rht_flips(q, cfg->rht_sign_mask); q.col_ld = col ? col_capacity : 0;
  q.amax_row = amax_row ? amax_row : ((row || two_d) ? row_slot : nullptr);
  q.amax_col = amax_col ? amax_col : col_gscale;
  q.amax_row_stride = amax_row ? 1 : 2; q.amax_col_stride = amax_col ? 1 : 2;
  q.row_codes = row_codes; q.row_scales = row_scales; q.row_gscale = row_gscale;
  q.col_codes = col_codes; q.col_scales = col_scales; q.col_gscale = col_gscale;
  q.col_tma = col && make_col_codes_map(&q.tmap_colc, col_codes, q.cols, q.col_ld) ? 1 : 0;
  q.seed = cfg->rng_seed; set_philox_keys(q, cfg->rng_seed); q.rng_offset = cfg->rng_offset; q.status = ds->workspace;
  q.fast = (cfg->fast_math && !two_d) ? 1 : 0;  // weights (2D blocks) have no fast variant
  const QuantMode mode{row, col, rht, two_d, sr_row != 0, sr_col != 0, q.fast && rht};
  const int64_t tiles = ((T + kTileM - 1) / kTileM + E) * ((H + kTileN - 1) / kTileN);
  const int grid = (int)(tiles < ds->sm_count ? tiles : ds->sm_count);
  return cuda_status(launch_quantize(mode, q, launch_grid(grid), s));
}

NVFP4_EXPORT nvfp4_status nvfp4_dequantize(const uint8_t* codes, const uint8_t* scales,
                                           const float* gscale, int64_t R, int64_t C, float* out,
                                           void* stream) {
  if (R < 0 || C < 0) return NVFP4_ERR_INVALID_ARG;
  if (C % 16 != 0) return NVFP4_ERR_SHAPE;
  if (R * C == 0) return NVFP4_OK;
  if (codes == nullptr || scales == nullptr || gscale == nullptr || out == nullptr)
    return NVFP4_ERR_INVALID_ARG;
  if (!aligned(codes, 8) || !aligned(gscale, 4) || !aligned(out, 16)) return NVFP4_ERR_ALIGN;
  DeviceState* ds = nullptr;
  nvfp4_status st = device_state(&ds);
  if (st != NVFP4_OK) return st;
  return cuda_status(launch_dequantize(codes, scales, gscale, R, C, false, 0u, false, out,
                                       amax_grid(ds, R * (C / 16), 256),
                                       static_cast<cudaStream_t>(stream)));
}

NVFP4_EXPORT nvfp4_status nvfp4_dequantize_ex(const uint8_t* codes, const uint8_t* scales,
                                              const float* gscale, int64_t R, int64_t C,
                                              int32_t inverse_rht, uint32_t rht_sign_mask,
                                              int32_t out_bf16, void* out, void* stream) {
  if (R < 0 || C < 0 || (inverse_rht != 0 && inverse_rht != 1) || (out_bf16 != 0 && out_bf16 != 1) ||
      rht_sign_mask > 0xFFFFu)
    return NVFP4_ERR_INVALID_ARG;
  if (C % 16 != 0) return NVFP4_ERR_SHAPE;
  if (R * C == 0) return NVFP4_OK;
  if (codes == nullptr || scales == nullptr || gscale == nullptr || out == nullptr)
    return NVFP4_ERR_INVALID_ARG;
  if (!aligned(codes, 8) || !aligned(gscale, 4) || !aligned(out, 16)) return NVFP4_ERR_ALIGN;
  DeviceState* ds = nullptr;
  nvfp4_status st = device_state(&ds);
  if (st != NVFP4_OK) return st;
  return cuda_status(launch_dequantize(codes, scales, gscale, R, C, inverse_rht != 0,
                                       rht_sign_mask, out_bf16 != 0, out,
                                       amax_grid(ds, R * (C / 16), 256),
                                       static_cast<cudaStream_t>(stream)));
}

NVFP4_EXPORT nvfp4_status nvfp4_swizzle_scales(const uint8_t* scales, int64_t R, int64_t C,
                                               uint8_t* out, void* stream) {
  if (R < 0 || C < 0) return NVFP4_ERR_INVALID_ARG;
  if (R * C == 0) return NVFP4_OK;
  if (scales == nullptr || out == nullptr) return NVFP4_ERR_INVALID_ARG;
  if (!aligned(out, 16)) return NVFP4_ERR_ALIGN;
  DeviceState* ds = nullptr;
  nvfp4_status st = device_state(&ds);
  if (st != NVFP4_OK) return st;
  const int64_t chunks = ((R + 127) / 128) * ((C + 3) / 4) * 32;
  return cuda_status(launch_swizzle_scales(scales, R, C, out, amax_grid(ds, chunks, 256),
                                           static_cast<cudaStream_t>(stream)));
}

NVFP4_EXPORT nvfp4_status nvfp4_rmsnorm_amax(const void* x, const void* weight, int64_t M,
                                             int64_t N, float eps, float weight_bias, void* y,
                                             float* amax, void* stream) {
  if (M < 0 || N < 0 || amax == nullptr || !std::isfinite(eps) || !std::isfinite(weight_bias))
    return NVFP4_ERR_INVALID_ARG;
  if (N % 8 != 0) return NVFP4_ERR_SHAPE;
  if (M * N > 0 && (x == nullptr || weight == nullptr || y == nullptr)) return NVFP4_ERR_INVALID_ARG;
  if ((M * N > 0 && (!aligned(x, 16) || !aligned(weight, 16) || !aligned(y, 16))) ||
      !aligned(amax, 4))
    return NVFP4_ERR_ALIGN;
  DeviceState* ds = nullptr;
  nvfp4_status st = device_state(&ds);
  if (st != NVFP4_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(amax, 0, 4, s) != cudaSuccess) return NVFP4_ERR_CUDA;
  if (M * N == 0) return NVFP4_OK;
  const int64_t rows = rmsnorm_rows_per_cta();
  int64_t grid = (M + rows - 1) / rows;
  if (grid > (int64_t)ds->sm_count * 8) grid = (int64_t)ds->sm_count * 8;
  return cuda_status(launch_rmsnorm_amax(x, weight, M, N, eps, weight_bias, y, amax, (int)grid, s));
}

NVFP4_EXPORT nvfp4_status nvfp4_rmsnorm_quantize(const void* x, const void* weight, int64_t M,
                                                 int64_t N, float eps, float weight_bias,
                                                 const nvfp4_config* cfg, void* y, float* amax,
                                                 uint8_t* row_codes, uint8_t* row_scales,
                                                 float* row_gscale, uint8_t* col_codes,
                                                 uint8_t* col_scales, float* col_gscale,
                                                 void* stream) {
  nvfp4_status st = check_config(cfg);
  if (st != NVFP4_OK) return st;
  if (N % 16 != 0) return NVFP4_ERR_SHAPE;
  if ((st = nvfp4_rmsnorm_amax(x, weight, M, N, eps, weight_bias, y, amax, stream)) != NVFP4_OK)
    return st;
  // the producer's amax serves every orientation except the RHT columnwise one, whose amax is
  // that of the transformed columns
  const bool rht = cfg->rht_col != 0 && cfg->columnwise != 0;
  return nvfp4_quantize(y, M, N, cfg, amax, rht ? nullptr : amax, row_codes, row_scales,
                        row_gscale, col_codes, col_scales, col_gscale, stream);
}

NVFP4_EXPORT nvfp4_status nvfp4_mx_quantize(const void* x, int64_t M, int64_t N, int32_t format,
                                            int32_t rowwise, int32_t columnwise,
                                            uint8_t* row_codes, uint8_t* row_scales,
                                            uint8_t* col_codes, uint8_t* col_scales,
                                            void* stream) {
  if (format < NVFP4_MX_E4M3 || format > NVFP4_MX_E2M1 || M < 0 || N < 0)
    return NVFP4_ERR_INVALID_ARG;
  const bool row = rowwise != 0, col = columnwise != 0;
  if (!row && !col) return NVFP4_ERR_UNSUPPORTED;
  if ((row && N % 32 != 0) || (col && (M % 32 != 0 || N % 8 != 0))) return NVFP4_ERR_SHAPE;
  if (M > INT32_MAX - kMxUnitM || N > INT32_MAX - kMxUnitN ||
      ((M + kMxUnitM - 1) / kMxUnitM) * ((N + kMxUnitN - 1) / kMxUnitN) > INT32_MAX / 2)
    return NVFP4_ERR_SHAPE;
  if (M * N == 0) return NVFP4_OK;
  if (x == nullptr || (row && (row_codes == nullptr || row_scales == nullptr)) ||
      (col && (col_codes == nullptr || col_scales == nullptr)))
    return NVFP4_ERR_INVALID_ARG;
  const uintptr_t code_align = format == NVFP4_MX_E2M1 ? 16 : 32;  // one block per store
  if (!aligned(x, 16) || (row && (!aligned(row_codes, code_align) || !aligned(row_scales, 4))) ||
      (col && !aligned(col_codes, code_align)))
    return NVFP4_ERR_ALIGN;
  DeviceState* ds = nullptr;
  nvfp4_status st = device_state(&ds);
  if (st != NVFP4_OK) return st;
  MxArgs a;
  std::memset(&a, 0, sizeof a);
  // x: 32 x 64 BF16 boxes (128-byte rows: the 128-byte swizzle span); outputs: byte tensors
  // stored from swizzled staging, one box per unit and orientation
  auto encode = [&](CUtensorMap* map, CUtensorMapDataType type, const void* p, int64_t inner,
                    int64_t rows, int64_t pitch, uint32_t box_inner, uint32_t box_rows,
                    CUtensorMapSwizzle swizzle) {
    cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)pitch};
    cuuint32_t box[2] = {box_inner, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return g_encode(map, type, 2, const_cast<void*>(p), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  };
  // column codes [N][Mb] (Mb bytes per column) as a 3D tensor {Mb, N/4, 4}: column 4 g + j at
  // (., g, j); a unit's box {32 (FP4: 16), 32, 4} is staged as [j][g][row], which the kernel
  // writes without shared-memory bank conflicts
  auto encode_col_codes = [&](CUtensorMap* map, void* p, int64_t mb, int64_t n, bool fp4_) {
    cuuint64_t dims[3] = {(cuuint64_t)mb, (cuuint64_t)(n / 4), 4};
    cuuint64_t strides[2] = {(cuuint64_t)(4 * mb), (cuuint64_t)mb};
    cuuint32_t box[3] = {fp4_ ? 16u : 32u, (cuuint32_t)(kMxUnitN / 4), 4};
    cuuint32_t estr[3] = {1, 1, 1};
    return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, p, dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE,
                    fp4_ ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_32B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
  };
  const bool fp4 = format == NVFP4_MX_E2M1;
  // each box's swizzle span is its row: 128 bytes for x and FP8 row codes, 64 for FP4 row
  // codes, 32 for FP8 column codes, none for the 16-byte rows of FP4 column codes
  if (!encode(&a.tmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, N, M, N * 2, 64, kMxUnitM,
              CU_TENSOR_MAP_SWIZZLE_128B) ||
      (row && !encode(&a.tmap_row, CU_TENSOR_MAP_DATA_TYPE_UINT8, row_codes, fp4 ? N / 2 : N, M,
                      fp4 ? N / 2 : N, fp4 ? 64 : 128, kMxUnitM,
                      fp4 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B)) ||
      (col && !encode_col_codes(&a.tmap_col, col_codes, fp4 ? M / 2 : M, N, fp4)))
    return NVFP4_ERR_CUDA;
  a.rows = M; a.cols = N;
  a.row_codes = row ? row_codes : nullptr; a.row_scales = row ? row_scales : nullptr;
  a.col_codes = col ? col_codes : nullptr; a.col_scales = col ? col_scales : nullptr;
  a.status = ds->workspace;
  // one CTA per SM at most; a CTA round is kMxWarps vertically adjacent units
  const int64_t units_m = (M + kMxUnitM - 1) / kMxUnitM;
  const int64_t groups = ((units_m + kMxWarps - 1) / kMxWarps) * ((N + kMxUnitN - 1) / kMxUnitN);
  const int grid = (int)(groups < ds->sm_count ? groups : ds->sm_count);
  return cuda_status(launch_mx_quantize(format, row, col, a, grid, static_cast<cudaStream_t>(stream)));
}

NVFP4_EXPORT nvfp4_status nvfp4_mx_dequantize(const uint8_t* codes, const uint8_t* scales,
                                              int32_t format, int64_t R, int64_t C, float* out,
                                              void* stream) {
  if (format < NVFP4_MX_E4M3 || format > NVFP4_MX_E2M1 || R < 0 || C < 0)
    return NVFP4_ERR_INVALID_ARG;
  if (C % 32 != 0) return NVFP4_ERR_SHAPE;
  if (R * C == 0) return NVFP4_OK;
  if (codes == nullptr || scales == nullptr || out == nullptr) return NVFP4_ERR_INVALID_ARG;
  if (!aligned(codes, 16) || !aligned(out, 16)) return NVFP4_ERR_ALIGN;
  DeviceState* ds = nullptr;
  nvfp4_status st = device_state(&ds);
  if (st != NVFP4_OK) return st;
  return cuda_status(launch_mx_dequantize(format, codes, scales, R, C, out,
                                          amax_grid(ds, R * (C / 32), 256),
                                          static_cast<cudaStream_t>(stream)));
}

NVFP4_EXPORT nvfp4_status nvfp4_set_workspace(void* workspace, size_t bytes) {
  if (workspace != nullptr && bytes < kWorkspaceBytes) return NVFP4_ERR_INVALID_ARG;
  if (workspace != nullptr && !aligned(workspace, 256)) return NVFP4_ERR_ALIGN;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return NVFP4_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState& st = g_devices[dev];
  nvfp4_status r = init_device(st, dev);
  if (r != NVFP4_OK) return r;
  // the single-launch amax keeps its counts, maxima and claim bits on the workspace: a
  // workspace taken into use starts from zero
  uint32_t* ws = workspace != nullptr ? static_cast<uint32_t*>(workspace) : st.own;
  if (ws != nullptr && (cudaMemset(ws, 0, kWorkspaceBytes) != cudaSuccess ||
                        cudaDeviceSynchronize() != cudaSuccess))
    return NVFP4_ERR_CUDA;
  st.workspace = ws;  // NULL: the library's own, allocated on the next call if it has none
  return NVFP4_OK;
}

NVFP4_EXPORT nvfp4_status nvfp4_debug_fused_extra_arrivals(int32_t extra) {
  if (extra < 0 || extra > kFuseMaxCtas) return NVFP4_ERR_INVALID_ARG;
  g_fuse_extra.store(extra);
  return NVFP4_OK;
}

NVFP4_EXPORT nvfp4_status nvfp4_debug_fused_late_ctas(int32_t count) {
  if (count < 0 || count > kFuseMaxCtas) return NVFP4_ERR_INVALID_ARG;
  g_fuse_late.store(count);
  return NVFP4_OK;
}

NVFP4_EXPORT nvfp4_status nvfp4_debug_fused_takeovers(void* stream, uint32_t* count) {
  if (count == nullptr) return NVFP4_ERR_INVALID_ARG;
  DeviceState* ds = nullptr;
  nvfp4_status st = device_state(&ds);
  if (st != NVFP4_OK) return st;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return cuda_status(cudaErrorUnknown);
  uint32_t* word = ds->workspace + kFuseWsOffset + kFuseStatsWord;
  uint32_t v = 0;
  if (cudaMemcpy(&v, word, 4, cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemset(word, 0, 4) != cudaSuccess)
    return cuda_status(cudaErrorUnknown);
  *count = v;
  return NVFP4_OK;
}

NVFP4_EXPORT nvfp4_status nvfp4_debug_fail_next_launch(int32_t on) {
  if (on != 0 && on != 1) return NVFP4_ERR_INVALID_ARG;
  g_fail_next.store(on);
  return NVFP4_OK;
}

NVFP4_EXPORT nvfp4_status nvfp4_get_status(void* stream, uint32_t* device_status) {
  if (device_status == nullptr) return NVFP4_ERR_INVALID_ARG;
  DeviceState* ds = nullptr;
  nvfp4_status st = device_state(&ds);
  if (st != NVFP4_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return NVFP4_ERR_CUDA;
  uint32_t v = 0;
  if (cudaMemcpy(&v, ds->workspace, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return NVFP4_ERR_CUDA;
  if (cudaMemset(ds->workspace, 0, 4) != cudaSuccess) return NVFP4_ERR_CUDA;
  *device_status = v;
  if (v & NVFP4_DEVICE_TIMEOUT) return NVFP4_ERR_TIMEOUT;
  if (v) return NVFP4_ERR_DEVICE_STATUS;
  return NVFP4_OK;
}
