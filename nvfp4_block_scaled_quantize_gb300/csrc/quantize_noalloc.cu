// nvfp4_quantize_noalloc: the single-launch (fused amax) quantization for callers that cannot
// allocate device memory -- e.g. code running inside a caching allocator's own callbacks, a
// real-time path that must never reach cudaMalloc (which can synchronize the device), or a
// host that hands this library a fixed memory budget. The regular entry points allocate a
// small per-device workspace on their first call; this one keeps its scratch (a status word,
// the single-launch amax's counts, maxima and claim bits) in a file-scope device array
// instead, so it calls no cudaMalloc, cudaFree or other allocating routine.
// nvfp4_noalloc_get_status reads (and clears) the array's status word, also without
// allocating.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <atomic>
#include <cstring>
#include <mutex>

#include "nvfp4.h"
#include "nvfp4_internal.h"

#define NVFP4_EXPORT extern "C" __attribute__((visibility("default")))

namespace nvfp4 {
namespace {

// Scratch of every nvfp4_quantize_noalloc call on a device (64 words, 256 bytes): word 0 the
// device status word, words 4 .. 4 + kFuseWsWords the counts, maxima and claim bits of the
// single-launch amax (fused_amax.cuh). Zero when the library is loaded and kept until exit.
constexpr int kScratchStatus = 0;
constexpr int kScratchFuse = 4;
constexpr int kScratchWords = 64;
static_assert(kScratchFuse + kFuseWsWords <= kScratchWords, "scratch too small");
static __device__ __align__(256) uint32_t g_noalloc_scratch[kScratchWords];

constexpr int kMaxDevices = 64;

struct NoAllocDevice {
  bool ready = false;
  int sm_count = 0;
  uint32_t* scratch = nullptr;  // device address of g_noalloc_scratch on this device
};

std::mutex g_mutex;
NoAllocDevice g_dev[kMaxDevices];

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

// Once per device, with that device current: the array's device address, the SM count, the
// kernels' shared-memory limit and the TMA descriptor encoder. Nothing here allocates.
nvfp4_status setup(NoAllocDevice** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return NVFP4_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mutex);
  NoAllocDevice& d = g_dev[dev];
  if (!d.ready) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr)
      return NVFP4_ERR_CUDA;
    if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
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
    d.scratch = static_cast<uint32_t*>(ptr);
    d.ready = true;
  }
  *out = &d;
  return NVFP4_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace
}  // namespace nvfp4

using namespace nvfp4;

NVFP4_EXPORT nvfp4_status nvfp4_quantize_noalloc(const void* x, int64_t M, int64_t N,
                                                 const nvfp4_config* cfg, uint8_t* row_codes,
                                                 uint8_t* row_scales, float* row_gscale,
                                                 uint8_t* col_codes, uint8_t* col_scales,
                                                 float* col_gscale, void* stream) {
  if (cfg == nullptr || (cfg->fast_math != 0 && cfg->fast_math != 1) ||
      (cfg->swizzle_scales != 0 && cfg->swizzle_scales != 1))
    return NVFP4_ERR_INVALID_ARG;
  if ((cfg->round_row != NVFP4_ROUND_RN && cfg->round_row != NVFP4_ROUND_SR) ||
      (cfg->round_col != NVFP4_ROUND_RN && cfg->round_col != NVFP4_ROUND_SR) ||
      cfg->rht_sign_mask > 0xFFFFu)
    return NVFP4_ERR_INVALID_ARG;
  const bool two_d = cfg->block2d != 0;
  const bool row = cfg->rowwise != 0;
  const bool col = cfg->columnwise != 0;
  const bool rht = cfg->rht_col != 0 && col;
  if (!row && !col) return NVFP4_ERR_UNSUPPORTED;
  if (two_d && (cfg->rht_col || cfg->round_row == NVFP4_ROUND_SR || cfg->round_col == NVFP4_ROUND_SR))
    return NVFP4_ERR_UNSUPPORTED;
  if (M <= 0 || N <= 0) return NVFP4_ERR_SHAPE;
  if (N % 16 != 0 || ((col || two_d) && M % 16 != 0)) return NVFP4_ERR_SHAPE;
  if (M > INT32_MAX - kTileM || N > INT32_MAX - kTileN) return NVFP4_ERR_SHAPE;
  if ((row && (row_codes == nullptr || row_scales == nullptr || row_gscale == nullptr)) ||
      (col && (col_codes == nullptr || col_scales == nullptr || col_gscale == nullptr)) ||
      x == nullptr)
    return NVFP4_ERR_INVALID_ARG;
  if (!aligned(x, 16) ||
      (row && (!aligned(row_codes, 16) || !aligned(row_scales, 16) || !aligned(row_gscale, 4))) ||
      (col && (!aligned(col_codes, 16) || !aligned(col_scales, 16) || !aligned(col_gscale, 4))))
    return NVFP4_ERR_ALIGN;
  NoAllocDevice* d = nullptr;
  nvfp4_status st = setup(&d);
  if (st != NVFP4_OK) return st;
  const int64_t tiles = ((M + kTileM - 1) / kTileM) * ((N + kTileN - 1) / kTileN);
  const int grid = (int)(tiles < d->sm_count ? tiles : d->sm_count);
  // one claim bit per CTA in the array (GB300 launches one CTA per SM, 152)
  if (grid > kFuseMaxCtas) return NVFP4_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  QuantArgs q;
  std::memset(&q, 0, sizeof q);
  cuuint64_t dims[2] = {(cuuint64_t)N, (cuuint64_t)M};
  cuuint64_t strides[1] = {(cuuint64_t)N * 2};
  cuuint32_t box[2] = {(cuuint32_t)kTileN, (cuuint32_t)kTileM};
  cuuint32_t estr[2] = {1, 1};
  if (g_encode(&q.tmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(x), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return NVFP4_ERR_CUDA;
  q.x = x;
  q.rows = M; q.cols = N; q.offsets = nullptr; q.segments = 1;
  set_rht_flips(q, cfg->rht_sign_mask); q.col_ld = M;
  q.amax_row = nullptr; q.amax_col = nullptr;  // computed in the launch (fused)
  q.amax_row_stride = 2; q.amax_col_stride = 2;
  q.row_codes = row_codes; q.row_scales = row_scales; q.row_gscale = row_gscale;
  q.col_codes = col_codes; q.col_scales = col_scales; q.col_gscale = col_gscale;
  if (col && (M / 2) % 16 == 0 && N % 8 == 0) {
    cuuint64_t cdims[3] = {(cuuint64_t)(M / 2), (cuuint64_t)(N / 8), 8};
    cuuint64_t cstrides[2] = {(cuuint64_t)(8 * (M / 2)), (cuuint64_t)(M / 2)};
    cuuint32_t cbox[3] = {(cuuint32_t)(kTileM / 2), (cuuint32_t)(kTileN / 8), 8};
    cuuint32_t cestr[3] = {1, 1, 1};
    q.col_tma = g_encode(&q.tmap_colc, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, col_codes, cdims, cstrides,
                         cbox, cestr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_32B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS ? 1 : 0;
  }
  q.seed = cfg->rng_seed; set_philox_keys(q, cfg->rng_seed); q.rng_offset = cfg->rng_offset;
  q.status = d->scratch + kScratchStatus;
  q.fused = 1;
  q.fast = (cfg->fast_math && !two_d) ? 1 : 0;  // weights (2D blocks) have no fast variant
  q.fuse_ws = d->scratch + kScratchFuse;
  take_fuse_debug(q);  // the test hooks of the single-launch amax apply here too
  if (cfg->swizzle_scales &&
      prepare_swizzled_scales(q, row ? row_scales : nullptr, col ? col_scales : nullptr, M, N, s) !=
          cudaSuccess) {
    (void)cudaGetLastError();
    return NVFP4_ERR_CUDA;
  }
  // the single-launch amax keeps its counts in the array (zero when loaded; the last CTA to
  // finish with them readies them for the next launch), so nothing is cleared before a launch
  const QuantMode mode{row, col, rht, two_d, cfg->round_row == NVFP4_ROUND_SR,
                       cfg->round_col == NVFP4_ROUND_SR, q.fast && rht};
  if (launch_quantize(mode, q, grid, s) != cudaSuccess) {
    (void)cudaGetLastError();  // leave no error behind for the caller's next check
    return NVFP4_ERR_CUDA;
  }
  return NVFP4_OK;
}

NVFP4_EXPORT nvfp4_status nvfp4_noalloc_get_status(void* stream, uint32_t* device_status) {
  if (device_status == nullptr) return NVFP4_ERR_INVALID_ARG;
  NoAllocDevice* d = nullptr;
  nvfp4_status st = setup(&d);
  if (st != NVFP4_OK) return st;
  // the status word is read and cleared by synchronous copies to and from the array itself:
  // nothing is allocated
  const uint32_t zero = 0u;
  uint32_t v = 0u;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess ||
      cudaMemcpyFromSymbol(&v, g_noalloc_scratch, 4, 4 * kScratchStatus, cudaMemcpyDeviceToHost) !=
          cudaSuccess ||
      cudaMemcpyToSymbol(g_noalloc_scratch, &zero, 4, 4 * kScratchStatus, cudaMemcpyHostToDevice) !=
          cudaSuccess) {
    (void)cudaGetLastError();
    return NVFP4_ERR_CUDA;
  }
  *device_status = v;
  if (v & NVFP4_DEVICE_TIMEOUT) return NVFP4_ERR_TIMEOUT;
  if (v) return NVFP4_ERR_DEVICE_STATUS;
  return NVFP4_OK;
}
