// Host pipeline: quantization of host-resident tensors with the copies of consecutive
// submissions overlapped. On GB300 the host link moves about 210 GB/s host-to-device and
// 190 GB/s device-to-host, and close to 300 GB/s when both directions run at once, so a
// stream of tensors is bound by the link, not by the quantize kernel (~40 us for 64 MiB).
// Each submission takes the next of `depth` device slots; three streams carry the copy in,
// the quantization and the copy out, ordered by per-slot events:
//   copy in  (slot k) after the slot's previous quantization has read its input;
//   quantize (slot k) after the copy in landed and the slot's previous outputs left;
//   copy out (slot k) after the quantization.
// With depth 2 the copy in of submission i+1 runs while submission i is quantized and copied
// out. Runtime plumbing only: the quantization is nvfp4_quantize (grouped tensors:
// nvfp4_quantize_grouped, the expert offsets copied in with x) on the compute stream.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <new>

#include "nvfp4.h"

#define NVFP4_EXPORT extern "C" __attribute__((visibility("default")))

namespace {

constexpr int kMaxDepth = 4;

struct Slot {
  void* x = nullptr;  // BF16 [M][N]
  int32_t* offsets = nullptr;  // grouped: the submission's expert offsets [E]
  uint8_t* row_codes = nullptr;
  uint8_t* row_scales = nullptr;
  float* row_gscale = nullptr;
  uint8_t* col_codes = nullptr;
  uint8_t* col_scales = nullptr;
  float* col_gscale = nullptr;
  cudaEvent_t in_done = nullptr, quant_done = nullptr, out_done = nullptr;
};

bool ok(cudaError_t e) { return e == cudaSuccess; }

}  // namespace

struct nvfp4_host_pipeline {
  int device = 0;
  int64_t M = 0, N = 0;
  int32_t E = 0;             // grouped: experts (0: plain tensors)
  int64_t col_capacity = 0;  // grouped: columns of the columnwise outputs
  nvfp4_config cfg{};
  bool row = false, col = false;
  int depth = 0;
  uint64_t submitted = 0;
  cudaStream_t s_in = nullptr, s_quant = nullptr, s_out = nullptr;
  cudaEvent_t caller = nullptr;  // the caller's stream position at submission
  Slot slot[kMaxDepth];
};

namespace {

// Restores the caller's current device on scope exit.
struct DeviceGuard {
  int prev = -1;
  bool ok_ = false;
  explicit DeviceGuard(int dev) {
    ok_ = cudaGetDevice(&prev) == cudaSuccess && (prev == dev || cudaSetDevice(dev) == cudaSuccess);
  }
  ~DeviceGuard() {
    int cur = -1;
    if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
  }
};

void release(nvfp4_host_pipeline* p) {
  for (cudaStream_t s : {p->s_in, p->s_quant, p->s_out})
    if (s) cudaStreamSynchronize(s);
  for (int k = 0; k < kMaxDepth; k++) {
    Slot& sl = p->slot[k];
    for (void* b : {sl.x, (void*)sl.offsets, (void*)sl.row_codes, (void*)sl.row_scales,
                    (void*)sl.row_gscale,
                    (void*)sl.col_codes, (void*)sl.col_scales, (void*)sl.col_gscale})
      if (b) cudaFree(b);
    for (cudaEvent_t e : {sl.in_done, sl.quant_done, sl.out_done})
      if (e) cudaEventDestroy(e);
  }
  for (cudaStream_t s : {p->s_in, p->s_quant, p->s_out})
    if (s) cudaStreamDestroy(s);
  if (p->caller) cudaEventDestroy(p->caller);
  delete p;
}

template <typename T>
bool alloc(T** out, size_t bytes) {
  void* b = nullptr;
  if (!ok(cudaMalloc(&b, bytes))) return false;
  *out = static_cast<T*>(b);
  return true;
}

}  // namespace

namespace {

// Shared by both create calls: E = 0 for plain tensors [M][N]; grouped tensors [T = M][H = N]
// with E experts and col_capacity columns of columnwise outputs.
nvfp4_status create(int64_t M, int64_t N, int32_t E, int64_t cap, const nvfp4_config* cfg,
                    int32_t depth, nvfp4_host_pipeline** out) {
  if (cfg != nullptr && cfg->swizzle_scales != 0) return NVFP4_ERR_UNSUPPORTED;
  if (out == nullptr || cfg == nullptr || (cfg->fast_math != 0 && cfg->fast_math != 1))
    return NVFP4_ERR_INVALID_ARG;
  *out = nullptr;
  if (depth < 1 || depth > kMaxDepth) return NVFP4_ERR_INVALID_ARG;
  const bool row = cfg->rowwise != 0, col = cfg->columnwise != 0;
  if (!row && !col) return NVFP4_ERR_UNSUPPORTED;
  if (M <= 0 || N <= 0) return NVFP4_ERR_SHAPE;
  if (E > 0) {
    if (cfg->fused_amax != 0) return NVFP4_ERR_UNSUPPORTED;
    if (N % 16 != 0 || (col && (cap <= 0 || cap % 16 != 0))) return NVFP4_ERR_SHAPE;
  } else if (N % 16 != 0 || ((col || cfg->block2d) && M % 16 != 0)) {
    return NVFP4_ERR_SHAPE;
  }
  nvfp4_host_pipeline* p = new (std::nothrow) nvfp4_host_pipeline;
  if (p == nullptr) return NVFP4_ERR_CUDA;
  if (!ok(cudaGetDevice(&p->device))) { delete p; return NVFP4_ERR_CUDA; }
  p->M = M;
  p->N = N;
  p->E = E;
  p->col_capacity = E > 0 ? cap : M;
  p->cfg = *cfg;
  p->row = row;
  p->col = col;
  p->depth = depth;
  const size_t elems = (size_t)M * (size_t)N;
  const size_t col_elems = (size_t)p->col_capacity * (size_t)N;
  const size_t gscale = 2 * sizeof(float) * (size_t)(E > 0 ? E : 1);
  bool good = ok(cudaStreamCreateWithFlags(&p->s_in, cudaStreamNonBlocking)) &&
              ok(cudaStreamCreateWithFlags(&p->s_quant, cudaStreamNonBlocking)) &&
              ok(cudaStreamCreateWithFlags(&p->s_out, cudaStreamNonBlocking)) &&
              ok(cudaEventCreateWithFlags(&p->caller, cudaEventDisableTiming));
  for (int k = 0; good && k < depth; k++) {
    Slot& sl = p->slot[k];
    good = alloc(&sl.x, elems * 2) &&
           (E == 0 || alloc(&sl.offsets, sizeof(int32_t) * (size_t)E)) &&
           (!row || (alloc(&sl.row_codes, elems / 2) && alloc(&sl.row_scales, elems / 16) &&
                     alloc(&sl.row_gscale, gscale))) &&
           (!col || (alloc(&sl.col_codes, col_elems / 2) && alloc(&sl.col_scales, col_elems / 16) &&
                     alloc(&sl.col_gscale, gscale))) &&
           ok(cudaEventCreateWithFlags(&sl.in_done, cudaEventDisableTiming)) &&
           ok(cudaEventCreateWithFlags(&sl.quant_done, cudaEventDisableTiming)) &&
           ok(cudaEventCreateWithFlags(&sl.out_done, cudaEventDisableTiming));
  }
  if (!good) {
    release(p);
    return NVFP4_ERR_CUDA;
  }
  *out = p;
  return NVFP4_OK;
}

nvfp4_status submit(nvfp4_host_pipeline* p, const void* x_host, const int32_t* offsets_host,
                    uint8_t* row_codes, uint8_t* row_scales, float* row_gscale,
                    uint8_t* col_codes, uint8_t* col_scales, float* col_gscale, void* stream) {
  if (p == nullptr || x_host == nullptr || ((p->E > 0) != (offsets_host != nullptr)))
    return NVFP4_ERR_INVALID_ARG;
  if ((p->row && (row_codes == nullptr || row_scales == nullptr || row_gscale == nullptr)) ||
      (p->col && (col_codes == nullptr || col_scales == nullptr || col_gscale == nullptr)))
    return NVFP4_ERR_INVALID_ARG;
  DeviceGuard guard(p->device);
  if (!guard.ok_) return NVFP4_ERR_CUDA;
  // The rows and columnwise columns the quantization writes: all of them for a plain tensor;
  // for a grouped one the experts' rows [0, offsets[E-1]) and their padded columnwise blocks
  // [0, sum_e pad16(n_e)), so that the rest of the caller's host buffers stays untouched, as
  // with nvfp4_quantize_grouped. Offsets that break its rules are refused here.
  int64_t rows_out = p->M, cols_out = p->col_capacity;
  if (p->E > 0) {
    int64_t prev = 0, used = 0;
    for (int32_t e = 0; e < p->E; e++) {
      const int64_t end = offsets_host[e];
      if (end < prev || end > p->M) return NVFP4_ERR_INVALID_ARG;
      used += (end - prev + 15) / 16 * 16;
      prev = end;
    }
    if (p->col && used > p->col_capacity) return NVFP4_ERR_INVALID_ARG;
    rows_out = prev;
    cols_out = used;
  }
  Slot& sl = p->slot[p->submitted % (uint64_t)p->depth];
  const size_t elems = (size_t)p->M * (size_t)p->N;
  const size_t row_elems = (size_t)rows_out * (size_t)p->N;
  const size_t gscale = 2 * sizeof(float) * (size_t)(p->E > 0 ? p->E : 1);
  cudaStream_t caller = static_cast<cudaStream_t>(stream);
  // copy in: after the caller's earlier work and after the slot's previous input was read
  if (!ok(cudaEventRecord(p->caller, caller)) || !ok(cudaStreamWaitEvent(p->s_in, p->caller, 0)) ||
      !ok(cudaStreamWaitEvent(p->s_in, sl.quant_done, 0)) ||
      !ok(cudaMemcpyAsync(sl.x, x_host, elems * 2, cudaMemcpyHostToDevice, p->s_in)) ||
      (p->E > 0 && !ok(cudaMemcpyAsync(sl.offsets, offsets_host, sizeof(int32_t) * (size_t)p->E,
                                       cudaMemcpyHostToDevice, p->s_in))) ||
      !ok(cudaEventRecord(sl.in_done, p->s_in)))
    return NVFP4_ERR_CUDA;
  // quantize: after the copy in and after the slot's previous outputs were copied out
  if (!ok(cudaStreamWaitEvent(p->s_quant, sl.in_done, 0)) ||
      !ok(cudaStreamWaitEvent(p->s_quant, sl.out_done, 0)))
    return NVFP4_ERR_CUDA;
  const nvfp4_status st =
      p->E > 0 ? nvfp4_quantize_grouped(sl.x, p->M, p->N, sl.offsets, p->E, p->col_capacity,
                                        &p->cfg, nullptr, nullptr, sl.row_codes, sl.row_scales,
                                        sl.row_gscale, sl.col_codes, sl.col_scales,
                                        sl.col_gscale, p->s_quant)
               : nvfp4_quantize(sl.x, p->M, p->N, &p->cfg, nullptr, nullptr, sl.row_codes,
                                sl.row_scales, sl.row_gscale, sl.col_codes, sl.col_scales,
                                sl.col_gscale, p->s_quant);
  if (st != NVFP4_OK) return st;
  if (!ok(cudaEventRecord(sl.quant_done, p->s_quant)) ||
      !ok(cudaStreamWaitEvent(p->s_out, sl.quant_done, 0)))
    return NVFP4_ERR_CUDA;
  // copy out, largest buffers first (columnwise rows of col_capacity columns, of which the
  // first cols_out were written)
  bool good = true;
  const size_t cpitch = (size_t)p->col_capacity;
  if (p->col && cols_out == p->col_capacity)  // every column: one contiguous copy each
    good = good && ok(cudaMemcpyAsync(col_codes, sl.col_codes, cpitch * p->N / 2, cudaMemcpyDeviceToHost, p->s_out)) &&
           ok(cudaMemcpyAsync(col_scales, sl.col_scales, cpitch * p->N / 16, cudaMemcpyDeviceToHost, p->s_out));
  else if (p->col && cols_out > 0)
    good = good && ok(cudaMemcpy2DAsync(col_codes, cpitch / 2, sl.col_codes, cpitch / 2,
                                        (size_t)cols_out / 2, (size_t)p->N,
                                        cudaMemcpyDeviceToHost, p->s_out)) &&
           ok(cudaMemcpy2DAsync(col_scales, cpitch / 16, sl.col_scales, cpitch / 16,
                                (size_t)cols_out / 16, (size_t)p->N, cudaMemcpyDeviceToHost,
                                p->s_out));
  if (p->col)
    good = good && ok(cudaMemcpyAsync(col_gscale, sl.col_gscale, gscale, cudaMemcpyDeviceToHost, p->s_out));
  if (p->row && row_elems > 0)
    good = good && ok(cudaMemcpyAsync(row_codes, sl.row_codes, row_elems / 2, cudaMemcpyDeviceToHost, p->s_out)) &&
           ok(cudaMemcpyAsync(row_scales, sl.row_scales, row_elems / 16, cudaMemcpyDeviceToHost, p->s_out));
  if (p->row)
    good = good && ok(cudaMemcpyAsync(row_gscale, sl.row_gscale, gscale, cudaMemcpyDeviceToHost, p->s_out));
  if (!good || !ok(cudaEventRecord(sl.out_done, p->s_out))) return NVFP4_ERR_CUDA;
  p->submitted++;
  return NVFP4_OK;
}

}  // namespace

NVFP4_EXPORT nvfp4_status nvfp4_host_pipeline_create(int64_t M, int64_t N,
                                                     const nvfp4_config* cfg, int32_t depth,
                                                     nvfp4_host_pipeline** out) {
  return create(M, N, 0, 0, cfg, depth, out);
}

NVFP4_EXPORT nvfp4_status nvfp4_host_pipeline_create_grouped(int64_t T, int64_t H, int32_t E,
                                                             int64_t col_capacity,
                                                             const nvfp4_config* cfg,
                                                             int32_t depth,
                                                             nvfp4_host_pipeline** out) {
  if (E < 1 || E > 256) return NVFP4_ERR_INVALID_ARG;
  return create(T, H, E, col_capacity, cfg, depth, out);
}

NVFP4_EXPORT nvfp4_status nvfp4_host_pipeline_submit(nvfp4_host_pipeline* p, const void* x_host,
                                                     uint8_t* row_codes, uint8_t* row_scales,
                                                     float* row_gscale, uint8_t* col_codes,
                                                     uint8_t* col_scales, float* col_gscale,
                                                     void* stream) {
  return submit(p, x_host, nullptr, row_codes, row_scales, row_gscale, col_codes, col_scales,
                col_gscale, stream);
}

NVFP4_EXPORT nvfp4_status nvfp4_host_pipeline_submit_grouped(
    nvfp4_host_pipeline* p, const void* x_host, const int32_t* offsets_host, uint8_t* row_codes,
    uint8_t* row_scales, float* row_gscale, uint8_t* col_codes, uint8_t* col_scales,
    float* col_gscale, void* stream) {
  if (offsets_host == nullptr) return NVFP4_ERR_INVALID_ARG;
  return submit(p, x_host, offsets_host, row_codes, row_scales, row_gscale, col_codes,
                col_scales, col_gscale, stream);
}

NVFP4_EXPORT nvfp4_status nvfp4_host_pipeline_join(nvfp4_host_pipeline* p, void* stream) {
  if (p == nullptr) return NVFP4_ERR_INVALID_ARG;
  if (p->submitted == 0) return NVFP4_OK;
  DeviceGuard guard(p->device);
  if (!guard.ok_) return NVFP4_ERR_CUDA;
  // the copy-out stream runs in submission order: its last event covers every submission
  const Slot& last = p->slot[(p->submitted - 1) % (uint64_t)p->depth];
  return ok(cudaStreamWaitEvent(static_cast<cudaStream_t>(stream), last.out_done, 0))
             ? NVFP4_OK : NVFP4_ERR_CUDA;
}

NVFP4_EXPORT nvfp4_status nvfp4_host_pipeline_destroy(nvfp4_host_pipeline* p) {
  if (p == nullptr) return NVFP4_OK;
  DeviceGuard guard(p->device);
  release(p);
  return NVFP4_OK;
}
