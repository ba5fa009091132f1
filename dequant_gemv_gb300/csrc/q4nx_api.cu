// q4nx_api.cu -- the C ABI of libq4nx.so (declared in include/q4nx.h).
//
// Validation follows the "Q4NX chunks" section of the 1bit engine "NPU engine"
// page: a tensor's chunk kind must be one of the known sizes and the tensor
// must not be shorter than its layout needs; everything is checked before any
// work is enqueued, and no C++ exception crosses this boundary.
#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <set>
#include <utility>

#include "../../include/q4nx.h"
#include "q4nx_checks.h"
#include "q4nx_device.cuh"
#include "q4nx_kernels.h"

namespace q4nx {

namespace {
constexpr int kMaxDevices = 64;
std::atomic<int> g_sms[kMaxDevices];
std::atomic<int> g_smem[kMaxDevices];
std::atomic<int> g_smem_pair[kMaxDevices];
// the (device, kernel) pairs whose dynamic shared-memory limit has been raised
std::mutex g_attr_mu;
std::set<std::pair<int, const void*>> g_attr_set;
}  // namespace

cudaError_t device_info(DeviceInfo* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  int sms = g_sms[dev].load(std::memory_order_relaxed);
  int smem = g_smem[dev].load(std::memory_order_relaxed);
  int pair = g_smem_pair[dev].load(std::memory_order_relaxed);
  if (sms <= 0 || smem <= 0 || pair <= 0) {
    int per_sm = 0, reserved = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev);
    if (e != cudaSuccess) return e;
    pair = per_sm / 2 - reserved;
    if (pair > smem) pair = smem;
    if (pair < 1) pair = 1;
    g_sms[dev].store(sms, std::memory_order_relaxed);
    g_smem[dev].store(smem, std::memory_order_relaxed);
    g_smem_pair[dev].store(pair, std::memory_order_relaxed);
  }
  out->sms = sms;
  out->max_smem_optin = smem;
  out->smem_two_per_sm = pair;
  return cudaSuccess;
}

// Raise a kernel's dynamic shared-memory limit to the device maximum (less the
// kernel's static shared memory), once per (device, kernel).
cudaError_t set_max_dynamic_smem(const void* func) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices || func == nullptr) return cudaErrorInvalidValue;
  {
    std::lock_guard<std::mutex> lock(g_attr_mu);
    if (g_attr_set.count({dev, func})) return cudaSuccess;
  }
  DeviceInfo info;
  e = device_info(&info);
  if (e != cudaSuccess) return e;
  // the opt-in limit covers static and dynamic shared memory together
  cudaFuncAttributes fa;
  e = cudaFuncGetAttributes(&fa, func);
  if (e != cudaSuccess) return e;
  const int dyn = info.max_smem_optin - static_cast<int>(fa.sharedSizeBytes);
  if (dyn <= 0) return cudaErrorInvalidValue;
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_attr_mu);
  g_attr_set.insert({dev, func});
  return cudaSuccess;
}

}  // namespace q4nx

using namespace q4nx;

namespace q4nx {

int check_grid(int64_t rows, int64_t cols) {
  if (rows <= 0 || cols <= 0 || rows % 32 != 0 || cols % 256 != 0) return Q4NX_E_SHAPE;
  if (rows / 32 > (int64_t(1) << 31) / (cols / 256)) return Q4NX_E_SHAPE;    // tile count must fit 31 bits
  return Q4NX_OK;
}

int check_weight(const q4nx_weight* w) {
  if (w == nullptr || w->chunks_dev == nullptr) return Q4NX_E_NULL;
  const uint64_t cb = q4nx_chunk_bytes(w->kind);
  if (cb == 0 || w->reserved != 0) return Q4NX_E_KIND;
  int st = check_grid(w->rows, w->cols);
  if (st) return st;
  const uint64_t need = static_cast<uint64_t>(w->rows / 32) * static_cast<uint64_t>(w->cols / 256) * cb;
  if (w->bytes < need) return Q4NX_E_SHORT;
  if (!aligned16(w->chunks_dev)) return Q4NX_E_ALIGN;
  return Q4NX_OK;
}

}  // namespace q4nx

namespace {

int from_cuda(cudaError_t e) { return e == cudaSuccess ? Q4NX_OK : Q4NX_E_CUDA; }

}  // namespace

extern "C" {

uint64_t q4nx_chunk_bytes(int kind) { return static_cast<uint64_t>(chunk_bytes_of(kind)); }

int q4nx_abi_version(void) { return 1; }

const char* q4nx_status_str(int status) {
  switch (status) {
    case Q4NX_OK: return "ok";
    case Q4NX_E_NULL: return "a required pointer is NULL";
    case Q4NX_E_KIND: return "unknown chunk kind";
    case Q4NX_E_SHAPE: return "rows must be a positive multiple of 32 and cols of 256";
    case Q4NX_E_SHORT: return "buffer shorter than its layout needs";
    case Q4NX_E_ALIGN: return "device buffer not 16-byte aligned";
    case Q4NX_E_M: return "M must be in 1..64";
    case Q4NX_E_WORKSPACE: return "workspace missing or too small";
    case Q4NX_E_UNSUPPORTED: return "kind or size not supported by this operation";
    case Q4NX_E_CUDA: return "CUDA launch failed";
    case Q4NX_E_DEVICE_TIMEOUT: return "a bounded in-kernel wait gave up";
    case Q4NX_E_DTYPE: return "unknown output dtype";
    default: return "unknown status";
  }
}

int q4nx_decode(const q4nx_weight* w, void* out_dev, uint64_t out_bytes, void* stream) {
  int st = check_weight(w);
  if (st) return st;
  if (out_dev == nullptr) return Q4NX_E_NULL;
  if (out_bytes < static_cast<uint64_t>(w->rows) * static_cast<uint64_t>(w->cols) * 2) return Q4NX_E_SHORT;
  if (!aligned16(out_dev)) return Q4NX_E_ALIGN;
  return from_cuda(launch_decode(w->kind, w->chunks_dev, w->rows / 32, w->cols / 256, out_dev,
                                 static_cast<cudaStream_t>(stream)));
}

uint64_t q4nx_gemv_workspace(const q4nx_weight* w) {
  if (w == nullptr || check_grid(w->rows, w->cols) != Q4NX_OK) return 0;
  return gemv_workspace_bytes(w->rows / 32, (w->rows / 32) * (w->cols / 256));
}

uint64_t q4nx_gemv_batch_workspace(const q4nx_gemv_item* items, int count) {
  if (items == nullptr || count < 1 || count > Q4NX_MAX_BATCH) return 0;
  int64_t tr = 0, t = 0;
  for (int i = 0; i < count; ++i) {
    const q4nx_weight& w = items[i].w;
    if (check_grid(w.rows, w.cols) != Q4NX_OK) return 0;
    tr += w.rows / 32;
    t += (w.rows / 32) * (w.cols / 256);
  }
  return gemv_workspace_bytes(tr, t);
}

int q4nx_gemv_batch(const q4nx_gemv_item* items, int count, int out_dtype, void* workspace_dev,
                    uint64_t workspace_bytes, void* stream) {
  if (items == nullptr) return Q4NX_E_NULL;
  if (count < 1 || count > Q4NX_MAX_BATCH) return Q4NX_E_SHAPE;
  if (out_dtype != Q4NX_OUT_BF16 && out_dtype != Q4NX_OUT_F32) return Q4NX_E_DTYPE;
  GemvItem it[kMaxGemvItems];
  int64_t tr = 0, t = 0;
  for (int i = 0; i < count; ++i) {
    const q4nx_gemv_item& item = items[i];
    int st = check_weight(&item.w);
    if (st) return st;
    if (item.w.kind != items[0].w.kind) return Q4NX_E_KIND;
    if (item.x_dev == nullptr || item.y_dev == nullptr) return Q4NX_E_NULL;
    if (!aligned16(item.x_dev) || !aligned16(item.y_dev)) return Q4NX_E_ALIGN;
    it[i].chunks = item.w.chunks_dev;
    it[i].x = item.x_dev;
    it[i].y = item.y_dev;
    it[i].TR = item.w.rows / 32;
    it[i].TC = item.w.cols / 256;
    tr += it[i].TR;
    t += it[i].TR * it[i].TC;
  }
  if (t > (int64_t(1) << 40) || tr > (int64_t(1) << 31)) return Q4NX_E_SHAPE;
  if (workspace_dev == nullptr || workspace_bytes < gemv_workspace_bytes(tr, t)) return Q4NX_E_WORKSPACE;
  if (!aligned16(workspace_dev)) return Q4NX_E_ALIGN;
  DeviceInfo info;
  if (device_info(&info) != cudaSuccess) return Q4NX_E_CUDA;
  return from_cuda(launch_gemv_batch(items[0].w.kind, it, count, out_dtype == Q4NX_OUT_F32, workspace_dev, info,
                                     static_cast<cudaStream_t>(stream)));
}

int q4nx_gemv(const q4nx_weight* w, const void* x_dev, void* y_dev, int out_dtype, void* workspace_dev,
              uint64_t workspace_bytes, void* stream) {
  int st = check_weight(w);
  if (st) return st;
  if (x_dev == nullptr || y_dev == nullptr) return Q4NX_E_NULL;
  q4nx_gemv_item item;
  item.w = *w;
  item.x_dev = x_dev;
  item.y_dev = y_dev;
  return q4nx_gemv_batch(&item, 1, out_dtype, workspace_dev, workspace_bytes, stream);
}

int q4nx_gemv_top1(const q4nx_weight* w, const void* x_dev, int32_t* idx_dev, void* workspace_dev,
                   uint64_t workspace_bytes, void* stream) {
  int st = check_weight(w);
  if (st) return st;
  if (x_dev == nullptr || idx_dev == nullptr) return Q4NX_E_NULL;
  if (!aligned16(x_dev) || (reinterpret_cast<uintptr_t>(idx_dev) & 3u)) return Q4NX_E_ALIGN;
  const int64_t TR = w->rows / 32, TC = w->cols / 256;
  if (workspace_dev == nullptr || workspace_bytes < gemv_workspace_bytes(TR, TR * TC)) return Q4NX_E_WORKSPACE;
  if (!aligned16(workspace_dev)) return Q4NX_E_ALIGN;
  DeviceInfo info;
  if (device_info(&info) != cudaSuccess) return Q4NX_E_CUDA;
  GemvItem item;
  item.chunks = w->chunks_dev;
  item.x = x_dev;
  item.y = nullptr;
  item.TR = TR;
  item.TC = TC;
  return from_cuda(launch_gemv_top1(w->kind, item, idx_dev, nullptr, 0u, workspace_dev, info,
                                    static_cast<cudaStream_t>(stream)));
}

int q4nx_gemv_top1_key(const q4nx_weight* w, const void* x_dev, int64_t row_base, int64_t* key_dev,
                       void* workspace_dev, uint64_t workspace_bytes, void* stream) {
  int st = check_weight(w);
  if (st) return st;
  if (x_dev == nullptr || key_dev == nullptr) return Q4NX_E_NULL;
  if (row_base < 0 || row_base > static_cast<int64_t>(INT32_MAX) - w->rows) return Q4NX_E_SHAPE;
  if (!aligned16(x_dev) || (reinterpret_cast<uintptr_t>(key_dev) & 7u)) return Q4NX_E_ALIGN;
  const int64_t TR = w->rows / 32, TC = w->cols / 256;
  if (workspace_dev == nullptr || workspace_bytes < gemv_workspace_bytes(TR, TR * TC)) return Q4NX_E_WORKSPACE;
  if (!aligned16(workspace_dev)) return Q4NX_E_ALIGN;
  DeviceInfo info;
  if (device_info(&info) != cudaSuccess) return Q4NX_E_CUDA;
  GemvItem item;
  item.chunks = w->chunks_dev;
  item.x = x_dev;
  item.y = nullptr;
  item.TR = TR;
  item.TC = TC;
  return from_cuda(launch_gemv_top1(w->kind, item, nullptr, key_dev, static_cast<uint32_t>(row_base), workspace_dev,
                                    info, static_cast<cudaStream_t>(stream)));
}

// Workspace of q4nx_gemm_m64: the GEMM's part (error word, partial tiles,
// posting counters; partial tiles stay behind after a call) followed by the
// few-token GEMV's part (posted row sums, left zero-filled).  Both share the
// error word at offset 0, and one size serves every M.
static uint64_t gemm_part_bytes(const q4nx_weight* w) {
  return align16(gemm_workspace_bytes(w->rows / 32, w->cols / 256, 64));
}

uint64_t q4nx_gemm_workspace(const q4nx_weight* w, int M) {
  if (w == nullptr || check_grid(w->rows, w->cols) != Q4NX_OK || M < 1 || M > 64) return 0;
  return gemm_part_bytes(w) + gemv_workspace_bytes(w->rows / 32, (w->rows / 32) * (w->cols / 256), kGemvTokensMax);
}

int q4nx_gemm_m64(const q4nx_weight* w, const void* X_dev, int M, void* Y_dev, int out_dtype, void* workspace_dev,
                  uint64_t workspace_bytes, void* stream) {
  int st = check_weight(w);
  if (st) return st;
  if (X_dev == nullptr || Y_dev == nullptr) return Q4NX_E_NULL;
  if (M < 1 || M > 64) return Q4NX_E_M;
  if (out_dtype != Q4NX_OUT_BF16 && out_dtype != Q4NX_OUT_F32) return Q4NX_E_DTYPE;
  if (!aligned16(X_dev) || !aligned16(Y_dev)) return Q4NX_E_ALIGN;
  const bool tokens = M <= gemv_max_tokens(w->kind);
  if (!tokens && !gemm_supports(w->kind)) return Q4NX_E_UNSUPPORTED;
  if (workspace_dev == nullptr || workspace_bytes < q4nx_gemm_workspace(w, M)) return Q4NX_E_WORKSPACE;
  if (!aligned16(workspace_dev)) return Q4NX_E_ALIGN;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (tokens) {
    // a few tokens: each chunk is decoded once for all of them on the CUDA
    // cores, cheaper than the tensor-core path's decode of every weight to bf16
    DeviceInfo info;
    if (device_info(&info) != cudaSuccess) return Q4NX_E_CUDA;
    GemvItem item;
    item.chunks = w->chunks_dev;
    item.x = X_dev;
    item.y = Y_dev;
    item.TR = w->rows / 32;
    item.TC = w->cols / 256;
    uint8_t* ws = static_cast<uint8_t*>(workspace_dev);
    return from_cuda(launch_gemv_tokens(w->kind, item, M, out_dtype == Q4NX_OUT_F32, reinterpret_cast<uint32_t*>(ws),
                                        ws + gemm_part_bytes(w), info, s));
  }
  return from_cuda(launch_gemm(w->kind, w->chunks_dev, w->rows / 32, w->cols / 256, X_dev, M, Y_dev,
                               out_dtype == Q4NX_OUT_F32, workspace_dev, s));
}

int q4nx_pack_q4_1(int src_type, const void* src_dev, uint64_t src_bytes, int64_t rows, int64_t cols, void* out_dev,
                   uint64_t out_bytes, void* stream) {
  if (src_dev == nullptr || out_dev == nullptr) return Q4NX_E_NULL;
  const int bpb = pack_src_bytes_per_32(src_type);
  if (bpb == 0) return Q4NX_E_KIND;
  int st = check_grid(rows, cols);
  if (st) return st;
  const uint64_t T = static_cast<uint64_t>(rows / 32) * static_cast<uint64_t>(cols / 256);
  if (src_bytes < static_cast<uint64_t>(rows) * static_cast<uint64_t>(cols / 32) * bpb || out_bytes < T * kQ41Bytes)
    return Q4NX_E_SHORT;
  if (!aligned16(src_dev) || !aligned16(out_dev)) return Q4NX_E_ALIGN;
  return from_cuda(launch_pack_q4_1(src_type, src_dev, rows / 32, cols / 256, out_dev, static_cast<cudaStream_t>(stream)));
}

int q4nx_repack_q4k(const void* in_dev, uint64_t in_bytes, int64_t rows, int64_t cols, void* out_dev,
                    uint64_t out_bytes, void* stream) {
  if (in_dev == nullptr || out_dev == nullptr) return Q4NX_E_NULL;
  int st = check_grid(rows, cols);
  if (st) return st;
  const uint64_t T = static_cast<uint64_t>(rows / 32) * static_cast<uint64_t>(cols / 256);
  if (in_bytes < T * kQ4KBytes || out_bytes < T * kQ41Bytes) return Q4NX_E_SHORT;
  if (!aligned16(in_dev) || !aligned16(out_dev)) return Q4NX_E_ALIGN;
  return from_cuda(launch_repack_q4k(in_dev, rows / 32, cols / 256, out_dev, static_cast<cudaStream_t>(stream)));
}

int q4nx_argmax(const float* logits_dev, int M, int64_t V, int32_t* idx_dev, void* stream) {
  if (logits_dev == nullptr || idx_dev == nullptr) return Q4NX_E_NULL;
  if (M < 1 || M > 65535 || V < 1 || V >= (int64_t(1) << 31)) return Q4NX_E_SHAPE;
  if ((reinterpret_cast<uintptr_t>(logits_dev) & 3u) || (reinterpret_cast<uintptr_t>(idx_dev) & 3u))
    return Q4NX_E_ALIGN;
  return from_cuda(launch_argmax(logits_dev, M, V, idx_dev, static_cast<cudaStream_t>(stream)));
}

int q4nx_check(void* workspace_dev, void* stream) {
  if (workspace_dev == nullptr) return Q4NX_E_NULL;
  uint32_t err = 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(&err, workspace_dev, sizeof err, cudaMemcpyDeviceToHost, s) != cudaSuccess) return Q4NX_E_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return Q4NX_E_CUDA;
  if (err == 0) return Q4NX_OK;
  const uint32_t zero = 0;
  if (cudaMemcpyAsync(workspace_dev, &zero, sizeof zero, cudaMemcpyHostToDevice, s) != cudaSuccess) return Q4NX_E_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return Q4NX_E_CUDA;
  return Q4NX_E_DEVICE_TIMEOUT;
}

}  // extern "C"
