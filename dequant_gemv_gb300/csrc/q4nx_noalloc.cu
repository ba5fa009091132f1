// q4nx_noalloc.cu -- q4nx_gemv_noalloc: the fused decode + GEMV with its scratch
// memory built into the library, for callers that cannot allocate device memory.
//
// The GEMV needs scratch (an error word and the posted partial sums of tile
// rows shared between CTAs, 16 B + 256 KiB whatever the weight's size).  q4nx_gemv takes it from
// the caller; this entry point instead uses kNoAllocScratchBytes of statically
// allocated device memory that every GPU loading the library holds until the
// process exits.  Host code never dereferences the array's name: the device
// address of the current device's copy is looked up with cudaGetSymbolAddress
// on every call (a host-side lookup; it stays right after a device reset, which
// can load the library's device code at another address) and passed to the
// kernel like any other pointer.
#include <cstdint>

#include "../../include/q4nx.h"
#include "q4nx_checks.h"
#include "q4nx_device.cuh"
#include "q4nx_kernels.h"

namespace q4nx {
namespace {

constexpr uint64_t kNoAllocScratchBytes = uint64_t(1) << 20;   // 1 MiB

static __device__ __align__(256) uint8_t g_gemv_scratch[kNoAllocScratchBytes];

// Device address of the current device's copy of the scratch array.
cudaError_t scratch_address(void** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_gemv_scratch);
  if (e != cudaSuccess) return e;
  *out = p;
  return cudaSuccess;
}

}  // namespace
}  // namespace q4nx

using namespace q4nx;

extern "C" {

uint64_t q4nx_noalloc_scratch_bytes(void) { return kNoAllocScratchBytes; }

int q4nx_gemv_noalloc(const q4nx_weight* w, const void* x_dev, void* y_dev, int out_dtype, void* stream) {
  // the same checks, in the same order, as q4nx_gemv
  int st = check_weight(w);
  if (st) return st;
  if (x_dev == nullptr || y_dev == nullptr) return Q4NX_E_NULL;
  if (out_dtype != Q4NX_OUT_BF16 && out_dtype != Q4NX_OUT_F32) return Q4NX_E_DTYPE;
  if (!aligned16(x_dev) || !aligned16(y_dev)) return Q4NX_E_ALIGN;
  const int64_t TR = w->rows / 32, TC = w->cols / 256;
  const uint64_t need = gemv_workspace_bytes(TR, TR * TC);
  if (need > kNoAllocScratchBytes) return Q4NX_E_WORKSPACE;          // cannot happen: the need is a constant
  void* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return Q4NX_E_CUDA;
  DeviceInfo info;
  if (device_info(&info) != cudaSuccess) return Q4NX_E_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The error word and the posted words (value + ready flag) must start at
  // zero; the array keeps whatever the previous call left, an abandoned call
  // included, so clear them.
  if (cudaMemsetAsync(scratch, 0, need, s) != cudaSuccess) return Q4NX_E_CUDA;
  GemvItem item;
  item.chunks = w->chunks_dev;
  item.x = x_dev;
  item.y = y_dev;
  item.TR = TR;
  item.TC = TC;
  return launch_gemv_batch(w->kind, &item, 1, out_dtype == Q4NX_OUT_F32, scratch, info, s) ==
                 cudaSuccess
             ? Q4NX_OK
             : Q4NX_E_CUDA;
}

int q4nx_check_noalloc(void* stream) {
  void* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return Q4NX_E_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t err = 0;
  if (cudaMemcpyAsync(&err, scratch, sizeof err, cudaMemcpyDeviceToHost, s) != cudaSuccess) return Q4NX_E_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return Q4NX_E_CUDA;
  if (err == 0) return Q4NX_OK;
  // a wait gave up: clear the whole array (a call that gave up may have left
  // posted sums in it; the next call clears what it uses anyway)
  if (cudaMemsetAsync(scratch, 0, kNoAllocScratchBytes, s) != cudaSuccess) return Q4NX_E_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return Q4NX_E_CUDA;
  return Q4NX_E_DEVICE_TIMEOUT;
}

}  // extern "C"
