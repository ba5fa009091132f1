// q4nx_noalloc.cu -- q4nx_gemv_noalloc: the fused decode + GEMV with its scratch
// memory built into the library, for callers that cannot allocate device memory.
//
// The GEMV needs scratch (an error word and the posted partial sums of tile
// rows shared between CTAs, 16 B + 256 KiB whatever the weight's size).  q4nx_gemv takes it from
// the caller; this entry point instead uses kNoAllocScratchBytes of statically
// allocated device memory that every GPU loading the library holds until the
// process exits.  Host code never dereferences the array's name: the device
// address is looked up once per device with cudaGetSymbolAddress and passed
// to the kernel like any other pointer.
#include <atomic>
#include <cstdint>

#include "../../include/q4nx.h"
#include "q4nx_device.cuh"
#include "q4nx_kernels.h"

namespace q4nx {
namespace {

constexpr uint64_t kNoAllocScratchBytes = uint64_t(1) << 20;   // 1 MiB
constexpr int kMaxDevicesNoAlloc = 64;

static __device__ __align__(256) uint8_t g_gemv_scratch[kNoAllocScratchBytes];

std::atomic<void*> g_scratch_addr[kMaxDevicesNoAlloc];

// Device address of this device's copy of the scratch array; looked up on the
// first call made with that device current.
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevicesNoAlloc) return cudaErrorInvalidDevice;
  void* p = g_scratch_addr[dev].load(std::memory_order_acquire);
  if (p == nullptr) {
    e = cudaGetSymbolAddress(&p, g_gemv_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev].store(p, std::memory_order_release);
  }
  *out = p;
  return cudaSuccess;
}

}  // namespace
}  // namespace q4nx

using namespace q4nx;

extern "C" {

uint64_t q4nx_noalloc_scratch_bytes(void) { return kNoAllocScratchBytes; }

int q4nx_gemv_noalloc(const q4nx_weight* w, const void* x_dev, void* y_dev, int out_dtype, void* stream) {
  if (w == nullptr || w->chunks_dev == nullptr || x_dev == nullptr || y_dev == nullptr) return Q4NX_E_NULL;
  const uint64_t cb = q4nx_chunk_bytes(w->kind);
  if (cb == 0 || w->reserved != 0) return Q4NX_E_KIND;
  if (w->rows <= 0 || w->cols <= 0 || w->rows % 32 != 0 || w->cols % 256 != 0) return Q4NX_E_SHAPE;
  const int64_t TR = w->rows / 32, TC = w->cols / 256;
  if (TR > (int64_t(1) << 31) / TC) return Q4NX_E_SHAPE;
  if (w->bytes < static_cast<uint64_t>(TR) * static_cast<uint64_t>(TC) * cb) return Q4NX_E_SHORT;
  if ((reinterpret_cast<uintptr_t>(w->chunks_dev) | reinterpret_cast<uintptr_t>(x_dev) |
       reinterpret_cast<uintptr_t>(y_dev)) & 15u)
    return Q4NX_E_ALIGN;
  if (out_dtype != Q4NX_OUT_BF16 && out_dtype != Q4NX_OUT_F32) return Q4NX_E_DTYPE;
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

}  // extern "C"
