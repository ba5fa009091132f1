// q4nx_gemm.cu -- fused decode + GEMM for blocks of up to 64 tokens (tcgen05).
#include "q4nx_device.cuh"
#include "q4nx_kernels.h"

namespace q4nx {

bool gemm_available() { return false; }

uint64_t gemm_workspace_bytes(int64_t, int64_t, int) { return kWsErrBytes; }

cudaError_t launch_gemm(int, const void*, int64_t, int64_t, const void*, int, void*, int, void*, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace q4nx
