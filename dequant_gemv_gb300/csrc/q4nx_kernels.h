// q4nx_kernels.h -- host-side launchers of the Q4NX kernels (internal to libq4nx.so).
// The C ABI in include/q4nx.h validates arguments and then calls these.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace q4nx {

struct DeviceInfo {
  int sms = 0;
  int max_smem_optin = 0;      // dynamic shared memory one CTA may opt in to
  int smem_two_per_sm = 0;     // the most dynamic shared memory a CTA may use with two CTAs on one SM
};
// Properties of the current device (cached per device ordinal).
cudaError_t device_info(DeviceInfo* out);

// Raise a kernel's dynamic shared-memory limit to the device maximum once per
// (device, kernel).
cudaError_t set_max_dynamic_smem(const void* func);

// ---- GEMV (M = 1), a batch of independent items of one kind per launch ----
constexpr int kMaxGemvItems = 256;
struct GemvItem {
  const void* chunks;
  const void* x;
  void* y;
  int64_t TR, TC;
};
struct GemvPlan {
  int warps = 0;       // warps per CTA, each owning a contiguous part of the CTA's chunks
  int stages = 0;      // ring stages per warp
  int grid = 0;        // CTAs, each owning a contiguous range of chunks
  size_t smem = 0;     // dynamic shared memory bytes
  int xslots = 0;      // x-slice cache slots, one per slice holding every token (4-bit kinds)
  int quarter = 0;     // the units are quarters of chunks (small 4-bit launches, one token)
};
// tc: tile columns of the launch's one weight (several tokens), else 0
bool gemv_plan(int kind, int64_t total_chunks, const DeviceInfo& info, GemvPlan* plan, int tokens, int64_t tc = 0);
uint64_t gemv_workspace_bytes(int64_t total_tile_rows, int64_t total_chunks, int tokens = 1);
cudaError_t launch_gemv_batch(int kind, const GemvItem* items, int n, int out_f32, void* workspace,
                              const DeviceInfo& info, cudaStream_t s);

// GEMV of one item fused with top-1: the largest fp32 output (ties: lowest
// row; a NaN output wins, the first one), y not written.  Writes the row to
// *idx and/or the 64-bit key (top bit flipped, see q4nx.h) to *key, the rows
// numbered from row_base.  The workspace's bytes 4..15 hold the launch's
// top-1 words (zero between launches).
cudaError_t launch_gemv_top1(int kind, const GemvItem& item, int32_t* idx, int64_t* key, uint32_t row_base,
                             void* workspace, const DeviceInfo& info, cudaStream_t s);

// ---- GEMV of one weight against M tokens (X [M][cols], Y [M][rows]) ----
// Each chunk is read once for all M tokens.  M up to gemv_max_tokens(kind),
// the M up to which this beats the tensor-core GEMM on GB300 (measured: two
// tokens for q4_1, one for Q8, whose float path costs more per token); Q4_K
// has no tensor-core path, so it goes to four.  `workspace`:
// gemv_workspace_bytes(.., .., 4) bytes, zero-filled and left so; `err`: the
// error word to report a failed wait in.
constexpr int kGemvTokensQ41 = 2, kGemvTokensQ4K = 4, kGemvTokensQ8 = 1, kGemvTokensMax = 4;
int gemv_max_tokens(int kind);
cudaError_t launch_gemv_tokens(int kind, const GemvItem& item, int M, int out_f32, uint32_t* err, void* workspace,
                               const DeviceInfo& info, cudaStream_t s);

// ---- standalone decode ----
cudaError_t launch_decode(int kind, const void* chunks, int64_t TR, int64_t TC, void* out, cudaStream_t s);

// ---- Q4_K -> q4_1 repack ----
cudaError_t launch_repack_q4k(const void* in, int64_t TR, int64_t TC, void* out, cudaStream_t s);

// ---- GGUF-type tensor -> q4_1 chunks ----
enum : int { kSrcQ4_0 = 1, kSrcQ4_1 = 2, kSrcQ8_0 = 3, kSrcF32 = 4, kSrcF16 = 5, kSrcBF16 = 6 };
int pack_src_bytes_per_32(int src_type);        // 0 for an unknown type
cudaError_t launch_pack_q4_1(int src_type, const void* src, int64_t TR, int64_t TC, void* out, cudaStream_t s);

// ---- top-1 ----
cudaError_t launch_argmax(const float* logits, int M, int64_t V, int32_t* idx, cudaStream_t s);

// ---- GEMM (M <= 64, tcgen05) ----
bool gemm_supports(int kind);
uint64_t gemm_workspace_bytes(int64_t TR, int64_t TC, int M);
cudaError_t launch_gemm(int kind, const void* chunks, int64_t TR, int64_t TC, const void* X, int M, void* Y,
                        int out_f32, void* workspace, cudaStream_t s);

// Workspace layout shared by the GEMV launcher and kernel.
constexpr uint64_t kWsErrBytes = 16;              // error word (+ padding)
constexpr int kMaxCtas = 1024;                    // upper bound of CTAs per GEMV launch
__host__ __device__ inline uint64_t align16(uint64_t v) { return (v + 15) & ~uint64_t(15); }

}  // namespace q4nx
