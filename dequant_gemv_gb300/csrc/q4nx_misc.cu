// q4nx_misc.cu -- standalone decode, Q4_K -> q4_1 repack and top-1 kernels.
//
// Formulas: the "Q4NX chunks" section of the 1bit engine "NPU engine" page
// (chunk-kind table; the decoders-and-repack paragraph below it).  Greedy
// top-1: the page's "Serving" section (greedy decoding).
#include <algorithm>
#include <cooperative_groups.h>
#include <cuda_fp16.h>

#include "q4nx_device.cuh"
#include "q4nx_kernels.h"

namespace cg = cooperative_groups;

namespace q4nx {

// ------------------------------------------------------------- decode ----
//
// Every weight is formed in binary32 one operation at a time and rounded to
// bf16 nearest-even:  q4_1 (c*s)+z;  Q4_K ((S*sc)*c)+(M*mn);  Q8 d*c.
// The products are exact in binary32; __fmul_rn/__fadd_rn keep the compiler
// from contracting them into an FMA.

// 4-bit kinds: one CTA of 256 threads per chunk; warp w handles rows
// 4w..4w+3, lane L the 8 columns 8L..8L+7 (one 32-bit code word), and each
// row of 256 outputs is one coalesced 512-byte store.
template <int KIND>
__global__ void __launch_bounds__(256) decode_q4_kernel(const uint8_t* __restrict__ chunks, int64_t TC,
                                                        uint16_t* __restrict__ out) {
  constexpr int CB = chunk_bytes_of(KIND);
  const int64_t t = blockIdx.x;
  const int64_t tr = t / TC, tc = t - tr * TC;
  const int64_t K = TC * 256;
  const uint8_t* ch = chunks + t * CB;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int r = warp * 4 + j;
    const uint32_t w = __ldg(reinterpret_cast<const uint32_t*>(ch + r * 128) + lane);
    float s, z, S = 0.f, M = 0.f, sc = 0.f, mn = 0.f;
    if constexpr (KIND == kQ4_1) {
      s = bf16_bits_to_f32(__ldg(reinterpret_cast<const uint16_t*>(ch + kQ41Scale) + r * 8 + g));
      z = bf16_bits_to_f32(__ldg(reinterpret_cast<const uint16_t*>(ch + kQ41Zero) + r * 8 + g));
    } else {
      S = bf16_bits_to_f32(__ldg(reinterpret_cast<const uint16_t*>(ch + kQ4KS) + r));
      M = bf16_bits_to_f32(__ldg(reinterpret_cast<const uint16_t*>(ch + kQ4KM) + r));
      sc = static_cast<float>(__ldg(ch + kQ4KSc + r * 8 + g));
      mn = static_cast<float>(__ldg(ch + kQ4KMn + r * 8 + g));
      s = __fmul_rn(S, sc);      // exact
      z = __fmul_rn(M, mn);      // exact
    }
    uint32_t o[4];
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      const float c0 = static_cast<float>((w >> (8 * p)) & 0xF);
      const float c1 = static_cast<float>((w >> (8 * p + 4)) & 0xF);
      const float w0 = __fadd_rn(__fmul_rn(c0, s), z);
      const float w1 = __fadd_rn(__fmul_rn(c1, s), z);
      o[p] = static_cast<uint32_t>(f32_to_bf16_bits(w0)) | (static_cast<uint32_t>(f32_to_bf16_bits(w1)) << 16);
    }
    uint16_t* dst = out + (tr * 32 + r) * K + tc * 256 + lane * 8;
    *reinterpret_cast<uint4*>(dst) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// Q8 kinds: persistent CTAs, each walking the chunks c = blockIdx, +grid, ...
// through a two-stage ring filled by 1-D bulk copies (the next chunk is on its
// way while this one is decoded).  The codes are column-oriented, so a chunk
// is decoded from shared memory with lane = row, each thread forming 8
// consecutive columns; the decoded 32 x 256 tile is staged again in shared
// memory (rows padded by 16 bytes, so that the 16-byte writes of a warp's 32
// rows are free of bank conflicts) and leaves as one coalesced 512-byte store
// per row.  Waits are bounded: a copy that never lands ends the CTA early.
constexpr int kDecRowPitch = 512 + 16;
constexpr int kDecStage = kQ8Bytes;
constexpr int kDecQ8Smem = 2 * kDecStage + 32 * kDecRowPitch + 16;

__device__ __forceinline__ void decode_q8_fetch(uint8_t* dst, const uint8_t* src, uint64_t* bar) {
  mbar_arrive_expect_tx(bar, kQ8Bytes);
  bulk_g2s(dst, src, kQ8Bytes, bar);
}

template <int KIND>
__global__ void __launch_bounds__(256) decode_q8_kernel(const uint8_t* __restrict__ chunks, int64_t T, int64_t TC,
                                                        uint16_t* __restrict__ out) {
  extern __shared__ __align__(128) uint8_t dsm[];
  uint8_t* so = dsm + 2 * kDecStage;
  uint64_t* bar = reinterpret_cast<uint64_t*>(so + 32 * kDecRowPitch);
  const int64_t K = TC * 256;
  const int64_t stride = gridDim.x;
  if (threadIdx.x == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    fence_barrier_init();
    for (int st = 0; st < 2; ++st) {
      const int64_t c = blockIdx.x + st * stride;
      if (c < T) decode_q8_fetch(dsm + st * kDecStage, chunks + c * kQ8Bytes, &bar[st]);
    }
  }
  __syncthreads();
  const int r = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int i = 0;
  for (int64_t c = blockIdx.x; c < T; c += stride, ++i) {
    const int st = i & 1;
    if (!mbar_wait_bounded(&bar[st], (i >> 1) & 1)) break;
    const uint8_t* sc = dsm + st * kDecStage;
    const int64_t tr = c / TC, tc = c - tr * TC;
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      const int j = warp + 8 * jj;           // 8-column block 0..31
      const int gidx = j >> 2;
      const float d = bf16_bits_to_f32(reinterpret_cast<const uint16_t*>(sc + kQ8D)[r * 8 + gidx]);
      uint32_t o[4];
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        float wv[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int k = 8 * j + 2 * p + e;
          int off;
          if constexpr (KIND == kQ8_KR) off = k * 32 + r;
          else off = (r >> 4) * 4096 + (k >> 5) * 512 + (k & 31) * 16 + (r & 15);
          wv[e] = __fmul_rn(d, static_cast<float>(static_cast<int8_t>(sc[off])));
        }
        o[p] = static_cast<uint32_t>(f32_to_bf16_bits(wv[0])) | (static_cast<uint32_t>(f32_to_bf16_bits(wv[1])) << 16);
      }
      *reinterpret_cast<uint4*>(so + r * kDecRowPitch + j * 16) = make_uint4(o[0], o[1], o[2], o[3]);
    }
    __syncthreads();                         // the stage is read out and the tile is staged
    if (threadIdx.x == 0 && c + 2 * stride < T)
      decode_q8_fetch(dsm + st * kDecStage, chunks + (c + 2 * stride) * kQ8Bytes, &bar[st]);
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int row = warp * 4 + q;
      uint16_t* dst = out + (tr * 32 + row) * K + tc * 256 + lane * 8;
      *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(so + row * kDecRowPitch + lane * 16);
    }
    __syncthreads();                         // the staged tile is written out before the next one
  }
  // a CTA that stopped early lets its copies in flight land before it exits
  if (threadIdx.x == 0)
    for (int k = 0; k < 2; ++k) {
      const int64_t c = blockIdx.x + static_cast<int64_t>(i + k) * stride;
      if (c < T) mbar_wait_bounded(&bar[(i + k) & 1], ((i + k) >> 1) & 1);
    }
}

cudaError_t launch_decode(int kind, const void* chunks, int64_t TR, int64_t TC, void* out, cudaStream_t s) {
  const int64_t T = TR * TC;
  const uint8_t* c = static_cast<const uint8_t*>(chunks);
  uint16_t* o = static_cast<uint16_t*>(out);
  if (T > 0x7FFFFFFF) return cudaErrorInvalidValue;
  const dim3 grid(static_cast<unsigned>(T));
  switch (kind) {
    case kQ4_1: decode_q4_kernel<kQ4_1><<<grid, 256, 0, s>>>(c, TC, o); break;
    case kQ4_K: decode_q4_kernel<kQ4_K><<<grid, 256, 0, s>>>(c, TC, o); break;
    case kQ8_KR:
    case kQ8_BLK: {
      // persistent: as many CTAs as fit on the GPU at once, never more than chunks
      const void* f = kind == kQ8_KR ? reinterpret_cast<const void*>(decode_q8_kernel<kQ8_KR>)
                                     : reinterpret_cast<const void*>(decode_q8_kernel<kQ8_BLK>);
      cudaError_t e = set_max_dynamic_smem(f);
      if (e != cudaSuccess) return e;
      int dev = 0, sms = 0, per_sm = 0;
      if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
      if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
      if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, f, 256, kDecQ8Smem)) != cudaSuccess) return e;
      const int64_t g = std::min<int64_t>(T, static_cast<int64_t>(sms) * std::max(per_sm, 1));
      if (kind == kQ8_KR)
        decode_q8_kernel<kQ8_KR><<<static_cast<unsigned>(g), 256, kDecQ8Smem, s>>>(c, T, TC, o);
      else
        decode_q8_kernel<kQ8_BLK><<<static_cast<unsigned>(g), 256, kDecQ8Smem, s>>>(c, T, TC, o);
      break;
    }
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

// ------------------------------------------------------------- repack ----
//
// Q4_K chunk -> q4_1 chunk: the 4096 code bytes are copied unchanged;
// scale = bf16(S*sc), zero = bf16(M*mn) per (row, group).  S*sc and M*mn are
// exact binary32 products (8 x 8 significant bits), so the bf16 rounding is
// the only rounding.  One CTA of 256 threads per chunk.
__global__ void __launch_bounds__(256) repack_q4k_kernel(const uint8_t* __restrict__ in, uint8_t* __restrict__ out) {
  const int64_t t = blockIdx.x;
  const uint8_t* src = in + t * kQ4KBytes;
  uint8_t* dst = out + t * kQ41Bytes;
  const int i = threadIdx.x;                          // 256 threads: 16 B of codes each
  reinterpret_cast<uint4*>(dst)[i] = __ldg(reinterpret_cast<const uint4*>(src) + i);
  const int r = i >> 3;                               // (row, group) pair i = r*8 + g
  const float S = bf16_bits_to_f32(__ldg(reinterpret_cast<const uint16_t*>(src + kQ4KS) + r));
  const float M = bf16_bits_to_f32(__ldg(reinterpret_cast<const uint16_t*>(src + kQ4KM) + r));
  const float sc = static_cast<float>(__ldg(src + kQ4KSc + i));
  const float mn = static_cast<float>(__ldg(src + kQ4KMn + i));
  reinterpret_cast<uint16_t*>(dst + kQ41Scale)[i] = f32_to_bf16_bits(__fmul_rn(S, sc));
  reinterpret_cast<uint16_t*>(dst + kQ41Zero)[i] = f32_to_bf16_bits(__fmul_rn(M, mn));
}

cudaError_t launch_repack_q4k(const void* in, int64_t TR, int64_t TC, void* out, cudaStream_t s) {
  const int64_t T = TR * TC;
  if (T > 0x7FFFFFFF) return cudaErrorInvalidValue;
  repack_q4k_kernel<<<static_cast<unsigned>(T), 256, 0, s>>>(static_cast<const uint8_t*>(in),
                                                              static_cast<uint8_t*>(out));
  return cudaGetLastError();
}

// --------------------------------------------------- GGUF-type -> q4_1 ----
//
// "NPU engine" page, section "From a GGUF", GGUF-type table: Q4_0 becomes
// scale d, zero -8d and Q4_1 scale d, zero m, codes unchanged (the only error
// is the bf16 rounding of scale and zero); Q8_0, F32, F16 and BF16 are
// dequantized, then quantized to a min/max q4_1 per 32 columns.  One CTA per
// chunk, one thread per (row, 32-column group).  Source: row-major blocks of 32
// columns (Q4_0: fp16 d + 16 code bytes, element i < 16 in the low nibble of
// byte i and i >= 16 in the high nibble of byte i - 16; Q4_1: fp16 d, fp16 m +
// the same 16 bytes; Q8_0: fp16 d + 32 int8), or N*K dense values.  Min/max
// of 32 values x: lo, hi (first of equal minima / maxima); s = bf16((hi - lo)
// / 15), z = bf16(lo); code = clamp(rint((x - z) / s), 0, 15) with the stored
// s, z, ties to even, every code 0 if s == 0 -- each step one IEEE binary32
// operation, so the codes are the same on every machine.

__device__ __forceinline__ uint32_t ld_u16_global(const uint8_t* p) {
  return *reinterpret_cast<const uint16_t*>(p);                   // 2-byte aligned by construction
}

template <int SRC>
__global__ void __launch_bounds__(256) pack_q4_1_kernel(const uint8_t* __restrict__ src, int64_t K, int64_t TC,
                                                        uint8_t* __restrict__ out) {
  const int64_t t = blockIdx.x;
  const int64_t tr = t / TC, tc = t - tr * TC;
  const int r = threadIdx.x >> 3, g = threadIdx.x & 7;
  const int64_t n = tr * 32 + r;                   // tensor row
  const int64_t blk = n * (K / 32) + tc * 8 + g;   // 32-column block of that row
  int q[32];
  uint16_t s_bits, z_bits;
  if constexpr (SRC == kSrcQ4_0 || SRC == kSrcQ4_1) {
    constexpr int BS = SRC == kSrcQ4_0 ? 18 : 20;
    const uint8_t* b = src + blk * BS;
    const float d = __half2float(__ushort_as_half(static_cast<unsigned short>(ld_u16_global(b))));
    const uint8_t* qs = b + (SRC == kSrcQ4_0 ? 2 : 4);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t h = ld_u16_global(qs + 2 * j);   // bytes 2j, 2j+1
      q[2 * j] = h & 15;
      q[2 * j + 1] = (h >> 8) & 15;
      q[16 + 2 * j] = (h >> 4) & 15;
      q[16 + 2 * j + 1] = (h >> 12) & 15;
    }
    s_bits = f32_to_bf16_bits(d);
    if constexpr (SRC == kSrcQ4_0) {
      z_bits = f32_to_bf16_bits(__fmul_rn(-8.0f, d));                 // exact product
    } else {
      z_bits = f32_to_bf16_bits(__half2float(__ushort_as_half(static_cast<unsigned short>(ld_u16_global(b + 2)))));
    }
  } else {
    float x[32];
    if constexpr (SRC == kSrcQ8_0) {
      const uint8_t* b = src + blk * 34;
      const float d = __half2float(__ushort_as_half(static_cast<unsigned short>(ld_u16_global(b))));
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const uint32_t h = ld_u16_global(b + 2 + 2 * j);
        x[2 * j] = __fmul_rn(static_cast<float>(static_cast<int8_t>(h & 0xFF)), d);     // exact
        x[2 * j + 1] = __fmul_rn(static_cast<float>(static_cast<int8_t>(h >> 8)), d);
      }
    } else if constexpr (SRC == kSrcF32) {
      const uint4* v = reinterpret_cast<const uint4*>(src + blk * 128);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint4 u = v[j];
        x[4 * j] = __uint_as_float(u.x);
        x[4 * j + 1] = __uint_as_float(u.y);
        x[4 * j + 2] = __uint_as_float(u.z);
        x[4 * j + 3] = __uint_as_float(u.w);
      }
    } else {                                      // F16 or BF16: 32 values of 2 bytes
      const uint4* v = reinterpret_cast<const uint4*>(src + blk * 64);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint4 u = v[j];
        const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const uint32_t h = hh ? (w4[e] >> 16) : (w4[e] & 0xFFFF);
            x[8 * j + 2 * e + hh] = SRC == kSrcF16 ? __half2float(__ushort_as_half(static_cast<unsigned short>(h)))
                                                  : bf16_bits_to_f32(h);
          }
        }
      }
    }
    float lo = x[0], hi = x[0];
#pragma unroll
    for (int i = 1; i < 32; ++i) {
      if (x[i] < lo) lo = x[i];
      if (x[i] > hi) hi = x[i];
    }
    s_bits = f32_to_bf16_bits(__fdiv_rn(__fsub_rn(hi, lo), 15.0f));
    z_bits = f32_to_bf16_bits(lo);
    const float sv = bf16_bits_to_f32(s_bits), zv = bf16_bits_to_f32(z_bits);
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      if (sv == 0.0f) { q[i] = 0; continue; }
      const float c = rintf(__fdiv_rn(__fsub_rn(x[i], zv), sv));      // nearest, ties to even
      q[i] = c < 0.0f ? 0 : (c > 15.0f ? 15 : static_cast<int>(c));
    }
  }
  uint8_t* ch = out + t * kQ41Bytes;
  uint32_t w[4];
#pragma unroll
  for (int j = 0; j < 4; ++j)
    w[j] = static_cast<uint32_t>(q[8 * j] | (q[8 * j + 1] << 4) | (q[8 * j + 2] << 8) | (q[8 * j + 3] << 12) |
                                 (q[8 * j + 4] << 16) | (q[8 * j + 5] << 20) | (q[8 * j + 6] << 24) |
                                 (q[8 * j + 7] << 28));
  *reinterpret_cast<uint4*>(ch + r * 128 + g * 16) = make_uint4(w[0], w[1], w[2], w[3]);
  reinterpret_cast<uint16_t*>(ch + kQ41Scale)[r * 8 + g] = s_bits;
  reinterpret_cast<uint16_t*>(ch + kQ41Zero)[r * 8 + g] = z_bits;
}

int pack_src_bytes_per_32(int src_type) {
  switch (src_type) {
    case kSrcQ4_0: return 18;
    case kSrcQ4_1: return 20;
    case kSrcQ8_0: return 34;
    case kSrcF32: return 128;
    case kSrcF16:
    case kSrcBF16: return 64;
    default: return 0;
  }
}

cudaError_t launch_pack_q4_1(int src_type, const void* src, int64_t TR, int64_t TC, void* out, cudaStream_t s) {
  const int64_t T = TR * TC;
  if (T > 0x7FFFFFFF) return cudaErrorInvalidValue;
  const uint8_t* in = static_cast<const uint8_t*>(src);
  uint8_t* o = static_cast<uint8_t*>(out);
  const unsigned grid = static_cast<unsigned>(T);
  const int64_t K = TC * 256;
  switch (src_type) {
    case kSrcQ4_0: pack_q4_1_kernel<kSrcQ4_0><<<grid, 256, 0, s>>>(in, K, TC, o); break;
    case kSrcQ4_1: pack_q4_1_kernel<kSrcQ4_1><<<grid, 256, 0, s>>>(in, K, TC, o); break;
    case kSrcQ8_0: pack_q4_1_kernel<kSrcQ8_0><<<grid, 256, 0, s>>>(in, K, TC, o); break;
    case kSrcF32: pack_q4_1_kernel<kSrcF32><<<grid, 256, 0, s>>>(in, K, TC, o); break;
    case kSrcF16: pack_q4_1_kernel<kSrcF16><<<grid, 256, 0, s>>>(in, K, TC, o); break;
    case kSrcBF16: pack_q4_1_kernel<kSrcBF16><<<grid, 256, 0, s>>>(in, K, TC, o); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

// ------------------------------------------------------------- argmax ----
//
// Each (value, index) becomes a 64-bit key whose unsigned order is the
// wanted order: NaN above +inf above every number, +0 == -0, and for equal
// values the lower index above.  A cluster of 8 CTAs reduces one row: each
// CTA scans an eighth, then CTA 0 reads the others' maxima through
// distributed shared memory.  No workspace, no atomics, deterministic.
constexpr int kArgmaxCluster = 8;
constexpr int kArgmaxThreads = 512;


// BATCH: 16-byte loads a thread has in flight before it uses any.  Few rows
// (CTAs <= SMs): 12, so that a CTA's eighth of a ~150K-logit row is one round
// trip; many rows: 4, with the registers of four CTAs per SM.
template <int BATCH>
__global__ void __cluster_dims__(kArgmaxCluster, 1, 1) __launch_bounds__(kArgmaxThreads, BATCH > 4 ? 1 : 4)
    argmax_kernel(const float* __restrict__ logits, int64_t V, int32_t* __restrict__ idx) {
  __shared__ uint64_t warp_best[kArgmaxThreads / 32];
  __shared__ uint64_t cta_best;
  cg::cluster_group cluster = cg::this_cluster();
  const unsigned rank = cluster.block_rank();
  // No early trigger for the next grid: a GEMV launched behind this one would
  // start on every SM but the cluster's 8, and its CTAs there would start
  // late and finish late (lm_head q4_1 GEMV then argmax, back to back:
  // 45.8 us without the trigger, 60.5 us with it).
  asm volatile("griddepcontrol.wait;" ::: "memory");     // the logits may be the previous grid's output
  const int64_t m = blockIdx.y;
  const float* row = logits + m * V;
  const int64_t per = (V + kArgmaxCluster - 1) / kArgmaxCluster;
  const int64_t b0 = rank * per;
  const int64_t b1 = (b0 + per < V) ? b0 + per : V;
  uint64_t best = 0;
  const bool vec = ((reinterpret_cast<uintptr_t>(row) & 15) == 0) && ((b0 & 3) == 0);
  if (vec && b1 > b0) {
    const int64_t n4 = (b1 - b0) / 4;
    const float4* r4 = reinterpret_cast<const float4*>(row + b0);
    // every load of a batch is in flight before any is used: the scan is
    // latency-bound
    for (int64_t i = threadIdx.x; i < n4; i += BATCH * kArgmaxThreads) {
      float4 v[BATCH];
#pragma unroll
      for (int u = 0; u < BATCH; ++u)
        if (i + u * kArgmaxThreads < n4) v[u] = __ldg(r4 + i + u * kArgmaxThreads);
#pragma unroll
      for (int u = 0; u < BATCH; ++u) {
        if (i + u * kArgmaxThreads >= n4) break;
        const uint32_t k = static_cast<uint32_t>(b0 + 4 * (i + u * kArgmaxThreads));
        best = umax64(best, argmax_key(v[u].x, k));
        best = umax64(best, argmax_key(v[u].y, k + 1));
        best = umax64(best, argmax_key(v[u].z, k + 2));
        best = umax64(best, argmax_key(v[u].w, k + 3));
      }
    }
    for (int64_t i = b0 + 4 * n4 + threadIdx.x; i < b1; i += blockDim.x)
      best = umax64(best, argmax_key(__ldg(row + i), static_cast<uint32_t>(i)));
  } else {
    for (int64_t i = b0 + threadIdx.x; i < b1; i += blockDim.x)
      best = umax64(best, argmax_key(__ldg(row + i), static_cast<uint32_t>(i)));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) best = umax64(best, __shfl_xor_sync(0xffffffffu, best, o));
  if ((threadIdx.x & 31) == 0) warp_best[threadIdx.x >> 5] = best;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint64_t b = 0;
    for (int w = 0; w < kArgmaxThreads / 32; ++w) b = umax64(b, warp_best[w]);
    cta_best = b;
  }
  cluster.sync();
  if (rank == 0 && threadIdx.x == 0) {
    uint64_t b = 0;
    for (unsigned r = 0; r < kArgmaxCluster; ++r) b = umax64(b, *cluster.map_shared_rank(&cta_best, r));
    idx[m] = argmax_index(b);
  }
  cluster.sync();      // peers keep their shared memory until rank 0 has read it
}

cudaError_t launch_argmax(const float* logits, int M, int64_t V, int32_t* idx, cudaStream_t s) {
  // programmatic dependent launch: the CTAs start while the grid that writes
  // the logits drains, and wait for it before the first load; the next grid
  // starts when this one has finished
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kArgmaxCluster, static_cast<unsigned>(M));
  cfg.blockDim = dim3(kArgmaxThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  if (static_cast<int64_t>(M) * kArgmaxCluster <= sms) return cudaLaunchKernelEx(&cfg, argmax_kernel<12>, logits, V, idx);
  return cudaLaunchKernelEx(&cfg, argmax_kernel<4>, logits, V, idx);
}

}  // namespace q4nx
