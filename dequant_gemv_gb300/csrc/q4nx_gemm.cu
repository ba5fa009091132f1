// q4nx_gemm.cu -- fused decode + GEMM for a block of up to 64 tokens on the
// 5th-generation tensor cores (tcgen05, TMEM accumulators, TMA), sm_103a.
//
//   Y[m][n] = sum_k X[m][k] * w[n][k],   w in q4_1 chunks ("Q4NX chunks"
//   section of the 1bit engine "NPU engine" page: code*scale + zero).
//
// Tile: 128 weight rows (4 tile rows of the chunk grid) x 64 tokens; k-steps
// of 256 columns (one chunk column).  The weight rows are the MMA's M side and
// the tokens its N side, so one tcgen05.mma (M=128, N=64, K=16, bf16 x bf16 ->
// fp32 in TMEM) covers the whole token block.
//
// Warp roles (23 warps):
//   warp 0       weight producer: per k-step the 4 chunks' code regions (3-D
//                tensor copy, 128-byte swizzle) and scale/zero regions (1-D
//                bulk copies) into one of 4 weight stages;
//   warp 1       X producer: the 64 x 256 bf16 X slice of the k-step (4 boxes of
//                64 x 64, 128-byte swizzle) into one of 2 X stages;
//   warp 2       TMEM allocator and MMA issuer (one thread);
//   warps 3-18   dequant: warp d decodes tile row d%4, columns 64(d/4)..+63 of
//                the step, one thread per weight row, into A stage d/4 (bf16,
//                canonical K-major 128-byte-swizzled layout, 128 x 64);
//   warps 19-22  epilogue: TMEM -> registers -> Y, or a split-K partial.
// Two accumulators in TMEM (2 x 64 columns) let the epilogue of one tile
// overlap the main loop of the next.  Work is spread stream-K style: every CTA
// owns a contiguous range of (tile, k-step) units; a tile split between CTAs
// is finished by the last CTA to arrive, which adds the fp32 partials in CTA
// order (deterministic).  Every wait is bounded; if one gives up, the CTA sets
// a shared abort flag, records the error in the workspace and winds down.
#include <cuda.h>

#include "q4nx_device.cuh"
#include "q4nx_kernels.h"

namespace q4nx {
namespace gemm {

constexpr int kTileM = 128, kTileN = 64, kStepK = 256;
constexpr int kWStages = 4, kXStages = 2, kAStages = 4, kAccs = 2;
constexpr int kCodes = 4096, kScales = 1024;
constexpr int kWBytes = 4 * kCodes + 4 * kScales;     // 20 KB: codes (1024-aligned) then scales
constexpr int kXBox = 64 * 128;                        // 64 tokens x 64 k of bf16
constexpr int kXBytes = 4 * kXBox;                     // 32 KB
constexpr int kABytes = 128 * 128;                     // 128 rows x 64 k of bf16
constexpr int kWOff = 0;
constexpr int kXOff = kWOff + kWStages * kWBytes;
constexpr int kAOff = kXOff + kXStages * kXBytes;
constexpr int kBarOff = kAOff + kAStages * kABytes;
constexpr int kSmemBytes = kBarOff + 256 + 1024;       // barriers and flags, alignment slack
constexpr int kDequantWarps = 16;
constexpr int kWarpW = 0, kWarpX = 1, kWarpMma = 2, kWarpDequant0 = 3, kWarpEpi0 = kWarpDequant0 + kDequantWarps;
constexpr int kWarps = kWarpEpi0 + 4;
constexpr int kThreads = kWarps * 32;
static_assert(kWStages * kWBytes % 1024 == 0 && kXBytes % 1024 == 0, "swizzled regions must stay 1024-aligned");

// tcgen05 instruction descriptor: D fp32, A bf16, B bf16, both K-major, N = 64, M = 128
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((kTileN >> 3) << 17) | ((kTileM >> 4) << 24);

struct Args {
  const uint8_t* chunks;
  void* Y;
  uint32_t* err;
  uint32_t* counters;       // [tiles]
  float* partials;          // [grid][2][64 tok][128 rows]
  int64_t TR, TC, N;
  int tiles, M, out_f32, grid;
  int64_t units;            // tiles * TC
};

// --------------------------------------------------------------- PTX ----

__device__ __forceinline__ void tma_3d(void* dst, const CUtensorMap* map, int c0, int c1, int c2, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];"
      ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void tma_2d(void* dst, const CUtensorMap* map, int c0, int c1, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  // K-major, 128-byte swizzle: rows of 128 B, 8-row groups 1024 B apart.
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFF);
  d |= static_cast<uint64_t>(1) << 16;                 // leading byte offset (unused for this layout)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;         // stride byte offset: next 8-row group
  d |= static_cast<uint64_t>(1) << 46;                 // descriptor version for tcgen05
  d |= static_cast<uint64_t>(2) << 61;                 // swizzle 128B
  return d;
}
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(kIdesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}
__device__ __forceinline__ uint32_t lds_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ void named_bar(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

struct Shared {
  uint64_t w_full[kWStages], w_empty[kWStages];
  uint64_t x_full[kXStages], x_empty[kXStages];
  uint64_t a_full[kAStages], a_empty[kAStages];
  uint64_t acc_full[kAccs], acc_empty[kAccs];
  uint64_t drain;
  uint32_t tmem_base;
  volatile uint32_t abort_flag;
  uint32_t last_flag;
};
static_assert(sizeof(Shared) <= 256, "barrier block");

// Bounded wait that also gives up at once when another warp has aborted.
__device__ __forceinline__ bool wait_bar(Shared* sh, uint64_t* bar, uint32_t parity, uint32_t* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (sh->abort_flag) return false;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      sh->abort_flag = 1u;
      atomicOr(err, 1u);
      return false;
    }
  }
}

// One 32-token slice of an output row: Y[m][n] for m in [m0, m0 + 32), m < M.
__device__ __forceinline__ void store_slice(const Args& a, int64_t n, int m0, const float (&v)[32]) {
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const int m = m0 + i;
    if (m < a.M) {
      if (a.out_f32) static_cast<float*>(a.Y)[m * a.N + n] = v[i];
      else static_cast<uint16_t*>(a.Y)[m * a.N + n] = f32_to_bf16_bits(v[i]);
    }
  }
}

// Decode columns [64 qq, 64 qq + 64) of weight row r of one tile row (its
// 128-byte-swizzled code region and its scale/zero region) into row rowA of
// an A stage (128 x 64 bf16, K-major, 128-byte swizzle).
__device__ __forceinline__ void dequant_quarter(uint32_t codes, uint32_t scales, int r, int qq, uint32_t abase,
                                                int rowA) {
  // scales and zeros of groups 2qq, 2qq+1: one bf16 pair each
  const uint32_t sw = lds_u32(scales + r * 16 + qq * 4);
  const uint32_t zw = lds_u32(scales + 512 + r * 16 + qq * 4);
#pragma unroll
  for (int gg = 0; gg < 2; ++gg) {
    const int g = 2 * qq + gg;
    const float s = __uint_as_float(gg ? (sw & 0xFFFF0000u) : (sw << 16));
    const float z = __uint_as_float(gg ? (zw & 0xFFFF0000u) : (zw << 16));
    // w = (1 + c 2^-8)(256 s) + (z - 256 s) for even k, (1 + c 2^-4)(16 s) + (z - 16 s) for odd k
    const float2 s2 = make_float2(s * 256.f, s * 16.f);
    const float2 z2 = make_float2(z - s2.x, z - s2.y);
    const uint4 cw = lds128(codes + r * 128 + ((g ^ (r & 7)) << 4));
    const uint32_t words[4] = {cw.x, cw.y, cw.z, cw.w};
    const uint32_t ONE = 0x3F800000u;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const uint32_t w = words[t];
      const uint32_t a15 = w << 15, a7 = w << 7, b1 = w >> 1, b9 = w >> 9;
      const float2 v0 = make_float2(__uint_as_float(lop3_and_or(a15, 0x00078000u, ONE)),
                                    __uint_as_float(lop3_and_or(a15, 0x00780000u, ONE)));
      const float2 v1 = make_float2(__uint_as_float(lop3_and_or(a7, 0x00078000u, ONE)),
                                    __uint_as_float(lop3_and_or(a7, 0x00780000u, ONE)));
      const float2 v2 = make_float2(__uint_as_float(lop3_and_or(b1, 0x00078000u, ONE)),
                                    __uint_as_float(lop3_and_or(b1, 0x00780000u, ONE)));
      const float2 v3 = make_float2(__uint_as_float(lop3_and_or(b9, 0x00078000u, ONE)),
                                    __uint_as_float(lop3_and_or(b9, 0x00780000u, ONE)));
      const float2 w0 = ffma2(v0, s2, z2), w1 = ffma2(v1, s2, z2);
      const float2 w2 = ffma2(v2, s2, z2), w3 = ffma2(v3, s2, z2);
      // k within the stage = 32 gg + 8 t: 16-byte unit (4 gg + t) of the 128-byte row
      const int unit = 4 * gg + t;
      sts128(abase + rowA * 128 + ((unit ^ (rowA & 7)) << 4), pack_bf16x2(w0.x, w0.y), pack_bf16x2(w1.x, w1.y),
             pack_bf16x2(w2.x, w2.y), pack_bf16x2(w3.x, w3.y));
    }
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    gemm_q41_kernel(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap xmap,
                    const __grid_constant__ Args a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Shared* sh = reinterpret_cast<Shared*>(smem + kBarOff);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t lo = a.units * blockIdx.x / a.grid, hi = a.units * (blockIdx.x + 1) / a.grid;
  const int n = static_cast<int>(hi - lo);
  const int64_t KS = a.TC;
  const int64_t first_tile = lo / KS, last_tile = (hi - 1) / KS;
  const int ntiles = static_cast<int>(last_tile - first_tile + 1);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kWStages; ++s) { mbar_init(&sh->w_full[s], 1); mbar_init(&sh->w_empty[s], kDequantWarps); }
    for (int s = 0; s < kXStages; ++s) { mbar_init(&sh->x_full[s], 1); mbar_init(&sh->x_empty[s], 1); }
    for (int s = 0; s < kAStages; ++s) { mbar_init(&sh->a_full[s], 4); mbar_init(&sh->a_empty[s], 1); }
    for (int s = 0; s < kAccs; ++s) { mbar_init(&sh->acc_full[s], 1); mbar_init(&sh->acc_empty[s], 4); }
    mbar_init(&sh->drain, 1);
    sh->abort_flag = 0u;
    fence_barrier_init();
  }
  if (warp == kWarpMma) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&sh->tmem_base)),
                 "r"(kAccs * kTileN)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh->tmem_base;

  if (warp == kWarpW) {
    // ----------------------------------------------------------- weights
    if (lane == 0) {
      int64_t tile = lo / KS, ks = lo - tile * KS;
      int j = 0;
      for (; j < n; ++j) {
        const int s = j % kWStages;
        if (!wait_bar(sh, &sh->w_empty[s], ((j / kWStages) & 1) ^ 1u, a.err)) break;
        uint8_t* st = smem + kWOff + s * kWBytes;
        const int64_t left = a.TR - tile * 4;
        const int rows = left < 4 ? static_cast<int>(left) : 4;
        mbar_arrive_expect_tx(&sh->w_full[s], rows * (kCodes + kScales));
        for (int i = 0; i < rows; ++i) {
          const int64_t chunk = (tile * 4 + i) * a.TC + ks;
          tma_3d(st + i * kCodes, &wmap, 0, 0, static_cast<int>(chunk), &sh->w_full[s]);
          bulk_g2s(st + 4 * kCodes + i * kScales, a.chunks + chunk * kQ41Bytes + kQ41Scale, kScales, &sh->w_full[s]);
        }
        if (++ks == KS) { ks = 0; ++tile; }
      }
      for (int t = (j > kWStages ? j - kWStages : 0); t < j; ++t)      // copies still in flight land first
        mbar_wait_bounded(&sh->w_full[t % kWStages], (t / kWStages) & 1, 100000000ull);
    }
  } else if (warp == kWarpX) {
    // ----------------------------------------------------------- X
    if (lane == 0) {
      int64_t ks = lo % KS;
      int j = 0;
      for (; j < n; ++j) {
        const int s = j % kXStages;
        if (!wait_bar(sh, &sh->x_empty[s], ((j / kXStages) & 1) ^ 1u, a.err)) break;
        uint8_t* st = smem + kXOff + s * kXBytes;
        mbar_arrive_expect_tx(&sh->x_full[s], kXBytes);
        for (int b = 0; b < 4; ++b)
          tma_2d(st + b * kXBox, &xmap, static_cast<int>(ks * kStepK + b * 64), 0, &sh->x_full[s]);
        if (++ks == KS) ks = 0;
      }
      for (int t = (j > kXStages ? j - kXStages : 0); t < j; ++t)
        mbar_wait_bounded(&sh->x_full[t % kXStages], (t / kXStages) & 1, 100000000ull);
    }
  } else if (warp == kWarpMma) {
    // ----------------------------------------------------------- MMA issuer
    if (lane == 0) {
      int64_t ks = lo % KS;
      int tcount = 0;
      bool first_in_tile = true;
      for (int j = 0; j < n; ++j) {
        const int b = tcount % kAccs;
        if (first_in_tile) {
          if (!wait_bar(sh, &sh->acc_empty[b], ((tcount / kAccs) & 1) ^ 1u, a.err)) break;
          tc_fence_after();
        }
        const int xs = j % kXStages;
        if (!wait_bar(sh, &sh->x_full[xs], (j / kXStages) & 1, a.err)) break;
        const uint32_t xbase = smem_u32(smem + kXOff + xs * kXBytes);
        bool ok = true;
        for (int q = 0; q < kAStages; ++q) {
          if (!wait_bar(sh, &sh->a_full[q], j & 1, a.err)) { ok = false; break; }
          tc_fence_after();
          const uint32_t abase = smem_u32(smem + kAOff + q * kABytes);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t ad = sw128_desc(abase + kk * 32);
            const uint64_t bd = sw128_desc(xbase + q * kXBox + kk * 32);
            mma_bf16(tmem + b * kTileN, ad, bd, (first_in_tile && q == 0 && kk == 0) ? 0u : 1u);
          }
          mma_commit(&sh->a_empty[q]);
        }
        if (!ok) break;
        mma_commit(&sh->x_empty[xs]);
        first_in_tile = false;
        if (++ks == KS || j == n - 1) {             // this CTA's share of the tile is complete
          mma_commit(&sh->acc_full[b]);
          ++tcount;
          first_in_tile = true;
          if (ks == KS) ks = 0;
        }
      }
      mma_commit(&sh->drain);                       // every MMA issued so far has completed
      mbar_wait_bounded(&sh->drain, 0, 100000000ull);
    }
  } else if (warp < kWarpEpi0) {
    // ----------------------------------------------------------- dequant
    const int d = warp - kWarpDequant0;
    const int i = d & 3, qq = d >> 2;
    const int rowA = 32 * i + lane;
    const uint32_t abase = smem_u32(smem + kAOff + qq * kABytes);
    int64_t tile = lo / KS, ks = lo - tile * KS;
    for (int j = 0; j < n; ++j) {
      const int s = j % kWStages;
      if (!wait_bar(sh, &sh->w_full[s], (j / kWStages) & 1, a.err)) break;
      if (!wait_bar(sh, &sh->a_empty[qq], (j & 1) ^ 1u, a.err)) break;
      if (tile * 4 + i < a.TR) {
        const uint32_t st = smem_u32(smem + kWOff + s * kWBytes);
        dequant_quarter(st + i * kCodes, st + 4 * kCodes + i * kScales, lane, qq, abase, rowA);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&sh->a_full[qq]);
        mbar_arrive(&sh->w_empty[s]);
      }
      if (++ks == KS) { ks = 0; ++tile; }
    }
  } else {
    // ----------------------------------------------------------- epilogue
    const int e = warp & 3;                         // TMEM lane quarter of this warp
    const int row = 32 * e + lane;                  // row within the 128-row tile
    for (int t = 0; t < ntiles; ++t) {
      const int b = t % kAccs;
      if (!wait_bar(sh, &sh->acc_full[b], (t / kAccs) & 1, a.err)) break;
      tc_fence_after();
      const int64_t tile = first_tile + t;
      const int64_t u_lo = tile * KS, u_hi = u_lo + KS;
      const int64_t n0 = tile * kTileM;
      const bool valid_row = n0 + row < a.N;
      const bool whole = lo <= u_lo && u_hi <= hi;   // the whole tile was computed here
      const int slot = (lo >= u_lo) ? 0 : 1;          // split tile: this CTA's partial slot
      float* mine = a.partials + (static_cast<int64_t>(blockIdx.x) * 2 + slot) * (kTileN * kTileM) + row;
      const uint32_t taddr = tmem + (static_cast<uint32_t>(32 * e) << 16) + b * kTileN;
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {
        float v[32];
        tmem_ld32(taddr + 32 * h, v);
        if (whole) {
          if (valid_row) store_slice(a, n0 + row, 32 * h, v);
        } else {
#pragma unroll
          for (int m = 0; m < 32; ++m) mine[(32 * h + m) * kTileM] = v[m];
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh->acc_empty[b]);
      if (whole) continue;
      // split tile: the last CTA to arrive adds the partials (in CTA order) and stores the tile
      __threadfence();
      named_bar(1, 128);
      const int64_t c_first = ((u_lo + 1) * a.grid - 1) / a.units;
      const int64_t c_last = (u_hi * a.grid - 1) / a.units;
      if (threadIdx.x == kWarpEpi0 * 32) {
        const uint32_t old = atomicAdd(&a.counters[tile], 1u);
        sh->last_flag = (old == static_cast<uint32_t>(c_last - c_first)) ? 1u : 0u;
      }
      named_bar(1, 128);
      const bool last = sh->last_flag != 0u;
      named_bar(1, 128);                            // every thread has read the flag before it is reused
      if (!last) continue;
      __threadfence();
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {
        float v[32];
#pragma unroll
        for (int m = 0; m < 32; ++m) v[m] = 0.f;
        for (int64_t c = c_first; c <= c_last; ++c) {
          const int64_t clo = a.units * c / a.grid;
          float* p = a.partials + (c * 2 + ((clo >= u_lo) ? 0 : 1)) * (kTileN * kTileM) + row + 32 * h * kTileM;
#pragma unroll
          for (int m = 0; m < 32; ++m) v[m] += ld_cg_f32(p + m * kTileM);
#pragma unroll
          for (int m = 0; m < 32; ++m) p[m * kTileM] = 0.f;    // leave the workspace zero-filled
        }
        if (valid_row) store_slice(a, n0 + row, 32 * h, v);
      }
      if (threadIdx.x == kWarpEpi0 * 32) a.counters[tile] = 0u;
    }
  }

  __syncwarp();                                     // whole warps arrive at the CTA barrier
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kAccs * kTileN) : "memory");
  }
}

}  // namespace gemm

// ----------------------------------------------------------------- host ----

namespace {
using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiled encode_fn() {
  static EncodeTiled fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiled>(p);
  }
  return fn;
}
}  // namespace

bool gemm_supports(int kind) { return kind == kQ4_1; }

uint64_t gemm_workspace_bytes(int64_t TR, int64_t TC, int M) {
  (void)TC;
  (void)M;
  const int64_t tiles = (TR + 3) / 4;
  // error word, arrival counters, partial tiles of at most 1024 CTAs
  return kWsErrBytes + align16(static_cast<uint64_t>(tiles) * 4) +
         static_cast<uint64_t>(1024) * 2 * gemm::kTileN * gemm::kTileM * 4;
}

cudaError_t launch_gemm(int kind, const void* chunks, int64_t TR, int64_t TC, const void* X, int M, void* Y,
                        int out_f32, void* workspace, cudaStream_t s) {
  if (kind != kQ4_1) return cudaErrorNotSupported;
  EncodeTiled enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  DeviceInfo info;
  cudaError_t e = device_info(&info);
  if (e != cudaSuccess) return e;
  if (info.max_smem_optin < gemm::kSmemBytes) return cudaErrorNotSupported;

  CUtensorMap wmap, xmap;
  const int64_t T = TR * TC;
  {
    cuuint64_t dims[3] = {128, 32, static_cast<cuuint64_t>(T)};
    cuuint64_t strides[2] = {128, kQ41Bytes};
    cuuint32_t box[3] = {128, 32, 1};
    cuuint32_t es[3] = {1, 1, 1};
    if (enc(&wmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(chunks), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(TC * 256), static_cast<cuuint64_t>(M)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(TC * 256 * 2)};
    cuuint32_t box[2] = {64, 64};
    cuuint32_t es[2] = {1, 1};
    if (enc(&xmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(X), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  gemm::Args a;
  const int64_t tiles = (TR + 3) / 4;
  a.chunks = static_cast<const uint8_t*>(chunks);
  a.Y = Y;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  a.err = reinterpret_cast<uint32_t*>(ws);
  a.counters = reinterpret_cast<uint32_t*>(ws + kWsErrBytes);
  a.partials = reinterpret_cast<float*>(ws + kWsErrBytes + align16(static_cast<uint64_t>(tiles) * 4));
  a.TR = TR;
  a.TC = TC;
  a.N = TR * 32;
  a.tiles = static_cast<int>(tiles);
  a.M = M;
  a.out_f32 = out_f32;
  a.units = tiles * TC;
  int64_t grid = info.sms < 1024 ? info.sms : 1024;
  if (grid > a.units) grid = a.units;
  a.grid = static_cast<int>(grid);
  e = set_max_dynamic_smem(reinterpret_cast<const void*>(gemm::gemm_q41_kernel), 16);
  if (e != cudaSuccess) return e;
  gemm::gemm_q41_kernel<<<a.grid, gemm::kThreads, gemm::kSmemBytes, s>>>(wmap, xmap, a);
  return cudaGetLastError();
}

}  // namespace q4nx
