// q4nx_gemm.cu -- fused decode + GEMM for a block of up to 64 tokens on the
// 5th-generation tensor cores (tcgen05, TMEM, TMA), sm_103a.
//
//   Y[m][n] = sum_k X[m][k] * w[n][k],   w in q4_1 chunks (code*scale + zero)
//   or Q8 chunks in either code layout (d*code); "Q4NX chunks" section of the
//   1bit engine "NPU engine" page.
//
// Tile: 128 weight rows (4 tile rows of the chunk grid) x 64 tokens; k-steps
// of 256 columns (one chunk column).  The weight rows are the MMA's M side and
// the tokens its N side: one tcgen05.mma (M=128, N=64, K=16, bf16 x bf16 ->
// fp32) covers the whole token block.
//
// Data path of one k-step:
//   4 chunks --TMA--> shared memory --ld.shared--> dequant warps
//        --tcgen05.st--> TMEM (A operand, bf16, 128 lanes x 128 columns)
//   X[0:64, k-step] --TMA, 128-byte swizzle--> shared memory (B operand)
//   tcgen05.mma reads A from TMEM and B from shared memory, accumulates in TMEM.
// A never touches shared memory: with N = 64, an MMA that read A from shared
// memory would spend two thirds of the SM's shared-memory bandwidth on A
// alone, and the TMA fills, the code reads and the B reads need that bandwidth.
//
// Warp roles (16 warps; a warp reaches TMEM lanes 32*(warp%4) .. +31 only):
//   warp 0       weight producer: per k-step the 4 chunks into one of the
//                weight stages.  q4_1: the code regions (one 4-D tensor copy,
//                128-byte swizzle, so that row-wise 16-byte reads are free of
//                bank conflicts) and the scale/zero regions (one 4-D tensor
//                copy); Q8: the 4 whole chunks (one 4-D tensor copy), whose
//                column-wise codes the dequant warps read a byte at a time;
//   warp 1       X producer: the tokens' 256-column bf16 slice of X (four 2-D
//                tensor copies of 64 columns x M tokens rounded up to 8) into
//                one of kStages stages;
// The producers, like the MMA warp, run their loops warp-wide and issue from
// one elected lane: a copy instruction issued from a single-lane branch costs
// far more issue slots, and these slots are shared with the dequant warps.
//   warp 2       MMA issuer: the whole warp runs the loop (its values stay
//                warp-uniform) and one elected lane issues each k-step's 16
//                MMAs and their commit as one block;
//   warp 3       TMEM allocator;
//   warps 4-11   dequant: warp w decodes tile row w%4 (the TMEM lanes of that
//                tile row), columns 128*((w-4)/4) .. +127 of every k-step, one
//                thread per weight row, into the A half of one of kStages
//                stages (the A half in TMEM, the X half in shared memory);
//   warps 12-15  epilogue: TMEM -> registers -> Y, or a split-tile partial.
// Eight dequant warps rather than sixteen: the MMA warp shares its
// sub-partition's issue slots with the dequant warps there, and fewer of them
// let it keep the tensor pipe fed.
// Two accumulators (2 x 64 TMEM columns) let the epilogue of one tile overlap
// the main loop of the next.  A stage is filled by 9 arrivals (the X
// producer's, with the TMA byte count, and the 8 dequant warps') and emptied
// by one MMA commit, so the MMA thread waits once and commits once per k-step:
// each wait or commit in that single issuing thread delays the tensor pipe.
//
// Work split (stream-K): the (tile, k-step) units are cut into one contiguous
// range per CTA (for shapes whose tiles allow it, into equal parts of every
// tile; see the launch).  A tile shared by several CTAs is finished by the CTA that
// holds its first k-step.  That CTA reaches the tile at the end of its range,
// while the others (which hold the tile's later k-steps at the start of their
// ranges) post their fp32 partials early; the finisher gathers them into its
// epilogue warps' registers while its own main loop still runs, then adds
// them to its accumulator.  The sum order depends only on the shape (the next
// CTA's partial, those beyond the shared-memory gather slots, the gathered
// ones, each group in CTA order, then the finisher's own), so results are
// deterministic.  Every wait is
// bounded; if one gives up, the CTA records the error in the workspace and
// winds down.
//
// A CTA's last output tile leaves through shared memory (the X stages are
// free once its last MMA has completed): the epilogue warps stage the tile
// there and one thread writes it to Y with a single TMA tensor store, instead
// of thousands of 64-byte stores.  Partials always go out from registers as
// 512-byte coalesced stores, each warp then counting itself in with a release
// reduction: the finisher waits on them, and this is the quickest way there.
//
// The finisher waits for CTAs of the same launch, so the launch relies on all
// of its CTAs being resident at once: the grid is at most one CTA per SM, and
// a CTA needs most of an SM's shared memory.
//
// Programmatic dependent launch: the kernel lets the next grid in the stream
// launch as soon as all of its CTAs are running, and starts its own weight
// copies before waiting for the previous grid; X, Y and the workspace are
// touched only after that wait.
#include <cuda.h>

#include "q4nx_device.cuh"
#include "q4nx_kernels.h"

namespace q4nx {
namespace gemm {

constexpr int kTileM = 128, kTileN = 64, kStepK = 256;
constexpr int kStages = 3, kAccs = 2;
constexpr int kCodes = 4096, kScales = 1024;            // q4_1 stage: codes (1024-aligned), then scales and zeros
constexpr int kXBox = 64 * 128;                        // 64 tokens x 64 k of bf16
constexpr int kXBytes = 4 * kXBox;                     // 32 KB
constexpr int kWOff = 0;
constexpr int kMaxWStages = 6;
// Shared-memory plan per chunk kind: weight stages, then X stages, then barriers.
template <int KIND>
struct Plan {
  static constexpr bool kQ8 = KIND == kQ8_KR || KIND == kQ8_BLK;
  static constexpr int kWBytes = kQ8 ? 4 * kQ8Bytes : 4 * kCodes + 4 * kScales;   // one k-step of 4 chunks
  static constexpr int kWStages = kQ8 ? 3 : 6;
  static constexpr int kXOff = kWOff + kWStages * kWBytes;
  static constexpr int kBarOff = kXOff + kStages * kXBytes;
  static constexpr int kSmemBytes = kBarOff + 512 + 1024;   // barriers and flags, alignment slack
  static_assert(kWStages <= kMaxWStages, "weight stages");
  static_assert(kWBytes % 1024 == 0 && kXOff % 1024 == 0 && kXBytes % 1024 == 0, "swizzled regions 1024-aligned");
  static_assert(kSmemBytes <= 232448, "shared memory per CTA");
};
// Slots of shared memory for the last tile's later partials (32 KB each), free
// once the CTA's last MMA has completed: three in the weight stages, two in X
// stages 1 and 2 (X stage 0 stages the output tile).
constexpr int kGatherSlots = 5;
template <int KIND>
__host__ __device__ constexpr int gather_slot(int i) {
  return i < 3 ? kWOff + i * kXBytes : Plan<KIND>::kXOff + (i - 2) * kXBytes;
}
static_assert(3 * kXBytes <= Plan<kQ4_1>::kWStages * Plan<kQ4_1>::kWBytes, "three partials fit the q4_1 weight stages");
static_assert(3 * kXBytes <= Plan<kQ8_KR>::kWStages * Plan<kQ8_KR>::kWBytes, "three partials fit the Q8 weight stages");
static_assert(kStages == 3, "X stages 1 and 2 take two partials");

constexpr int kDequantWarps = 8;                       // two per TMEM lane quarter, one half of the k-step each
constexpr int kWarpW = 0, kWarpX = 1, kWarpMma = 2, kWarpAlloc = 3, kWarpDequant0 = 4;
constexpr int kWarpEpi0 = kWarpDequant0 + kDequantWarps;
constexpr int kWarps = kWarpEpi0 + 4;
constexpr int kThreads = kWarps * 32;
// TMEM columns: accumulators [0, 128); A stages from 128, 128 columns each
// (4 quarters of 32 columns; a column holds 2 bf16 of one weight row).
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemA = kAccs * kTileN;
constexpr uint32_t kAStageCols = kStepK / 2;
static_assert(kTmemA + kStages * kAStageCols <= kTmemCols, "TMEM budget");
static_assert(kWarpDequant0 % 4 == 0 && kWarpEpi0 % 4 == 0, "TMEM lane quarters follow warp % 4");
static_assert(kDequantWarps == 8, "dequant warps: two per TMEM lane quarter");

// tcgen05 instruction descriptor: D fp32, A bf16, B bf16, both K-major, N = 64, M = 128
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((kTileN >> 3) << 17) | ((kTileM >> 4) << 24);

// Workspace bytes of the partial tiles: one per CTA, at most 1024 CTAs.
constexpr uint64_t kPartialBytes = static_cast<uint64_t>(1024) * kTileN * kTileM * 4;

struct Args {
  const uint8_t* chunks;
  void* Y;
  uint32_t* err;
  uint32_t* counters;       // [tiles]: epilogue warps of other CTAs that posted a partial of the tile
  float* partials;          // [grid][16 token quads][128 rows][4]: at most one partial per CTA
  int64_t TR, TC, N;
  int tiles, M, out_f32, grid;
  int mrows;                // X box rows: M rounded up to 8
  int64_t units;            // tiles * TC
};

// --------------------------------------------------------------- PTX ----

// One k-step of weights, on one elected lane of a converged warp: arm `bar`
// for kWBytes, then copy the code regions of chunks (4 tr4 + i, ks), i < 4,
// to dst + 4096 i and their scale/zero regions to dst + 16384 + 1024 i (tile
// rows past the end read as zeros and still count their bytes).
__device__ __forceinline__ void issue_weights(uint32_t dst, const CUtensorMap* cmap, const CUtensorMap* smap, int ks,
                                              int tr4, uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e mbarrier.arrive.expect_tx.shared::cta.b64 _, [%5], %6;\n\t"
      "@e cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%2, {0, 0, %3, %4}], [%5];\n\t"
      "@e cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%1], [%7, {0, 0, %3, %4}], [%5];\n\t}"
      ::"r"(dst), "r"(dst + 4 * 4096), "l"(reinterpret_cast<uint64_t>(cmap)), "r"(ks), "r"(tr4), "r"(bar),
      "n"(4 * 4096 + 4 * 1024), "l"(reinterpret_cast<uint64_t>(smap))
      : "memory");
}
// Q8: one k-step of weights, on one elected lane: arm `bar` for 4 chunks,
// then copy chunks (4 tr4 + i, ks), i < 4, whole to dst + 8704 i.
__device__ __forceinline__ void issue_weights_q8(uint32_t dst, const CUtensorMap* map, int ks, int tr4, uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e mbarrier.arrive.expect_tx.shared::cta.b64 _, [%3], %4;\n\t"
      "@e cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%5, {0, 0, %1, %2}], [%3];\n\t}"
      ::"r"(dst), "r"(ks), "r"(tr4), "r"(bar), "n"(4 * kQ8Bytes), "l"(reinterpret_cast<uint64_t>(map))
      : "memory");
}
// One k-step of X, on one elected lane: arm `bar` for the four boxes' bytes,
// then copy X[0:mrows, 256 ks .. +255] (128-byte swizzle) as four boxes of
// 64 columns x mrows tokens (M rounded up to 8,
// so that a box reaches at most 7 token rows past the end of X: boxes mostly
// outside the tensor are slow to fill), each into its 8 KB slot of the stage.
// Rows from mrows to 63 of a slot keep whatever they held: they only reach
// accumulator columns of tokens that are never stored.
__device__ __forceinline__ void issue_x(uint32_t dst, const CUtensorMap* xmap, int ks, uint32_t bar, int mrows) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t.reg .b32 x1, x2, x3;\n\telect.sync _|e, 0xffffffff;\n\t"
      "add.u32 x1, %2, 64;\n\tadd.u32 x2, %2, 128;\n\tadd.u32 x3, %2, 192;\n\t"
      "@e mbarrier.arrive.expect_tx.shared::cta.b64 _, [%3], %4;\n\t"
      "@e cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, 0}], [%3];\n\t"
      "@e cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0+8192], [%1, {x1, 0}], [%3];\n\t"
      "@e cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0+16384], [%1, {x2, 0}], [%3];\n\t"
      "@e cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0+24576], [%1, {x3, 0}], [%3];\n\t}"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(xmap)), "r"(256 * ks), "r"(bar), "r"(4 * 128 * mrows)
      : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
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
// One k-step on one elected lane of a converged warp: D[tmem] (+)= A[tmem] *
// B[smem]^T as 16 MMAs of M = 128, N = 64, K = 16 (MMA u = 4q + kk reads A
// columns a + 32q + 8kk and the X box q at byte 32kk), then a commit to `bar`.
// `accumulate` = 0 starts the accumulator afresh.  One asm block keeps the
// issue sequence short: every extra instruction in the issuing thread
// competes with the dequant warps for the same issue slots.
__device__ __forceinline__ void mma_kstep(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t accumulate,
                                          uint64_t* bar) {
  static_assert(kXBox == 8192, "X box offsets below");
  asm volatile(
      "{\n\t.reg .pred e, p, t;\n\t.reg .b32 ra;\n\t.reg .b64 rb;\n\t"
      "setp.ne.b32 p, %3, 0;\n\tsetp.eq.b32 t, 1, 1;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %5, p;\n\t"
#define Q4NX_MMA_U(AO, BO)                                 \
  "add.u32 ra, %1, " #AO ";\n\tadd.u64 rb, %2, " #BO ";\n\t" \
  "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ra], rb, %5, t;\n\t"
      Q4NX_MMA_U(8, 2) Q4NX_MMA_U(16, 4) Q4NX_MMA_U(24, 6)
      Q4NX_MMA_U(32, 512) Q4NX_MMA_U(40, 514) Q4NX_MMA_U(48, 516) Q4NX_MMA_U(56, 518)
      Q4NX_MMA_U(64, 1024) Q4NX_MMA_U(72, 1026) Q4NX_MMA_U(80, 1028) Q4NX_MMA_U(88, 1030)
      Q4NX_MMA_U(96, 1536) Q4NX_MMA_U(104, 1538) Q4NX_MMA_U(112, 1540) Q4NX_MMA_U(120, 1542)
#undef Q4NX_MMA_U
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%4];\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(accumulate), "r"(smem_u32(bar)), "n"(kIdesc)
      : "memory");
}
// Commit (arrive on `bar` when every MMA issued so far has completed), one elected lane.
__device__ __forceinline__ void mma_commit_elect(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(smem_u32(bar))
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
__device__ __forceinline__ void sts_u16(uint32_t addr, uint16_t v) {
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}
__device__ __forceinline__ void sts_f32(uint32_t addr, float v) {
  asm volatile("st.shared.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
// shared -> global copies issued by one thread; `wait_written` returns once the
// data is in global memory, `wait_read` once the shared source may be reused.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, int c0, int c1, uint32_t ssrc) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1), "r"(ssrc)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ uint32_t lds_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}
// bf16x2 a + b and a * b + c, each rounded once to nearest even
__device__ __forceinline__ uint32_t add_bf16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t fma_bf16x2(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

struct Shared {
  uint64_t w_full[kMaxWStages], w_empty[kMaxWStages];
  uint64_t full[kStages], empty[kStages];   // X (TMA bytes) + A (8 dequant warps) of a k-step
  uint64_t acc_full[kAccs], acc_empty[kAccs];
  uint64_t drain;
  uint64_t staged;          // epilogue warps that have staged their rows of the last tile
  uint64_t gather;          // the last tile's later partials, copied into free stage memory
  uint32_t tmem_base;
  volatile uint32_t abort_flag;
  uint32_t fix_seen;        // finisher's epilogue warps that have gathered every posted partial
};
static_assert(sizeof(Shared) <= 512, "barrier block");

// Bounded wait that also gives up at once when another warp has aborted.
__device__ __forceinline__ bool wait_bar(Shared* sh, uint64_t* bar, uint32_t parity, uint32_t* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait_sleep(bar, parity, 1000000u)) return true;
    if (sh->abort_flag) return false;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      sh->abort_flag = 1u;
      atomicOr(err, 1u);
      return false;
    }
  }
}

// wait_bar for a whole warp: true only if every lane's wait succeeded.
__device__ __forceinline__ bool wait_bar_warp(Shared* sh, uint64_t* bar, uint32_t parity, uint32_t* err) {
  return __all_sync(0xFFFFFFFFu, wait_bar(sh, bar, parity, err));
}

// Bounded wait (lane 0 polls, the warp follows) until `expect` partials of a
// tile have been posted; true when they have.
__device__ __forceinline__ bool wait_posted(Shared* sh, const uint32_t* counter, uint32_t expect, uint32_t* err,
                                            int lane) {
  uint32_t ok = 1u;
  if (lane == 0 && ld_acquire_u32(counter) != expect) {
    const uint64_t t0 = globaltimer_ns();
    while (ld_acquire_u32(counter) != expect) {
      if (sh->abort_flag || globaltimer_ns() - t0 > kWaitLimitNs) {
        sh->abort_flag = 1u;
        atomicOr(err, 1u);
        ok = 0u;
        break;
      }
    }
  }
  __syncwarp();                                     // orders the other lanes' loads after lane 0's acquire
  return __shfl_sync(0xFFFFFFFFu, ok, 0) != 0u;
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

// Columns [128 qh, 128 qh + 128) of weight row r of one tile row, as 64
// bf16x2 words in k order: w = code*scale + zero, rounded once to bf16 (the
// product code*scale is exact; the fused add rounds once).  The code region
// is 128-byte swizzled (16-byte unit u of row r at u ^ (r & 7)).  All shared
// memory loads come first, so their latency is paid once.
__device__ __forceinline__ void dequant_half(uint32_t codes, uint32_t scales, int r, int qh, uint32_t (&out)[64]) {
  const uint2 sw = lds64(scales + r * 16 + qh * 8);                // scales of groups 4qh .. 4qh+3
  const uint2 zw = lds64(scales + 512 + r * 16 + qh * 8);          // zeros of the same groups
  uint4 cw[4];
#pragma unroll
  for (int gg = 0; gg < 4; ++gg) cw[gg] = lds128(codes + r * 128 + (((4 * qh + gg) ^ (r & 7)) << 4));
  const uint32_t kMagic = 0x43004300u;        // bf16x2 (128, 128): 128 + c is exact for c < 128
  const uint32_t kMinus128 = 0xC300C300u;     // bf16x2 (-128, -128)
#pragma unroll
  for (int gg = 0; gg < 4; ++gg) {
    const uint32_t sp = gg < 2 ? sw.x : sw.y, zp = gg < 2 ? zw.x : zw.y;
    const uint32_t s2 = prmt(sp, 0, (gg & 1) ? 0x3232u : 0x1010u);  // (s, s) of group 4qh + gg
    const uint32_t z2 = prmt(zp, 0, (gg & 1) ? 0x3232u : 0x1010u);
    const uint32_t words[4] = {cw[gg].x, cw[gg].y, cw[gg].z, cw[gg].w};
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const uint32_t w = words[t];
      const uint32_t hi = w >> 4;
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        // byte b of w holds codes k = 2b (low nibble) and 2b + 1 (high nibble):
        // move them to bits 0-3 and 16-19, into the mantissas of 128 + c
        const uint32_t sel = static_cast<uint32_t>(b | (b << 4) | ((4 + b) << 8) | ((4 + b) << 12));
        const uint32_t pair = lop3_and_or(prmt(w, hi, sel), 0x000F000Fu, kMagic);
        const uint32_t c = add_bf16x2(pair, kMinus128);                // (c_2b, c_2b+1), exact
        out[16 * gg + 4 * t + b] = fma_bf16x2(c, s2, z2);
      }
    }
  }
}
// Q8: columns [128 qh, 128 qh + 128) of weight row r of one chunk, as 64
// bf16x2 words in k order: w = d*code, computed exactly in fp32 and rounded
// once to bf16.  Code (r, k) is byte k*32 + r (layout KR) or
// (r/16)*4096 + (k/32)*512 + (k%32)*16 + r%16 (layout BLK); the warp's 32
// lanes read 32 rows of one column together.  Plain C++ loads: they stay
// behind the stage's barrier wait (an asm statement with a memory clobber).
template <int KIND>
// (shared-memory loads by explicit .shared address: a generic pointer would
// take the slower generic path for each of the 128 byte loads)
__device__ __forceinline__ void dequant_half_q8(uint32_t chunk, int r, int qh, uint32_t (&out)[64]) {
  const uint2 dw = lds64(chunk + kQ8D + r * 16 + qh * 8);   // d of groups 4qh .. 4qh+3
  const uint32_t c = chunk + (KIND == kQ8_KR ? r + qh * (128 * 32) : (r >> 4) * 4096 + (r & 15) + qh * (4 * 512));
  const float2 kBias = make_float2(-8388736.f, -8388736.f);   // 2^23 + 128
  const uint32_t hi16 = KIND == kQ8_BLK && r >= 16 ? 16u : 0u;  // BLK: the 16-byte stagger of the upper half-warp
  const uint32_t swap_sel = hi16 ? 0x1032u : 0x3210u;          // ... and the swap of its bf16 halves
#pragma unroll
  for (int gg = 0; gg < 4; ++gg) {
    const uint32_t dp = gg < 2 ? dw.x : dw.y;
    const float d = __uint_as_float((gg & 1) ? (dp & 0xFFFF0000u) : (dp << 16));
    const float2 d2 = make_float2(d, d);
#pragma unroll
    for (int p = 0; p < 16; ++p) {
      const int k = 32 * gg + 2 * p;                // column within the half
      const int o0 = KIND == kQ8_KR ? k * 32 : (k >> 5) * 512 + (k & 31) * 16;
      const int o1 = KIND == kQ8_KR ? (k + 1) * 32 : ((k + 1) >> 5) * 512 + ((k + 1) & 31) * 16;
      // BLK keeps rows 16-31 4096 bytes after rows 0-15, on the same banks:
      // the upper half-warp reads the pair's other column first (16 bytes
      // on), so that each load meets 8 distinct banks, and swaps the two
      // bf16 halves of its result back
      const uint32_t u0 = lds_u8(c + o0 + hi16), u1 = lds_u8(c + o1 - hi16);
      // int8 code -> exact fp32: the bits 0x4B000000 | (u ^ 0x80) are 2^23 + 128 + code
      const float2 f = make_float2(__uint_as_float((u0 ^ 0x80u) | 0x4B000000u), __uint_as_float((u1 ^ 0x80u) | 0x4B000000u));
      const float2 w = __fmul2_rn(fadd2(f, kBias), d2);
      if constexpr (KIND == kQ8_KR) {
        out[16 * gg + p] = pack_bf16x2(w.x, w.y);
      } else {
        out[16 * gg + p] = prmt(pack_bf16x2(w.x, w.y), 0u, swap_sel);
      }
    }
  }
}
// 32 consecutive TMEM columns of this thread's lane <- r[0..31]; in flight on
// return (tcgen05.wait::st completes it).
__device__ __forceinline__ void tmem_st32_async(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
      "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
      "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

template <int KIND>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap smap,
                    const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap ymap,
                    const __grid_constant__ Args a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  using P = Plan<KIND>;
  constexpr int kWStages = P::kWStages, kWBytes = P::kWBytes, kXOff = P::kXOff;
  Shared* sh = reinterpret_cast<Shared*>(smem + P::kBarOff);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t lo = a.units * blockIdx.x / a.grid, hi = a.units * (blockIdx.x + 1) / a.grid;
  const int n = static_cast<int>(hi - lo);
  const int64_t KS = a.TC;
  const int64_t first_tile = lo / KS, last_tile = (hi - 1) / KS;
  const int ntiles = static_cast<int>(last_tile - first_tile + 1);
  asm volatile("griddepcontrol.launch_dependents;");

  if (threadIdx.x == 0) {
    for (int s = 0; s < kWStages; ++s) { mbar_init(&sh->w_full[s], 1); mbar_init(&sh->w_empty[s], kDequantWarps); }
    for (int s = 0; s < kStages; ++s) { mbar_init(&sh->full[s], 1 + kDequantWarps); mbar_init(&sh->empty[s], 1); }
    for (int s = 0; s < kAccs; ++s) { mbar_init(&sh->acc_full[s], 1); mbar_init(&sh->acc_empty[s], 4); }
    mbar_init(&sh->drain, 1);
    mbar_init(&sh->staged, 4);
    mbar_init(&sh->gather, 1);
    sh->abort_flag = 0u;
    sh->fix_seen = 0u;
    fence_barrier_init();
  }
  if (warp == kWarpAlloc) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&sh->tmem_base)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh->tmem_base;

  if (warp == kWarpW) {
    // ----------------------------------------------------------- weights
    int64_t tile = lo / KS, ks = lo - tile * KS;
    int j = 0;
    for (; j < n; ++j) {
      const int s = j % kWStages;
      if (!wait_bar_warp(sh, &sh->w_empty[s], ((j / kWStages) & 1) ^ 1u, a.err)) break;
      if (P::kQ8)
        issue_weights_q8(smem_u32(smem + kWOff + s * kWBytes), &wmap, static_cast<int>(ks), static_cast<int>(tile * 4),
                         smem_u32(&sh->w_full[s]));
      else
        issue_weights(smem_u32(smem + kWOff + s * kWBytes), &wmap, &smap, static_cast<int>(ks), static_cast<int>(tile * 4),
                      smem_u32(&sh->w_full[s]));
      if (++ks == KS) { ks = 0; ++tile; }
    }
    for (int t = (j > kWStages ? j - kWStages : 0); t < j; ++t)        // copies still in flight land first
      mbar_wait_bounded(&sh->w_full[t % kWStages], (t / kWStages) & 1, 100000000ull);
  } else if (warp == kWarpX) {
    // ----------------------------------------------------------- X
    asm volatile("griddepcontrol.wait;" ::: "memory");     // X may be the previous grid's output
    int64_t ks = lo % KS;
    int j = 0;
    for (; j < n; ++j) {
      const int s = j % kStages;
      if (!wait_bar_warp(sh, &sh->empty[s], ((j / kStages) & 1) ^ 1u, a.err)) break;
      issue_x(smem_u32(smem + kXOff + s * kXBytes), &xmap, static_cast<int>(ks), smem_u32(&sh->full[s]), a.mrows);
      if (++ks == KS) ks = 0;
    }
    // copies still in flight land first (a stage whose dequant part stopped short stays incomplete:
    // then the wait gives up after its limit, which only happens on the error path)
    for (int t = (j > kStages ? j - kStages : 0); t < j; ++t)
      mbar_wait_bounded(&sh->full[t % kStages], (t / kStages) & 1, 100000000ull);
  } else if (warp == kWarpMma) {
    // ----------------------------------------------------------- MMA issuer
    // stage s's descriptor is stage 0's plus s * kXBytes in the address field (bits 0-13, in 16-byte units)
    const uint64_t xdesc0 = sw128_desc(smem_u32(smem + kXOff));
    int64_t ks = lo % KS;
    int tcount = 0;
    bool first_in_tile = true;
    int st = 0;
    uint32_t ph = 0;
    for (int j = 0; j < n; ++j) {
      const int b = tcount & 1;
      if (first_in_tile) {
        if (!wait_bar_warp(sh, &sh->acc_empty[b], ((tcount >> 1) & 1) ^ 1u, a.err)) break;
      }
      if (!wait_bar_warp(sh, &sh->full[st], ph, a.err)) break;
      tc_fence_after();
      mma_kstep(tmem + static_cast<uint32_t>(b * kTileN), tmem + kTmemA + static_cast<uint32_t>(st) * kAStageCols,
                xdesc0 + static_cast<uint64_t>(st * (kXBytes >> 4)), first_in_tile ? 0u : 1u, &sh->empty[st]);
      first_in_tile = false;
      if (++st == kStages) { st = 0; ph ^= 1u; }
      if (++ks == KS || j == n - 1) {               // this CTA's share of the tile is complete
        mma_commit_elect(&sh->acc_full[b]);
        ++tcount;
        first_in_tile = true;
        if (ks == KS) ks = 0;
      }
    }
    mma_commit_elect(&sh->drain);                   // every MMA issued so far has completed
    mbar_wait_bounded(&sh->drain, 0, 100000000ull);
  } else if (warp >= kWarpDequant0 && ntiles == 1) {
    // ------------------------------------- dequant, twelve warps (one tile)
    // A CTA that holds a single tile runs its epilogue only at its end, so
    // the epilogue warps share the decode until then: k-step j's 8 tasks
    // (TMEM lane quarter t & 3, half t >> 2 of the k-step) go to warps
    // 4 + (8j + t) mod 12, each of the 12 warps taking two of every three
    // k-steps, always on its own lane quarter (t & 3 == warp & 3).  A stage
    // still receives 8 arrivals per k-step, and a warp waits only on the
    // k-steps it works on, so every parity it waits for is the next one.
    const int d = warp - kWarpDequant0;              // 0 .. 11
    const int i = warp & 3;                          // tile row (= TMEM lane quarter)
    const uint32_t t_lane = static_cast<uint32_t>(32 * i) << 16;
    for (int j = 0; j < n; ++j) {
      const int t = (d + 12 - (8 * j) % 12) % 12;
      if (t >= 8) continue;                          // another warp's k-step
      const int qh = t >> 2;
      const int ws = j % kWStages, st = j % kStages;
      const uint32_t wph = (j / kWStages) & 1, ph = (j / kStages) & 1;
      if (!wait_bar_warp(sh, &sh->w_full[ws], wph, a.err)) break;
      uint32_t out[64];
      if constexpr (P::kQ8) {
        dequant_half_q8<KIND>(smem_u32(smem + kWOff + ws * kWBytes + i * kQ8Bytes), lane, qh, out);
      } else {
        const uint32_t wst = smem_u32(smem + kWOff + ws * kWBytes);
        dequant_half(wst + i * kCodes, wst + 4 * kCodes + i * kScales, lane, qh, out);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh->w_empty[ws]);  // the stage's bytes are in registers
      if (!wait_bar_warp(sh, &sh->empty[st], ph ^ 1u, a.err)) break;
      tc_fence_after();
      const uint32_t tdst = tmem + t_lane + kTmemA + static_cast<uint32_t>(st) * kAStageCols + static_cast<uint32_t>(qh * 64);
      tmem_st32_async(tdst, out);
      tmem_st32_async(tdst + 32, out + 32);
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh->full[st]);
    }
  } else if (warp >= kWarpDequant0 && warp < kWarpEpi0) {
    // ----------------------------------------------------------- dequant
    // Software-pipelined: the TMEM stores of k-step j stay in flight while
    // k-step j + 1 is decoded; only then are they completed and announced.
    // The barriers a step needs are tested (without blocking) one step ahead,
    // so the round trip of the test overlaps the decode; a step blocks only if
    // its stage is really not ready.  Every dequant warp takes part in every
    // k-step, so the stage a test looks at was last used by the same warp:
    // the phase it tests is the next one, never an older one.
    const int i = warp & 3, qh = (warp - kWarpDequant0) >> 2;   // tile row (= TMEM lane quarter), half of the k-step
    const uint32_t t_lane = static_cast<uint32_t>(32 * i) << 16;
    int st = 0, pst = -1;                           // stage of this k-step, stage stored but not yet announced
    uint32_t ph = 0;
    int ws = 0;                                     // weight stage of this k-step
    uint32_t wph = 0;
    bool w_ok = mbar_test_wait(&sh->w_full[0], 0);
    for (int j = 0; j < n; ++j) {
      if (!__all_sync(0xFFFFFFFFu, w_ok) && !wait_bar_warp(sh, &sh->w_full[ws], wph, a.err)) break;
      const int ws_next = ws + 1 == kWStages ? 0 : ws + 1;
      const uint32_t wph_next = ws + 1 == kWStages ? wph ^ 1u : wph;
      const bool w_ok_next = j + 1 < n ? mbar_test_wait(&sh->w_full[ws_next], wph_next) : true;
      const bool e_ok = mbar_test_wait(&sh->empty[st], ph ^ 1u);
      uint32_t out[64];
      // (the last tile may hold fewer than 4 tile rows: the rows past the end
      // decode whatever the stage holds, and their results are never stored)
      if constexpr (P::kQ8) {
        dequant_half_q8<KIND>(smem_u32(smem + kWOff + ws * kWBytes + i * kQ8Bytes), lane, qh, out);
      } else {
        const uint32_t wst = smem_u32(smem + kWOff + ws * kWBytes);
        dequant_half(wst + i * kCodes, wst + 4 * kCodes + i * kScales, lane, qh, out);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh->w_empty[ws]); // the stage's bytes are in registers
      if (pst >= 0) {
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh->full[pst]);
        pst = -1;
      }
      if (!__all_sync(0xFFFFFFFFu, e_ok) && !wait_bar_warp(sh, &sh->empty[st], ph ^ 1u, a.err)) break;
      tc_fence_after();
      const uint32_t tdst = tmem + t_lane + kTmemA + static_cast<uint32_t>(st) * kAStageCols + static_cast<uint32_t>(qh * 64);
      tmem_st32_async(tdst, out);
      tmem_st32_async(tdst + 32, out + 32);
      pst = st;
      if (++st == kStages) { st = 0; ph ^= 1u; }
      ws = ws_next;
      wph = wph_next;
      w_ok = w_ok_next;
    }
    if (pst >= 0) {
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh->full[pst]);
    }
  }
  if (warp >= kWarpEpi0) {
    // ----------------------------------------------------------- epilogue
    // Only a CTA's last tile can be one it finishes (its first k-step here,
    // later ones in other CTAs); the last CTA holding part of it is worked out
    // now, before the wait: a 64-bit division at the end of the launch sits on
    // its critical path.
    const int64_t c_last_tile = ((last_tile + 1) * KS * a.grid - 1) / a.units;
    asm volatile("griddepcontrol.wait;" ::: "memory");     // Y and the workspace may be the previous grid's
    const int e = warp & 3;                         // TMEM lane quarter of this warp
    const int row = 32 * e + lane;                  // row within the 128-row tile
    for (int t = 0; t < ntiles; ++t) {
      const int b = t & 1;
      const int64_t tile = first_tile + t;
      const int64_t u_lo = tile * KS, u_hi = u_lo + KS;
      const bool whole = lo <= u_lo && u_hi <= hi;   // the whole tile is computed here
      const bool contrib = u_lo < lo;                // another CTA holds the tile's first k-step
      const bool finisher = !whole && !contrib;
      // finisher: the later CTAs' partials of this thread's row, summed in an
      // order fixed by the shape, gathered before the accumulator is ready
      // (token quad k in fx[k])
      float4 fx[kTileN / 4];
      const bool last = t == ntiles - 1;
      if (finisher) {
        // each posting CTA counts once per epilogue warp
        const int64_t c_last = c_last_tile;          // (u_hi * grid - 1) / units: this is the last tile
        if (!wait_posted(sh, &a.counters[tile], static_cast<uint32_t>(4 * (c_last - blockIdx.x)), a.err, lane))
          break;
        const float4* p = reinterpret_cast<const float4*>(a.partials + (blockIdx.x + 1) * (kTileN * kTileM)) + row;
#pragma unroll
        for (int k = 0; k < kTileN / 4; ++k) fx[k] = ld_cg_f32x4(p + k * kTileM);   // one round trip
        // the later CTAs' partials: on the last tile, once the accumulator is
        // final, through bulk copies into the then free stage memory (one
        // round trip for all of them); beyond those slots, or on another tile,
        // here, half a partial per round trip
        for (int64_t c = blockIdx.x + 2 + (last ? kGatherSlots : 0); c <= c_last; ++c) {
          p = reinterpret_cast<const float4*>(a.partials + c * (kTileN * kTileM)) + row;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            float4 v[kTileN / 8];
#pragma unroll
            for (int k = 0; k < kTileN / 8; ++k) v[k] = ld_cg_f32x4(p + (8 * h + k) * kTileM);
#pragma unroll
            for (int k = 0; k < kTileN / 8; ++k) {
              float4& f = fx[8 * h + k];
              f = make_float4(f.x + v[k].x, f.y + v[k].y, f.z + v[k].z, f.w + v[k].w);
            }
          }
        }
        // the last epilogue warp through clears the count for the next launch
        if (lane == 0 && atomicAdd(&sh->fix_seen, 1u) == 3u) a.counters[tile] = 0u;
      }
      if (!wait_bar(sh, &sh->acc_full[b], (t >> 1) & 1, a.err)) break;
      tc_fence_after();
      const int64_t n0 = tile * kTileM;
      const bool valid_row = n0 + row < a.N;
      float4* mine = reinterpret_cast<float4*>(a.partials + static_cast<int64_t>(blockIdx.x) * (kTileN * kTileM)) + row;
      const uint32_t taddr = tmem + (static_cast<uint32_t>(32 * e) << 16) + static_cast<uint32_t>(b * kTileN);
      if (last && !contrib) {
        // last tile: stage it in X stage 0 ([64 tokens][128 rows] of the
        // output type), then one thread writes it to Y with a single tensor
        // copy.  (A partial goes out from registers below: its rows are
        // 512-byte coalesced stores, and the finisher waits on it, so it
        // should be visible as soon as possible.)
        const uint32_t stg = smem_u32(smem + kXOff);
        if (finisher) {
          const int64_t later = c_last_tile - blockIdx.x - 1;   // partials past the first
          const int nsm = static_cast<int>(later < kGatherSlots ? later : kGatherSlots);
          if (nsm > 0) {
            if (warp == kWarpEpi0 && lane == 0) {
              // the partials were seen through the counter's acquire; order that before the copies' reads
              asm volatile("fence.proxy.async.global;" ::: "memory");
              mbar_arrive_expect_tx(&sh->gather, static_cast<uint32_t>(nsm * kTileN * kTileM * 4));
              for (int i = 0; i < nsm; ++i)
                bulk_g2s(smem + gather_slot<KIND>(i), a.partials + (blockIdx.x + 2 + i) * (kTileN * kTileM),
                         kTileN * kTileM * 4, &sh->gather);
            }
            if (!wait_bar(sh, &sh->gather, 0, a.err)) break;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
#pragma unroll 1
              for (int i = 0; i < nsm; ++i) {
                const uint32_t src = smem_u32(smem + gather_slot<KIND>(i)) + static_cast<uint32_t>(row * 16);
                float4 v[kTileN / 8];
#pragma unroll
                for (int k = 0; k < kTileN / 8; ++k) v[k] = lds_f32x4(src + static_cast<uint32_t>((8 * h + k) * kTileM * 16));
#pragma unroll
                for (int k = 0; k < kTileN / 8; ++k) {
                  float4& f = fx[8 * h + k];
                  f = make_float4(f.x + v[k].x, f.y + v[k].y, f.z + v[k].z, f.w + v[k].w);
                }
              }
            }
          }
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          float v[32];
          tmem_ld32(taddr + 32 * h, v);
          if (finisher) {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              v[4 * k] += fx[8 * h + k].x;
              v[4 * k + 1] += fx[8 * h + k].y;
              v[4 * k + 2] += fx[8 * h + k].z;
              v[4 * k + 3] += fx[8 * h + k].w;
            }
          }
#pragma unroll
          for (int m = 0; m < 32; ++m) {
            const uint32_t idx = static_cast<uint32_t>((32 * h + m) * kTileM + row);
            if (a.out_f32) sts_f32(stg + idx * 4, v[m]);
            else sts_u16(stg + idx * 2, f32_to_bf16_bits(v[m]));
          }
        }
        tc_fence_before();
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // staged bytes visible to the bulk copy
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&sh->acc_empty[b]);
          mbar_arrive(&sh->staged);
        }
        if (warp == kWarpEpi0 && lane == 0) {
          if (!wait_bar(sh, &sh->staged, 0, a.err)) break;
          tma_store_2d(&ymap, static_cast<int>(n0), 0, stg);
          bulk_commit();
          bulk_wait_read();
        }
        continue;
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float v[32];
        tmem_ld32(taddr + 32 * h, v);
        if (contrib) {
#pragma unroll
          for (int k = 0; k < 8; ++k)
            mine[(8 * h + k) * kTileM] = make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
        } else {
          if (finisher) {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              v[4 * k] += fx[8 * h + k].x;
              v[4 * k + 1] += fx[8 * h + k].y;
              v[4 * k + 2] += fx[8 * h + k].z;
              v[4 * k + 3] += fx[8 * h + k].w;
            }
          }
          if (valid_row) store_slice(a, n0 + row, 32 * h, v);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh->acc_empty[b]);
      if (contrib) {
        // post this warp's rows of the partial: every lane's stores, then one release count
        __threadfence();
        __syncwarp();
        if (lane == 0) red_release_add(&a.counters[tile], 1u);
      }
    }
  }

  __syncwarp();                                     // whole warps arrive at the CTA barrier
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpAlloc) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
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

bool gemm_supports(int kind) { return kind == kQ4_1 || kind == kQ8_KR || kind == kQ8_BLK; }

uint64_t gemm_workspace_bytes(int64_t TR, int64_t TC, int M) {
  (void)TC;
  (void)M;
  const int64_t tiles = (TR + 3) / 4;
  // error word, one partial tile per CTA (at most 1024 CTAs), posting
  // counters.  The partials come first: their region has the same place and
  // size for every weight, and the regions whose place depends on the weight
  // (the counters, and the few-token GEMV's part after them) are left
  // zero-filled by every call, so weights of different sizes can share one
  // workspace without stale partials reaching another weight's counters.
  return kWsErrBytes + gemm::kPartialBytes + align16(static_cast<uint64_t>(tiles) * 4);
}

namespace {
template <int KIND>
cudaError_t launch_gemm_kind(EncodeTiled enc, const DeviceInfo& info, const void* chunks, int64_t TR, int64_t TC,
                             const void* X, int M, void* Y, int out_f32, void* workspace, cudaStream_t s) {
  using P = gemm::Plan<KIND>;
  if (info.max_smem_optin < P::kSmemBytes) return cudaErrorNotSupported;
  // weights, q4_1: code regions as [128 B][32 rows][TC chunk columns][TR tile rows] (128-byte swizzle)
  // and scale/zero regions as [256 B][4][TC][TR] from byte 4096 of each chunk; Q8: whole chunks as
  // [256 B][34][TC][TR].  X as [64 k][M tokens][K / 64]; Y as [N][M].
  CUtensorMap wmap, smap, xmap, ymap;
  if (P::kQ8) {
    cuuint64_t dims[4] = {256, kQ8Bytes / 256, static_cast<cuuint64_t>(TC), static_cast<cuuint64_t>(TR)};
    cuuint64_t strides[3] = {256, kQ8Bytes, static_cast<cuuint64_t>(kQ8Bytes) * static_cast<cuuint64_t>(TC)};
    cuuint32_t box[4] = {256, kQ8Bytes / 256, 1, 4};
    cuuint32_t es[4] = {1, 1, 1, 1};
    static_assert(kQ8Bytes % 256 == 0, "Q8 chunk as rows of 256 bytes");
    if (enc(&wmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(chunks), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
    smap = wmap;                                    // unused for Q8
  } else {
    {
      cuuint64_t dims[4] = {128, 32, static_cast<cuuint64_t>(TC), static_cast<cuuint64_t>(TR)};
      cuuint64_t strides[3] = {128, kQ41Bytes, static_cast<cuuint64_t>(kQ41Bytes) * static_cast<cuuint64_t>(TC)};
      cuuint32_t box[4] = {128, 32, 1, 4};
      cuuint32_t es[4] = {1, 1, 1, 1};
      if (enc(&wmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(chunks), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    }
    {
      cuuint64_t dims[4] = {256, 4, static_cast<cuuint64_t>(TC), static_cast<cuuint64_t>(TR)};
      cuuint64_t strides[3] = {256, kQ41Bytes, static_cast<cuuint64_t>(kQ41Bytes) * static_cast<cuuint64_t>(TC)};
      cuuint32_t box[4] = {256, 4, 1, 4};
      cuuint32_t es[4] = {1, 1, 1, 1};
      void* base = const_cast<uint8_t*>(static_cast<const uint8_t*>(chunks) + kQ41Scale);
      if (enc(&smap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, base, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    }
  }
  {
    // X [M][K]: boxes of 64 columns x mrows tokens
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(TC * 256), static_cast<cuuint64_t>(M)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(TC * 256 * 2)};
    cuuint32_t box[2] = {64, static_cast<cuuint32_t>((M + 7) & ~7)};
    cuuint32_t es[2] = {1, 1};
    if (enc(&xmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(X), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    // Y [M][N] of the output type, box of 128 rows x 64 tokens (rows or tokens past the end are not written)
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(TR * 32), static_cast<cuuint64_t>(M)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(TR * 32) * (out_f32 ? 4u : 2u)};
    cuuint32_t box[2] = {128, 64};
    cuuint32_t es[2] = {1, 1};
    if (enc(&ymap, out_f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, Y, dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  gemm::Args a;
  const int64_t tiles = (TR + 3) / 4;
  a.chunks = static_cast<const uint8_t*>(chunks);
  a.Y = Y;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  a.err = reinterpret_cast<uint32_t*>(ws);
  a.partials = reinterpret_cast<float*>(ws + kWsErrBytes);
  a.counters = reinterpret_cast<uint32_t*>(ws + kWsErrBytes + gemm::kPartialBytes);
  a.TR = TR;
  a.TC = TC;
  a.N = TR * 32;
  a.tiles = static_cast<int>(tiles);
  a.M = M;
  a.mrows = (M + 7) & ~7;
  a.out_f32 = out_f32;
  a.units = tiles * TC;
  // at least 4 k-steps per CTA where the work allows it, at most one CTA per SM
  int64_t grid = (a.units + 3) / 4;
  if (grid > info.sms) grid = info.sms;
  // Where the tiles allow it, every tile in the same number s of equal parts
  // (s dividing the tile's k-steps, at least 4 k-steps a part, the grid
  // tiles * s filling at least 60 % of the SMs): no CTA's range then lies
  // inside a single tile, so a tile's parts finish together and its finisher
  // does not wait for a CTA that holds only its middle (which posts at its
  // own end); the SMs left free take the next launch's first copies.
  // Measured on GB300, back to back: 12288x4096 14.38 -> 13.86 us (96 CTAs of
  // one whole tile), 4096x12288 16.07 -> 15.06 us (128 CTAs of a quarter tile).
  {
    int64_t parts = 0;
    for (int64_t sp = 1; sp <= TC / 4 && tiles * sp <= info.sms; ++sp)
      if (TC % sp == 0) parts = sp;
    if (parts > 0 && tiles * parts * 10 >= 6 * static_cast<int64_t>(info.sms)) grid = tiles * parts;
  }
  if (grid > 1024) grid = 1024;
  if (grid < 1) grid = 1;
  a.grid = static_cast<int>(grid);
  cudaError_t e = set_max_dynamic_smem(reinterpret_cast<const void*>(gemm::gemm_kernel<KIND>));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.grid);
  cfg.blockDim = dim3(gemm::kThreads);
  cfg.dynamicSmemBytes = P::kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, gemm::gemm_kernel<KIND>, wmap, smap, xmap, ymap, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_gemm(int kind, const void* chunks, int64_t TR, int64_t TC, const void* X, int M, void* Y,
                        int out_f32, void* workspace, cudaStream_t s) {
  if (!gemm_supports(kind)) return cudaErrorNotSupported;
  EncodeTiled enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  DeviceInfo info;
  cudaError_t e = device_info(&info);
  if (e != cudaSuccess) return e;
  switch (kind) {
    case kQ4_1: return launch_gemm_kind<kQ4_1>(enc, info, chunks, TR, TC, X, M, Y, out_f32, workspace, s);
    case kQ8_KR: return launch_gemm_kind<kQ8_KR>(enc, info, chunks, TR, TC, X, M, Y, out_f32, workspace, s);
    default: return launch_gemm_kind<kQ8_BLK>(enc, info, chunks, TR, TC, X, M, Y, out_f32, workspace, s);
  }
}

}  // namespace q4nx
