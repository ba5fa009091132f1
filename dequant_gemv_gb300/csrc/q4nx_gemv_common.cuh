// q4nx_gemv_common.cuh -- pieces shared by the two GEMV kernels of libq4nx.so
// (sm_103a): the launch arguments, chunk positions, and the exact fixed-point
// preparation of the activations for the 4-bit chunk kinds.
//
// The weight formulas are the chunk-kind table's ("Q4NX chunks" section of the
// 1bit engine "NPU engine" page): q4_1 code*scale + zero, Q4_K
// S*scale*code + M*min.  The codes meet x in exact integer arithmetic: per
// 32-column group, x becomes NP-byte fixed point (NP = 3 or 4 signed digit
// planes), exact when the group's magnitudes span at most 2^14 (2^22), so
// that each plane's partial s*S_p*q_p + z*X_p*q_p is formed from exact
// operands and rounded once.
#pragma once

#include "q4nx_device.cuh"
#include "q4nx_kernels.h"

namespace q4nx {

constexpr int kXSliceBytes = 512;            // bf16 x of one tile column, per token
constexpr int kScratchBytes = 1024;          // per warp and token: x digit planes (or the raw x slice) of one chunk
constexpr int kSlotBytes = 2 * 32 * 4;       // per warp and token: sums of its first and last tile row
constexpr int kCntBytes = 8;                 // per warp: arrival counters of its first and last tile row
constexpr int kMaxBatch = kMaxGemvItems;

struct GemvItemDev {
  const uint8_t* chunks;
  const uint8_t* x;        // bf16 [K] (token m at x + m * x_stride)
  void* y;                 // [N] (token m at y + m * y_stride elements)
  int64_t cbase;           // first unit of this item in the batch index space
  int64_t nchunks;         // its units: TR * TC chunks (times 4 when the units are quarters of chunks)
  int32_t TC;              // units per tile row: tile columns (times 4 for quarters)
};

// Kernel parameters; MAXB batch slots (instantiated for 1, 8 and 256 items so
// that small launches do not carry a 12 KB parameter block).
template <int MAXB>
struct GemvArgsT {
  GemvItemDev items[MAXB];
  int nitems;
  int grid;                // CTAs; CTA b owns units [T b / grid, T (b+1) / grid)
  int stages;
  int xslots;              // 4-bit kinds: x-slice cache slots in shared memory, each m tokens (0: none)
  int out_f32;
  int m;                   // tokens (1 unless one item against several tokens)
  int64_t x_stride;        // bytes between tokens' x
  int64_t y_stride;        // elements between tokens' y
  int64_t T;               // units in the batch (chunks, or quarters of chunks)
  uint32_t* err;
  uint64_t* posted;        // [grid][MT][32]: a CTA's sums of its first tile row when an earlier CTA finishes it
  // top-1 mode (one item): instead of storing y, keep the largest (fp32 value,
  // row) key; the last CTA to finish writes the row index and/or the key
  int top1;                // 0: store y
  uint32_t top1_row_base;  // added to the rows in the keys (a shard's first row)
  int32_t* top1_idx;       // null, or where the row goes
  int64_t* top1_key_out;   // null, or where the key goes (top bit flipped: signed order = key order)
  uint64_t* top1_key;      // workspace word, zero between launches
  uint32_t* top1_done;     // workspace word, zero between launches
};


constexpr int kXRecBytes = 256;            // per token: the 8 groups' records in an x-slice cache slot
constexpr int kXSlotBytes = kScratchBytes + kXRecBytes;   // per token and slice
constexpr int kXTabItems = 16;
constexpr int kMaxXSlots = 32;

// CTA that holds chunk c: the largest b with floor(T*b/G) <= c
__device__ __forceinline__ int64_t cta_of(int64_t c, int64_t T, int64_t G) { return ((c + 1) * G - 1) / T; }


constexpr uint64_t kPosted = 1ull << 32;


__device__ __forceinline__ uint32_t dp4a_uu(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("dp4a.u32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) { return __fmul2_rn(a, b); }


// Per token, for the lane's group g = lane & 7 (prep and decode lanes of a
// group share the low three lane bits): the weight of the lowest digit plane
// and the digit sums times the plane weights.
struct XGroup {
  float q0;                        // 2^(E - 124 - 8 NP); plane p weighs q0 256^p
  float xq[4];                     // X_p q0 256^p
};

// How many digit planes one token's x slice needs for this lane's group (all
// four prep lanes of the group get the same answer): 3 when every value is a
// multiple of 2^(E-148) below 2^(E-126) (E the biased exponent of the group's
// largest |x|: nonzero values within 2^14 of the largest, 22 <= E <= 254), 4
// when within 2^22 (30 <= E <= 254, step 2^(E-156)), else 5 (none does: the
// binary32 path).  An all-zero group needs 3.
__device__ __forceinline__ int q4_x_need(const uint4 xr, int& E) {
  const uint32_t xw[4] = {xr.x, xr.y, xr.z, xr.w};
  const uint32_t m2 = __vmaxu2(__vmaxu2(xw[0] & 0x7FFF7FFFu, xw[1] & 0x7FFF7FFFu),
                               __vmaxu2(xw[2] & 0x7FFF7FFFu, xw[3] & 0x7FFF7FFFu));
  uint32_t mx = max(m2 & 0xFFFFu, m2 >> 16);
  // smallest nonzero |x| as (binary32 bits << 1) - 1: the sign drops out and
  // +-0 becomes 0xFFFFFFFF, above every other key
  uint32_t mn = 0xFFFFFFFFu;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    mn = min(mn, (xw[j] << 17) - 1u);
    mn = min(mn, ((xw[j] & 0xFFFF0000u) << 1) - 1u);
  }
  mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
  mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
  mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, 8));
  mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, 16));
  E = static_cast<int>(mx >> 7);
  const int emin = static_cast<int>((mn + 1u) >> 24);    // exponent field of the smallest nonzero |x|
  if (mx == 0 || (E >= 22 && E <= 254 && emin >= E - 14)) return 3;
  if (E >= 30 && E <= 254 && emin >= E - 22) return 4;
  return 5;
}

// One token's x slice (this prep lane's 8 columns) -> NP digit planes in
// `scratch`: region A [t][g] 16 B (p0 even, p0 odd, p1 even, p1 odd) and
// region B at +512 [t][g] 16 B (p2 even, p2 odd, p3 even, p3 odd); and the
// group's plane weight and digit sums.  v_k = x_k 2^(124 + 8 NP - E), |v_k| <
// 2^(8 NP - 2), exact by q4_x_need; v_k + 0x80..80 has the bytes d_p + 128.
template <int NP>
__device__ __forceinline__ void q4_x_planes(const uint4 xr, int E, uint32_t scratch, int lane, XGroup& G) {
  const int gp = lane & 7, tp = lane >> 3;
  E = min(max(E, 8 * NP - 2), 254);                              // (an all-zero group: any step)
  const float sc = __int_as_float((251 + 8 * NP - E) << 23);     // 2^(124 + 8 NP - E)
  const uint32_t xw[4] = {xr.x, xr.y, xr.z, xr.w};
  uint32_t v[8];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float f0 = __uint_as_float(xw[j] << 16), f1 = __uint_as_float(xw[j] & 0xFFFF0000u);
    if constexpr (NP == 3) {                                     // |v| < 2^22: round by the 1.5 * 2^23 magic number
      v[2 * j] = __float_as_uint(fmaf(f0, sc, 12582912.0f)) - 0x4ABF7F80u;
      v[2 * j + 1] = __float_as_uint(fmaf(f1, sc, 12582912.0f)) - 0x4ABF7F80u;
    } else {                                                     // |v| < 2^30: an integer conversion
      v[2 * j] = static_cast<uint32_t>(__float2int_rn(f0 * sc)) + 0x80808080u;
      v[2 * j + 1] = static_cast<uint32_t>(__float2int_rn(f1 * sc)) + 0x80808080u;
    }
  }
  // gather byte p of the even and of the odd columns, then flip the top bit
  // of each byte to get d_p
  const uint32_t ae = prmt(v[0], v[2], 0x5140), be = prmt(v[4], v[6], 0x5140);
  const uint32_t ao = prmt(v[1], v[3], 0x5140), bo = prmt(v[5], v[7], 0x5140);
  const uint32_t ce = prmt(v[0], v[2], 0x7362), de = prmt(v[4], v[6], 0x7362);
  const uint32_t co = prmt(v[1], v[3], 0x7362), dq = prmt(v[5], v[7], 0x7362);
  uint32_t P[4][2];
  P[0][0] = prmt(ae, be, 0x5410) ^ 0x80808080u;
  P[0][1] = prmt(ao, bo, 0x5410) ^ 0x80808080u;
  P[1][0] = prmt(ae, be, 0x7632) ^ 0x80808080u;
  P[1][1] = prmt(ao, bo, 0x7632) ^ 0x80808080u;
  P[2][0] = prmt(ce, de, 0x5410) ^ 0x80808080u;
  P[2][1] = prmt(co, dq, 0x5410) ^ 0x80808080u;
  P[3][0] = NP == 4 ? prmt(ce, de, 0x7632) ^ 0x80808080u : 0u;
  P[3][1] = NP == 4 ? prmt(co, dq, 0x7632) ^ 0x80808080u : 0u;
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(scratch + (tp * 8 + gp) * 16), "r"(P[0][0]),
               "r"(P[0][1]), "r"(P[1][0]), "r"(P[1][1])
               : "memory");
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(scratch + 512 + (tp * 8 + gp) * 16), "r"(P[2][0]),
               "r"(P[2][1]), "r"(P[3][0]), "r"(P[3][1])
               : "memory");
  G.q0 = __int_as_float((E + 3 - 8 * NP) << 23);                 // 2^(E - 124 - 8 NP)
#pragma unroll
  for (int p = 0; p < NP; ++p) {
    int X = dp4a_us(0x01010101u, P[p][0], dp4a_us(0x01010101u, P[p][1], 0));
    X += __shfl_xor_sync(0xffffffffu, X, 8);
    X += __shfl_xor_sync(0xffffffffu, X, 16);                    // X_p of group gp (|X_p| <= 4096)
    G.xq[p] = static_cast<float>(X) * __int_as_float((E + 3 - 8 * NP + 8 * p) << 23);   // exact
  }
}


// Position of a unit in the batch: item, tile row and column, with the
// chunk's address and its x slice's, and the item's tile columns and units
// left.  A unit is a chunk, or with QTR a quarter of one (8 of its 32 rows,
// quarter h): then the item table counts units (4 per chunk) and `tc` is the
// unit column (chunk column tc / 4).  Workers walk their ranges in order, so a
// position advances by one unit with pointer increments; the item table (kernel
// parameters, read with a dynamic index) is read only when the walk enters the
// next item.
struct Pos {
  int it;
  int32_t tr, tc;
  int32_t TC;
  int32_t h;                        // quarter of the chunk (QTR), else 0
  int32_t left;                     // units of the item from this one to its end (tile counts fit 31 bits)
  const uint8_t* w;                 // this chunk
  const uint8_t* x;                 // the x slice of its tile column (token 0)
  template <int CB, bool QTR, class GemvArgs>
  __device__ __forceinline__ void enter(const GemvArgs& a, int item, int64_t local) {
    const GemvItemDev& I = a.items[item];
    it = item;
    TC = I.TC;
    left = static_cast<int32_t>(I.nchunks - local);
    tr = static_cast<int32_t>(local / TC);
    tc = static_cast<int32_t>(local - static_cast<int64_t>(tr) * TC);
    const int32_t cc = QTR ? tc >> 2 : tc;                      // chunk column
    h = QTR ? tc & 3 : 0;
    w = I.chunks + (static_cast<int64_t>(tr) * (QTR ? TC >> 2 : TC) + cc) * CB;
    x = I.x + static_cast<int64_t>(cc) * kXSliceBytes;
  }
  template <int CB, bool QTR, class GemvArgs>
  __device__ __forceinline__ void seek(const GemvArgs& a, int64_t c) {
    int lo = 0, hi = a.nitems - 1;                  // last item with cbase <= c
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (a.items[mid].cbase <= c) lo = mid; else hi = mid - 1;
    }
    enter<CB, QTR>(a, lo, c - a.items[lo].cbase);
  }
  template <int CB, bool QTR, class GemvArgs>
  __device__ __forceinline__ void next(const GemvArgs& a) {
    if (!QTR || ++h == 4) {
      h = 0;
      w += CB;
      x += kXSliceBytes;
    }
    if (++tc == TC) { tc = 0; ++tr; x -= static_cast<int64_t>(QTR ? TC >> 2 : TC) * kXSliceBytes; }
    if (--left == 0 && it + 1 < a.nitems) {                         // the next item's first unit
      const GemvItemDev& I = a.items[++it];
      TC = I.TC;
      left = static_cast<int32_t>(I.nchunks);
      tr = 0;
      tc = 0;
      h = 0;
      w = I.chunks;
      x = I.x;
    }
  }
};


__device__ __forceinline__ uint4 ld_cg_u4(const void* p) {
  uint4 v;
  asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

// One x slice of each of m tokens (their bf16 values in this prep lane's
// xr[tok]) into the cache slot at sa: token tok's planes at
// sa + tok * kScratchBytes, as 3 or 4 digit planes (the most any group of any
// token needs, so that the chunk's arithmetic takes one mode for all tokens),
// or the raw slices for the binary32 path; its group records, q0, xq0..xq3
// and that mode, at sa + MT * kScratchBytes + tok * kXRecBytes.
template <int MT>
__device__ __forceinline__ void xslot_fill(const uint4 (&xr)[MT], uint32_t sa, int m, int lane) {
  const int gp = lane & 7, tp = lane >> 3;
  int E[MT];
  int need = 3;
#pragma unroll
  for (int tok = 0; tok < MT; ++tok)
    if (MT == 1 || tok < m) need = max(need, q4_x_need(xr[tok], E[tok]));
  need = __reduce_max_sync(0xffffffffu, need);
#pragma unroll
  for (int tok = 0; tok < MT; ++tok) {
    if (MT > 1 && tok >= m) break;
    const uint32_t st = sa + tok * kScratchBytes;
    XGroup G = {};
    if (need == 3) {
      q4_x_planes<3>(xr[tok], E[tok], st, lane, G);
    } else if (need == 4) {
      q4_x_planes<4>(xr[tok], E[tok], st, lane, G);
    } else {
      asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(st + (tp * 8 + gp) * 16), "r"(xr[tok].x),
                   "r"(xr[tok].y), "r"(xr[tok].z), "r"(xr[tok].w)
                   : "memory");
    }
    if (tp == 0) {
      const uint32_t gr = sa + MT * kScratchBytes + tok * kXRecBytes + gp * 32;
      asm volatile("st.shared.v4.f32 [%0], {%1,%2,%3,%4};" ::"r"(gr), "f"(G.q0), "f"(G.xq[0]), "f"(G.xq[1]),
                   "f"(G.xq[2])
                   : "memory");
      asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(gr + 16), "r"(__float_as_uint(G.xq[3])),
                   "r"(static_cast<uint32_t>(need)), "r"(0u), "r"(0u)
                   : "memory");
    }
  }
}


}  // namespace q4nx
