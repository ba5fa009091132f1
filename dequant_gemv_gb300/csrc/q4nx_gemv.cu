// q4nx_gemv.cu -- fused decode + GEMV over Q4NX chunks for one to a few
// tokens, sm_103a.
//
// y_m[n] = sum_k w[n][k] x_m[k], weights in the chunk kinds of the "Q4NX
// chunks" section of the 1bit engine "NPU engine" page (chunk-kind table:
// q4_1 code*scale+zero, Q4_K S*scale*code+M*min, Q8 d*code in layout KR or
// BLK).  One launch runs a batch of independent one-token GEMVs of one chunk
// kind (a single GEMV is a batch of one), or one weight against MT tokens.
//
// Design (HBM-bound: 0.625 B/weight for q4_1):
//  * Persistent grid, one CTA per SM (two for 4-bit launches of 128 chunks or
//    more per SM, each within half an SM).  One-token 4-bit launches of at most
//    8 chunks per SM (the projections of a small decode layer) take quarters
//    of chunks (8 rows) as units, up to 16 warps per CTA: a warp's arithmetic
//    on a whole chunk would otherwise be the launch's critical path.  The chunks of all items form one index
//    space (item after item, each row-major over its tile grid); CTA b owns an
//    even contiguous share, each warp a contiguous part of it.  A range is a
//    run of (item, tile row) segments.
//  * Each warp streams its chunks with 1-D bulk async copies (TMA
//    cp.async.bulk) into its own ring of shared-memory stages: the chunk and
//    the 512-byte bf16 slices of x for the chunk's tile column, completing on
//    one mbarrier per stage.  Every wait is bounded.  The chunks are fetched
//    before the kernel waits on the previous grid (weights never change
//    between launches); x only after.
//  * 4-bit kinds: the lanes first read their share of the stage into
//    registers and the stage is refilled at once; then x becomes 24-bit fixed
//    point per 32-column group (three signed digit planes) and the code dot
//    products are exact dp4a integer sums; scale and zero are applied per
//    (row, group, plane), each plane's partial rounded once.  A chunk whose x
//    groups that fixed point cannot hold exactly takes a binary32 path.
//  * Q8 kinds: codes become exact floats through the 2^23 magic number and
//    packed fp32 FMAs; d scales each lane's (row, group) partial.
//  * Row sums are finished with a warp transpose-reduce.  A tile row split
//    between warps of a CTA is finished by the last of them to arrive (a
//    shared-memory counter), one split between CTAs by the CTA holding its
//    first chunk, which reads the others' sums posted as (value, ready flag)
//    words.  Partials are added in a fixed order, so results do not depend on
//    timing, and the workspace is left zero-filled.
#include "q4nx_gemv_common.cuh"

namespace q4nx {

// This CTA's largest top-1 key so far (top-1 mode).
__shared__ unsigned long long s_top1_key;
// Where each warp's range starts, relative to the CTA's, and the last CTA that
// holds part of the tile row at the end of this CTA's range.  Both are worked
// out before the kernel waits on the previous grid: the row sums at the end of
// a launch then need no 64-bit division, which cost 0.3-0.7 us a launch on
// that critical path.
constexpr int kMaxGemvWarps = 16;          // warps per CTA the plan may choose (12 at most today)
__shared__ uint32_t s_wlo[kMaxGemvWarps + 1];     // [nwarps]: the CTA's chunk count
__shared__ long long s_clast;
// The CTA's range [Lc, Hc): kept here for the row sums, not in registers
// across the main loop.
__shared__ long long s_range[2];

// x-slice cache (4-bit kinds).  Every warp used to turn the x
// slice of each chunk it read into digit planes, although the chunks of one
// tile column share the slice: with a CTA's range spanning several tile rows,
// that preparation was repeated for every row (a fifth of the arithmetic).
// A CTA whose chunks touch at most kXTabItems items and as many (item, tile
// column) slices as the launch's cache slots holds prepares each slice once,
// after the wait on the previous grid, into a 1280-byte slot: regions A and B
// (512 B each) as in a warp's scratch, or the raw bf16 slice when the slice
// needs the binary32 path; then per group 32 B: q0, xq0..xq3 and the slice's
// mode (3 or 4 digit planes, 5 for binary32).  With several tokens a slot
// holds every token's 1024 bytes of planes (the token stride of a warp's
// scratch) and then every token's 256 bytes of group records, all prepared
// in one mode: the largest any token's group needs.  Slots of one item are
// its touched tile columns in order, starting from column tc0 and wrapping.
__shared__ int4 s_xtab[kXTabItems];        // per touched item: {first slot, tc0, slots, TC}
__shared__ int s_xinfo[4];                 // cache used (0/1), first touched item, slots in use, items touched

// Lane-wise transpose-reduce of 8 values over the 8 lanes selected by masks
// (m2, m1, m0): afterwards the lane whose mask bits read (b2 b1 b0) holds the
// sum over those lanes of v[4 b2 + 2 b1 + b0].
__device__ __forceinline__ float transpose_reduce8(float v[8], int lane, int m2, int m1, int m0) {
  const bool b2 = lane & m2, b1 = lane & m1, b0 = lane & m0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    float send = b2 ? v[j] : v[j + 4];
    float keep = b2 ? v[j + 4] : v[j];
    v[j] = keep + __shfl_xor_sync(0xffffffffu, send, m2);
  }
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    float send = b1 ? v[j] : v[j + 2];
    float keep = b1 ? v[j + 2] : v[j];
    v[j] = keep + __shfl_xor_sync(0xffffffffu, send, m1);
  }
  float send = b0 ? v[0] : v[1];
  float keep = b0 ? v[1] : v[0];
  return keep + __shfl_xor_sync(0xffffffffu, send, m0);
}

// Row n's final value (called by all 32 lanes of a warp together, one row
// each): store it, or in top-1 mode fold it into the CTA's largest key.
template <class GemvArgs>
__device__ __forceinline__ void* token_y(const GemvArgs& a, void* y, int tok) {
  return static_cast<char*>(y) + static_cast<int64_t>(tok) * a.y_stride * (a.out_f32 ? 4 : 2);
}

template <class GemvArgs>
__device__ __forceinline__ void store_y(const GemvArgs& a, void* y, int64_t n, float v) {
  if (a.top1) {
    uint64_t key = argmax_key(v, a.top1_row_base + static_cast<uint32_t>(n));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) key = umax64(key, __shfl_xor_sync(0xffffffffu, key, o));
    if ((threadIdx.x & 31) == 0) atomicMax(&s_top1_key, static_cast<unsigned long long>(key));
    return;
  }
  if (a.out_f32) static_cast<float*>(y)[n] = v;
  else static_cast<uint16_t*>(y)[n] = f32_to_bf16_bits(v);
}


// A tile row [r0, r1) shared with other CTAs, after this CTA's warps have
// combined their parts (lane = row, `val` = this CTA's sum).  The CTA holding
// the row's first chunk finishes it: it reaches its part last (at the end of
// its range), so the others have usually posted theirs long before.  A
// poster writes, per row, one 64-bit word holding its sum and a ready flag,
// so the value and its readiness travel together and one read serves both;
// the finisher reads the posted words (waiting, bounded, for any not yet
// ready), adds them in CTA order after its own sum, stores y and clears the
// words it used.
template <int MT, class GemvArgs>
__device__ __noinline__ void cross_cta_row(const GemvArgs& a, int64_t b, int64_t Lc, int it, int64_t tr, int64_t r0,
                                           int64_t r1, const float (&val)[MT], int lane) {
  const GemvItemDev& item = a.items[it];
  const int m = (MT == 1) ? 1 : a.m;
  if (r0 < Lc) {                                      // not the finisher: post
#pragma unroll
    for (int tok = 0; tok < MT; ++tok)
      if (tok < m) st_relaxed_u64(&a.posted[(b * MT + tok) * 32 + lane], kPosted | __float_as_uint(val[tok]));
    return;
  }
  const int64_t c_last = s_clast;                     // cta_of(r1 - 1), worked out at the start
  float sum[MT];
#pragma unroll
  for (int tok = 0; tok < MT; ++tok) sum[tok] = val[tok];
  // With several contributors (a tile row of 38-48 chunks spreads over 2-3
  // CTAs) their words are loaded kBatch CTAs at a time, so that the L2 round
  // trips overlap; they are added in CTA order all the same.  One contributor
  // (the common case) takes the plain loop.
  constexpr int kBatch = 4;
  if (c_last == b + 1) {
#pragma unroll
    for (int tok = 0; tok < MT; ++tok) {
      if (tok >= m) break;
      uint64_t* p = &a.posted[((b + 1) * MT + tok) * 32 + lane];
      uint64_t w = ld_relaxed_u64(p);
      if (!__all_sync(0xffffffffu, (w & kPosted) != 0)) {
        const uint64_t t0 = globaltimer_ns();
        while ((w & kPosted) == 0) {
          w = ld_relaxed_u64(p);
          if ((w & kPosted) == 0 && globaltimer_ns() - t0 > kWaitLimitNs) break;
        }
        if (!__all_sync(0xffffffffu, (w & kPosted) != 0)) {
          if (lane == 0) atomicOr(a.err, 1u);
          return;
        }
      }
      sum[tok] += __uint_as_float(static_cast<uint32_t>(w));
      *p = 0ull;                                      // leave the workspace zero-filled
    }
  }
  for (int64_t c0 = b + 1; c_last > b + 1 && c0 <= c_last; c0 += kBatch) {
    uint64_t wb[kBatch][MT];
#pragma unroll
    for (int i = 0; i < kBatch; ++i)
#pragma unroll
      for (int tok = 0; tok < MT; ++tok)
        wb[i][tok] = (c0 + i <= c_last && tok < m) ? ld_relaxed_u64(&a.posted[((c0 + i) * MT + tok) * 32 + lane]) : 0ull;
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      const int64_t c = c0 + i;
      if (c > c_last) break;
#pragma unroll
      for (int tok = 0; tok < MT; ++tok) {
        if (tok >= m) break;
        uint64_t* p = &a.posted[(c * MT + tok) * 32 + lane];
        uint64_t w = wb[i][tok];
        if (!__all_sync(0xffffffffu, (w & kPosted) != 0)) {
          const uint64_t t0 = globaltimer_ns();
          while ((w & kPosted) == 0) {
            w = ld_relaxed_u64(p);
            if ((w & kPosted) == 0 && globaltimer_ns() - t0 > kWaitLimitNs) break;
          }
          if (!__all_sync(0xffffffffu, (w & kPosted) != 0)) {
            if (lane == 0) atomicOr(a.err, 1u);
            return;
          }
        }
        sum[tok] += __uint_as_float(static_cast<uint32_t>(w));
        *p = 0ull;                                    // leave the workspace zero-filled
      }
    }
  }
#pragma unroll
  for (int tok = 0; tok < MT; ++tok)
    if (tok < m) store_y(a, token_y(a, item.y, tok), tr * 32 + lane, sum[tok]);
}

// ------------------------------------------------------- chunk bodies ----

// q4 kinds.  The 32 x 256 codes are multiplied with x in exact integer
// arithmetic.  Per chunk and token, the warp writes each 32-column group of
// the bf16 x slice as 24-bit fixed point: v_k = x_k 2^(148 - E), E the biased
// exponent of the group's largest |x|, so |v_k| < 2^22.  This is exact when
// every nonzero x_k of the group lies within 2^14 of the largest (its lowest
// significant bit is then a multiple of the step 2^(E-148)) and 22 <= E <= 254.
// v_k + 0x808080 split into bytes gives three signed digits, v_k =
// d0 + 256 d1 + 65536 d2 with d_p in [-128, 127], kept as three byte planes
// packed four columns to a word in the order dp4a meets the codes: low
// nibbles (even k) and high nibbles (odd k) of a code word.  For each
// (row r, group g) and plane p the code dot product is an exact integer,
//   S_p = sum_k c_k d_p[k]  (dp4a, 4 codes per instruction, |S_p| <= 61440),
// and with X_p = sum_k d_p[k] and the plane weight q_p = 2^(E - 148 + 8p):
//   sum_k (c_k s + z) x_k = sum_p (s S_p q_p + z X_p q_p).
// S_p q_p and z X_p q_p are exact in binary32 (z has 8 significant bits for
// q4_1, |X_p| <= 4096), so each plane's partial s S_p q_p + z X_p q_p is
// rounded once (one fma), relative to its own exact value: there is no
// cancellation between the scale and the zero terms.  Q4_K's zero M*mn has up
// to 14 significant bits, so its z X_p q_p is split into a product and its
// exact error (the fma residue) and both are added.  Groups that do not fit
// (a range of magnitudes beyond 2^14, values below 2^-105, Inf or NaN) take
// the binary32 path instead for the whole chunk: w = fl(c s + z), then an fma
// per weight.
// A q4 chunk's share of one lane, read out of the ring stage at once so that
// the stage can be refilled before the arithmetic starts.  Prep lane
// (gp = lane & 7, tp = lane >> 3) reads the 8 columns gp*32 + 8tp .. +7 of
// each token's x slice (code word tp of group gp); decode lane (qr = lane >> 3,
// g = lane & 7) reads rows 4i + qr of group g: 16 code bytes and the group's
// scale fields per row.
template <int KIND, int MT>
struct Q4Lane {
  uint4 xr[MT];
  uint4 cw[8];
  uint32_t f0[8], f1[8];           // q4_1: scale, zero bf16 bits; Q4_K: the binary32 bits of S*sc, M*mn
};

// QTR: only quarter h's rows 8h + qr and 8h + 4 + qr, into entries 0 and 1.
template <int KIND, int MT, bool QTR = false>
__device__ __forceinline__ void q4_read(uint32_t st, uint32_t xs, bool with_x, int lane, int m, Q4Lane<KIND, MT>& L,
                                        int h = 0) {
  const int gp = lane & 7, tp = lane >> 3;
  if (with_x) {
#pragma unroll
    for (int tok = 0; tok < MT; ++tok)
      if (tok < m) L.xr[tok] = lds128(xs + tok * kXSliceBytes + gp * 64 + tp * 16);
  }
  const int qr = lane >> 3, g = lane & 7;
#pragma unroll
  for (int i = 0; i < (QTR ? 2 : 8); ++i) {
    const int r = QTR ? 8 * h + 4 * i + qr : 4 * i + qr;
    L.cw[i] = lds128(st + r * 128 + g * 16);
    if constexpr (KIND == kQ4_1) {
      L.f0[i] = lds_u16(st + kQ41Scale + (r * 8 + g) * 2);
      L.f1[i] = lds_u16(st + kQ41Zero + (r * 8 + g) * 2);
    } else {
      // the row's scale S*sc and min M*mn as binary32 bits (exact products:
      // 8 x 6 significant bits); sc, mn < 64 become binary32 through the bits
      // of 2^23 + v, less 2^23
      const float sc = __uint_as_float(0x4B000000u | lds_u8(st + kQ4KSc + r * 8 + g)) - 8388608.0f;
      const float mn = __uint_as_float(0x4B000000u | lds_u8(st + kQ4KMn + r * 8 + g)) - 8388608.0f;
      L.f0[i] = __float_as_uint(bf16_bits_to_f32(lds_u16(st + kQ4KS + r * 2)) * sc);
      L.f1[i] = __float_as_uint(bf16_bits_to_f32(lds_u16(st + kQ4KM + r * 2)) * mn);
    }
  }
}

// Scale and zero of row i of this lane's group.
template <int KIND, int MT>
__device__ __forceinline__ void q4_scale_zero(const Q4Lane<KIND, MT>& L, int i, float& s, float& z) {
  if constexpr (KIND == kQ4_1) {
    s = bf16_bits_to_f32(L.f0[i]);
    z = bf16_bits_to_f32(L.f1[i]);
  } else {                                         // formed when the stage was read
    s = __uint_as_float(L.f0[i]);
    z = __uint_as_float(L.f1[i]);
  }
}

// A quarter's two row sums into the lane's accumulators of rows 4(2h) + qr
// and 4(2h + 1) + qr (h is the same for the whole warp).
__device__ __forceinline__ void add_quarter(float (&y)[8], int h, float a, float b) {
  switch (h) {
    case 0: y[0] += a; y[1] += b; break;
    case 1: y[2] += a; y[3] += b; break;
    case 2: y[4] += a; y[5] += b; break;
    default: y[6] += a; y[7] += b; break;
  }
}

// 1.5 * 2^23 and its binary32 bits: for an integer |i| < 2^22 the bits
// kMagicBits + i are the binary32 number kMagic + i.
constexpr float kMagic = 12582912.0f;
constexpr int kMagicBits = 0x4B400000;

// One token's planes of this lane's group against two rows' codes: the
// per-plane partials added to (acc.x, acc.y).
template <int KIND, int NP>
__device__ __forceinline__ float2 q4_rows2(const uint32_t (&lo)[2][4], const uint32_t (&hi)[2][4], float2 s2,
                                           float2 z2, const uint4 (&PA)[4], const uint4 (&PB)[4], const XGroup& G,
                                           float2 acc) {
  // Each accumulator starts at the bits of 1.5 * 2^23, so that, with |S_p| <
  // 2^22, it ends as the binary32 number 1.5 * 2^23 + S_p exactly; one fma
  // with the plane weight then gives S_p q_p exactly (no int-to-float
  // conversion).
  int S[2][4];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    int a0 = kMagicBits, a1 = kMagicBits, a2 = kMagicBits, a3 = kMagicBits;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      a0 = dp4a_us(lo[r][t], PA[t].x, a0);
      a0 = dp4a_us(hi[r][t], PA[t].y, a0);
      a1 = dp4a_us(lo[r][t], PA[t].z, a1);
      a1 = dp4a_us(hi[r][t], PA[t].w, a1);
      a2 = dp4a_us(lo[r][t], PB[t].x, a2);
      a2 = dp4a_us(hi[r][t], PB[t].y, a2);
      if constexpr (NP == 4) {
        a3 = dp4a_us(lo[r][t], PB[t].z, a3);
        a3 = dp4a_us(hi[r][t], PB[t].w, a3);
      }
    }
    S[r][0] = a0;
    S[r][1] = a1;
    S[r][2] = a2;
    S[r][3] = a3;
  }
#pragma unroll
  for (int p = NP - 1; p >= 0; --p) {
    const float qp = G.q0 * static_cast<float>(1 << (8 * p));        // exact power of two
    const float2 qq = make_float2(qp, qp);
    const float2 mq = make_float2(-kMagic * qp, -kMagic * qp);
    const float2 xq = make_float2(G.xq[p], G.xq[p]);
    // exact: (1.5 * 2^23 + S_p) q_p - 1.5 * 2^23 q_p = S_p q_p, |S_p| < 2^22 times a power of two
    const float2 sq = ffma2(make_float2(__int_as_float(S[0][p]), __int_as_float(S[1][p])), qq, mq);
    if constexpr (KIND == kQ4_1) {
      const float2 zx = fmul2(z2, xq);                          // exact: 8 x 13 significant bits
      acc = fadd2(acc, ffma2(s2, sq, zx));
    } else {
      const float2 zx = fmul2(z2, xq);                          // rounded; its error added below
      const float2 ze = ffma2(z2, xq, make_float2(-zx.x, -zx.y));
      acc = fadd2(fadd2(acc, ffma2(s2, sq, zx)), ze);
    }
  }
  return acc;
}

// The exact-integer path for one chunk: rows 4i + qr of group g, every token,
// NP digit planes per token in `scratch` (token stride kScratchBytes, in a
// warp's scratch and in a slot of the x-slice cache alike).
template <int KIND, int MT, int NP, bool QTR = false>
__device__ __forceinline__ void q4_fixed(const Q4Lane<KIND, MT>& L, uint32_t scratch, int lane, int m,
                                         const XGroup (&G)[MT], float (&yacc)[MT][8], int h = 0) {
  const int g = lane & 7;
  auto load_planes = [&](int tok, uint4 (&PA)[4], uint4 (&PB)[4]) {
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      PA[t] = lds128(scratch + tok * kScratchBytes + (t * 8 + g) * 16);
      if constexpr (NP == 4) {
        PB[t] = lds128(scratch + tok * kScratchBytes + 512 + (t * 8 + g) * 16);
      } else {
        const uint2 b2 = lds64(scratch + tok * kScratchBytes + 512 + (t * 8 + g) * 16);
        PB[t] = make_uint4(b2.x, b2.y, 0u, 0u);
      }
    }
  };
  if constexpr (QTR) {
    // one quarter: its two rows (entries 0 and 1) are rows 4(2h) + qr and
    // 4(2h + 1) + qr of the chunk, accumulated in yacc[0][2h], yacc[0][2h + 1]
    static_assert(MT == 1, "quarters: one token");
    uint4 PA[4], PB[4];
    load_planes(0, PA, PB);
    float s[2], z[2];
    uint32_t lo[2][4], hi[2][4];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      q4_scale_zero(L, r, s[r], z[r]);
      const uint32_t w[4] = {L.cw[r].x, L.cw[r].y, L.cw[r].z, L.cw[r].w};
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        lo[r][t] = w[t] & 0x0F0F0F0Fu;
        hi[r][t] = (w[t] >> 4) & 0x0F0F0F0Fu;
      }
    }
    const float2 acc = q4_rows2<KIND, NP>(lo, hi, make_float2(s[0], s[1]), make_float2(z[0], z[1]), PA, PB, G[0],
                                          make_float2(0.f, 0.f));
    add_quarter(yacc[0], h, acc.x, acc.y);
  } else if constexpr (MT == 1) {
    uint4 PA[4], PB[4];
    load_planes(0, PA, PB);
#pragma unroll
    for (int i = 0; i < 8; i += 2) {                            // rows 4i + qr and 4(i+1) + qr, paired
      float s[2], z[2];
      uint32_t lo[2][4], hi[2][4];
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        q4_scale_zero(L, i + r, s[r], z[r]);
        const uint32_t w[4] = {L.cw[i + r].x, L.cw[i + r].y, L.cw[i + r].z, L.cw[i + r].w};
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          lo[r][t] = w[t] & 0x0F0F0F0Fu;
          hi[r][t] = (w[t] >> 4) & 0x0F0F0F0Fu;
        }
      }
      const float2 acc = q4_rows2<KIND, NP>(lo, hi, make_float2(s[0], s[1]), make_float2(z[0], z[1]), PA, PB, G[0],
                                            make_float2(yacc[0][i], yacc[0][i + 1]));
      yacc[0][i] = acc.x;
      yacc[0][i + 1] = acc.y;
    }
  } else {
    // several tokens: the codes are unpacked once for all rows, the planes
    // are read one token at a time
    uint32_t lo[4][2][4], hi[4][2][4];
    float2 s2[4], z2[4];
#pragma unroll
    for (int ip = 0; ip < 4; ++ip) {
      float s[2], z[2];
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        q4_scale_zero(L, 2 * ip + r, s[r], z[r]);
        const uint32_t w[4] = {L.cw[2 * ip + r].x, L.cw[2 * ip + r].y, L.cw[2 * ip + r].z, L.cw[2 * ip + r].w};
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          lo[ip][r][t] = w[t] & 0x0F0F0F0Fu;
          hi[ip][r][t] = (w[t] >> 4) & 0x0F0F0F0Fu;
        }
      }
      s2[ip] = make_float2(s[0], s[1]);
      z2[ip] = make_float2(z[0], z[1]);
    }
#pragma unroll
    for (int tok = 0; tok < MT; ++tok) {
      if (tok >= m) break;
      uint4 PA[4], PB[4];
      load_planes(tok, PA, PB);
#pragma unroll
      for (int ip = 0; ip < 4; ++ip) {
        const float2 acc = q4_rows2<KIND, NP>(lo[ip], hi[ip], s2[ip], z2[ip], PA, PB, G[tok],
                                              make_float2(yacc[tok][2 * ip], yacc[tok][2 * ip + 1]));
        yacc[tok][2 * ip] = acc.x;
        yacc[tok][2 * ip + 1] = acc.y;
      }
    }
  }
  __syncwarp();                                                 // scratch is rewritten by the next chunk
}

// The binary32 path for one chunk (x groups that 32-bit fixed point does not
// hold): every weight formed as fl(c s + z) and multiplied by x in an fma.
// The raw bf16 x slices are in region A of `scratch`, [t][g] 16 B.
template <int KIND, int MT, bool QTR = false>
__device__ __forceinline__ void q4_float(const Q4Lane<KIND, MT>& L, uint32_t scratch, int lane, int m,
                                         float (&yacc)[MT][8], int h = 0) {
  const int g = lane & 7;
  const float2 magic = make_float2(-8388608.0f, -8388608.0f);   // 2^23: float(2^23 + c) - 2^23 = c exactly
#pragma unroll 1
  for (int tok = 0; tok < m; ++tok) {
    float2 xf[16];                                              // columns 2j, 2j + 1 of group g
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const uint4 xw = lds128(scratch + tok * kScratchBytes + (t * 8 + g) * 16);
      const uint32_t w[4] = {xw.x, xw.y, xw.z, xw.w};
#pragma unroll
      for (int b = 0; b < 4; ++b)
        xf[4 * t + b] = make_float2(__uint_as_float(w[b] << 16), __uint_as_float(w[b] & 0xFFFF0000u));
    }
    float part[8];
#pragma unroll
    for (int i = 0; i < (QTR ? 2 : 8); ++i) {
      float s, z;
      q4_scale_zero(L, i, s, z);
      const float2 s2 = make_float2(s, s), z2 = make_float2(z, z);
      const uint32_t w[4] = {L.cw[i].x, L.cw[i].y, L.cw[i].z, L.cw[i].w};
      float2 acc = make_float2(0.f, 0.f);
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const uint32_t lo = w[t] & 0x0F0F0F0Fu, hi = (w[t] >> 4) & 0x0F0F0F0Fu;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          const float2 c = fadd2(make_float2(__uint_as_float(prmt(lo, 0x4B000000u, 0x7540 + b)),
                                             __uint_as_float(prmt(hi, 0x4B000000u, 0x7540 + b))), magic);
          acc = ffma2(ffma2(c, s2, z2), xf[4 * t + b], acc);
        }
      }
      part[i] = acc.x + acc.y;
    }
    // (tok is a loop variable: select the token's accumulators by comparison,
    // so that they stay in registers)
    if constexpr (QTR) {
      add_quarter(yacc[0], h, part[0], part[1]);
    } else {
#pragma unroll
      for (int u = 0; u < MT; ++u)
        if (u == tok)
#pragma unroll
          for (int i = 0; i < 8; ++i) yacc[u][i] += part[i];
    }
  }
  __syncwarp();                                                 // scratch is rewritten by the next chunk
}

// One chunk's x, prepared by the warp: each token's slice becomes digit
// planes in the warp's scratch (3 or 4 planes, the most any token's groups
// need), or, when some group spans more than 32-bit fixed point holds, the
// raw slices go to the scratch for the binary32 path.  Returns that mode (3,
// 4 or 5); the caller syncs the warp before the scratch is read.
template <int KIND, int MT>
__device__ __forceinline__ int q4_prep(const Q4Lane<KIND, MT>& L, uint32_t scratch, int lane, int m,
                                       XGroup (&G)[MT]) {
  int E[MT];
  int need = 3;
#pragma unroll
  for (int tok = 0; tok < MT; ++tok)
    if (tok < m) need = max(need, q4_x_need(L.xr[tok], E[tok]));
  need = __reduce_max_sync(0xffffffffu, need);
  if (need == 3) {
#pragma unroll
    for (int tok = 0; tok < MT; ++tok)
      if (tok < m) q4_x_planes<3>(L.xr[tok], E[tok], scratch + tok * kScratchBytes, lane, G[tok]);
  } else if (need == 4) {
#pragma unroll
    for (int tok = 0; tok < MT; ++tok)
      if (tok < m) q4_x_planes<4>(L.xr[tok], E[tok], scratch + tok * kScratchBytes, lane, G[tok]);
  } else {
    const int gp = lane & 7, tp = lane >> 3;
#pragma unroll
    for (int tok = 0; tok < MT; ++tok)
      if (tok < m)
        asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(scratch + tok * kScratchBytes + (tp * 8 + gp) * 16),
                     "r"(L.xr[tok].x), "r"(L.xr[tok].y), "r"(L.xr[tok].z), "r"(L.xr[tok].w)
                     : "memory");
  }
  return need;
}

// One chunk's arithmetic, its x prepared in `src` (the warp's scratch or a
// cache slot) in the given mode (uniform over the warp).
template <int KIND, int MT, bool QTR = false>
__device__ __forceinline__ void q4_math(const Q4Lane<KIND, MT>& L, uint32_t src, int lane, int m, int mode,
                                        const XGroup (&G)[MT], float (&yacc)[MT][8], int h = 0) {
  if (mode == 3) q4_fixed<KIND, MT, 3, QTR>(L, src, lane, m, G, yacc, h);
  else if (mode == 4) q4_fixed<KIND, MT, 4, QTR>(L, src, lane, m, G, yacc, h);
  else q4_float<KIND, MT, QTR>(L, src, lane, m, yacc, h);
}

// Q8: lane covers rows 8*qe + (0..7) of columns 8t + kc, t = 0..31.
template <int KIND>
__device__ __forceinline__ void q8_lane_map(int lane, int& qe, int& kc) {
  if constexpr (KIND == kQ8_KR) { qe = lane & 3; kc = lane >> 2; }
  else { qe = ((lane >> 4) << 1) | (lane & 1); kc = (lane >> 1) & 7; }
}

template <int KIND, int MT>
__device__ __forceinline__ void q8_chunk(uint32_t st, uint32_t xs, int lane, int m, float (&yacc)[MT][8]) {
  int qe, kc;
  q8_lane_map<KIND>(lane, qe, kc);
  const float MAGIC = 8388736.0f;   // 2^23 + 128: float(2^23 + (c ^ 0x80)) - MAGIC == c exactly
  const float2 nm = make_float2(-MAGIC, -MAGIC);
  const uint32_t B = 0x4B000000u;
  uint4 drow[8];                    // d of the lane's 8 rows, all 8 groups (16 bytes per row)
#pragma unroll
  for (int i = 0; i < 8; ++i) drow[i] = lds128(st + kQ8D + (qe * 8 + i) * 16);
#pragma unroll
  for (int g = 0; g < 8; ++g) {
    float2 acc[MT][4];
#pragma unroll
    for (int tok = 0; tok < MT; ++tok)
#pragma unroll
      for (int u = 0; u < 4; ++u) acc[tok][u] = make_float2(0.f, 0.f);
#pragma unroll
    for (int tt = 0; tt < 4; ++tt) {
      const int kk = 8 * tt + kc;                 // column within the group
      uint32_t off;
      if constexpr (KIND == kQ8_KR) off = (g * 32 + kk) * 32 + qe * 8;
      else off = (qe >> 1) * 4096 + g * 512 + kk * 16 + (qe & 1) * 8;
      const uint2 cw = lds64(st + off);
      const uint32_t w0 = cw.x ^ 0x80808080u, w1 = cw.y ^ 0x80808080u;
      float2 c01 = fadd2(make_float2(__uint_as_float(prmt(w0, B, 0x7540)), __uint_as_float(prmt(w0, B, 0x7541))), nm);
      float2 c23 = fadd2(make_float2(__uint_as_float(prmt(w0, B, 0x7542)), __uint_as_float(prmt(w0, B, 0x7543))), nm);
      float2 c45 = fadd2(make_float2(__uint_as_float(prmt(w1, B, 0x7540)), __uint_as_float(prmt(w1, B, 0x7541))), nm);
      float2 c67 = fadd2(make_float2(__uint_as_float(prmt(w1, B, 0x7542)), __uint_as_float(prmt(w1, B, 0x7543))), nm);
#pragma unroll
      for (int tok = 0; tok < MT; ++tok) {
        if (tok >= m) break;
        const float xk = bf16_bits_to_f32(lds_u16(xs + tok * kXSliceBytes + (g * 32 + kk) * 2));
        const float2 xx = make_float2(xk, xk);
        acc[tok][0] = ffma2(c01, xx, acc[tok][0]);
        acc[tok][1] = ffma2(c23, xx, acc[tok][1]);
        acc[tok][2] = ffma2(c45, xx, acc[tok][2]);
        acc[tok][3] = ffma2(c67, xx, acc[tok][3]);
      }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t wd = (g >> 1) == 0 ? drow[i].x : (g >> 1) == 1 ? drow[i].y : (g >> 1) == 2 ? drow[i].z : drow[i].w;
      const float d = __uint_as_float((g & 1) ? (wd & 0xFFFF0000u) : (wd << 16));
#pragma unroll
      for (int tok = 0; tok < MT; ++tok) {
        const float part = (i & 1) ? acc[tok][i >> 1].y : acc[tok][i >> 1].x;
        yacc[tok][i] = fmaf(d, part, yacc[tok][i]);
      }
    }
  }
}

template <int KIND>
__device__ __forceinline__ float finish_rows(float (&yacc)[8], int lane, int& row) {
  if constexpr (KIND == kQ4_1 || KIND == kQ4_K) {
    row = 4 * (lane & 7) + (lane >> 3);
    return transpose_reduce8(yacc, lane, 4, 2, 1);
  } else {
    int qe, kc;
    q8_lane_map<KIND>(lane, qe, kc);
    row = qe * 8 + kc;
    return (KIND == kQ8_KR) ? transpose_reduce8(yacc, lane, 16, 8, 4) : transpose_reduce8(yacc, lane, 8, 4, 2);
  }
}

// --------------------------------------------------------------- kernel ----

// ----------------------------------------------------- segment results ----

// End of a segment (item it, tile row tr) of warp w (range [lo, hi)); each
// lane holds, per token, the sum of the row `row`.  A row held by this warp
// alone is stored at once.  A row shared with other warps of the CTA is parked
// in the warp's slot (0: its first segment, 1: its last); the last of those
// warps to arrive (shared-memory counter of the row's first warp) adds the
// slots in warp order and stores y, or hands the row on to cross_cta_row when
// other CTAs share it too.
template <int MT, class GemvArgs>
__device__ __noinline__ void finish_segment(const GemvArgs& a, int64_t b, int w, int nw, int it, int64_t tr, int row,
                                            const float (&val)[MT], float* slots, uint32_t* cnt, int lane) {
  const GemvItemDev& item = a.items[it];
  const int m = (MT == 1) ? 1 : a.m;
  const int64_t Lc = s_range[0], Hc = s_range[1];
  const int64_t lo = Lc + s_wlo[w], hi = Lc + s_wlo[w + 1];      // this warp's range
  const int64_t r0 = item.cbase + tr * item.TC, r1 = r0 + item.TC;
  if (lo <= r0 && r1 <= hi) {
#pragma unroll
    for (int tok = 0; tok < MT; ++tok)
      if (tok < m) store_y(a, token_y(a, item.y, tok), tr * 32 + row, val[tok]);
    return;
  }
  const int k = (r0 <= lo) ? 0 : 1;                 // the warp's first segment iff the row holds lo
#pragma unroll
  for (int tok = 0; tok < MT; ++tok) slots[((w * 2 + k) * MT + tok) * 32 + row] = val[tok];
  // first and last warp holding part of the row: the warps whose ranges start
  // at or before the row's first and last chunk in this CTA, counted by ballot
  const uint32_t wlo = lane < nw ? s_wlo[lane] : 0xFFFFFFFFu;
  const int wa = __popc(__ballot_sync(0xffffffffu, wlo <= static_cast<uint32_t>((r0 > Lc ? r0 : Lc) - Lc))) - 1;
  const int wb = __popc(__ballot_sync(0xffffffffu, wlo <= static_cast<uint32_t>((r1 < Hc ? r1 : Hc) - 1 - Lc))) - 1;
  const int64_t lo_a = Lc + __shfl_sync(0xffffffffu, wlo, wa);
  const int ka = (r0 <= lo_a) ? 0 : 1;             // the row's slot in its first warp
  __threadfence_block();
  __syncwarp();
  uint32_t old = 0;
  if (lane == 0) old = atomicAdd(&cnt[wa * 2 + ka], 1u);
  old = __shfl_sync(0xffffffffu, old, 0);
  if (old != static_cast<uint32_t>(wb - wa)) return;   // another warp of the CTA finishes the row
  __threadfence_block();
  float sum[MT];
#pragma unroll
  for (int tok = 0; tok < MT; ++tok) {
    sum[tok] = slots[((wa * 2 + ka) * MT + tok) * 32 + lane];
    for (int v = wa + 1; v <= wb; ++v) sum[tok] += slots[((v * 2) * MT + tok) * 32 + lane];
  }
  if (r0 >= Lc && r1 <= Hc) {
#pragma unroll
    for (int tok = 0; tok < MT; ++tok)
      if (tok < m) store_y(a, token_y(a, item.y, tok), tr * 32 + lane, sum[tok]);
  } else {
    cross_cta_row<MT>(a, b, Lc, it, tr, r0, r1, sum, lane);
  }
}

// A stage's copies complete on its barrier: the chunk, plus `xbytes` of x
// slices (0 when the CTA's x-slice cache serves the chunk).
// QTR: only quarter p.h of the chunk (its 8 rows' codes and scale fields),
// each piece at its place in the stage.
template <int KIND, int MT, bool QTR, class GemvArgs>
__device__ __forceinline__ void issue_chunk(const GemvArgs& a, const Pos& p, uint32_t xbytes, uint8_t* dst,
                                            uint64_t* bar) {
  constexpr int CB = chunk_bytes_of(KIND);
  if constexpr (QTR) {
    const int h = p.h;
    if constexpr (KIND == kQ4_1) {
      mbar_arrive_expect_tx(bar, 1024 + 2 * 128 + xbytes);
      bulk_g2s(dst + 1024 * h, p.w + 1024 * h, 1024, bar);                       // codes of rows 8h .. 8h+7
      bulk_g2s(dst + kQ41Scale + 128 * h, p.w + kQ41Scale + 128 * h, 128, bar);  // their scales
      bulk_g2s(dst + kQ41Zero + 128 * h, p.w + kQ41Zero + 128 * h, 128, bar);    // their zeros
    } else {
      mbar_arrive_expect_tx(bar, 1024 + 2 * 64 + 2 * 16 + xbytes);
      bulk_g2s(dst + 1024 * h, p.w + 1024 * h, 1024, bar);
      bulk_g2s(dst + kQ4KSc + 64 * h, p.w + kQ4KSc + 64 * h, 64, bar);
      bulk_g2s(dst + kQ4KMn + 64 * h, p.w + kQ4KMn + 64 * h, 64, bar);
      bulk_g2s(dst + kQ4KS + 16 * h, p.w + kQ4KS + 16 * h, 16, bar);
      bulk_g2s(dst + kQ4KM + 16 * h, p.w + kQ4KM + 16 * h, 16, bar);
    }
  } else {
    mbar_arrive_expect_tx(bar, CB + xbytes);
    bulk_g2s(dst, p.w, CB, bar);
  }
}
template <int KIND, int MT, class GemvArgs>
__device__ __forceinline__ void issue_xslice(const GemvArgs& a, const Pos& p, int m, uint8_t* dst, uint64_t* bar) {
  const uint8_t* x = p.x;
#pragma unroll
  for (int tok = 0; tok < MT; ++tok)
    if (tok < m) bulk_g2s(dst + tok * kXSliceBytes, x + tok * a.x_stride, kXSliceBytes, bar);
}

// The cache slot of the chunk at position p (the CTA caches x slices).
__device__ __forceinline__ int xslot_of(const Pos& p) {
  const int4 e = s_xtab[p.it - s_xinfo[1]];
  int d = p.tc - e.y;
  if (d < 0) d += e.w;
  return e.x + d;
}

// Threads per CTA the kernel is compiled for.  One token: at most 128
// registers, so that two CTAs of 8 warps share an SM (consecutive launches
// overlap).  Several tokens: 8 warps with the register budget of a lone CTA
// (two warps per SM sub-partition: up to 255 registers; three would cap them
// at 168, below what the tokens' digit planes and unpacked codes need).
template <int KIND, int MT>
constexpr int gemv_max_threads() {
  return MT == 1 ? 512 : 256;
}

// QTR: the index space counts quarters of chunks (a small launch spreads each
// chunk's rows over four warps, so that one warp's arithmetic on one chunk is
// not the launch's critical path).
// XCT: the x-slice cache's code is compiled in (always for one token; for
// several, only into the launches planned to use it -- its branch alone costs
// those that do not up to 17 %).
template <int KIND, int MAXB, int MT, bool QTR = false, bool XCT = true>
__global__ void __launch_bounds__(gemv_max_threads<KIND, MT>(), 1) gemv_kernel(const __grid_constant__ GemvArgsT<MAXB> a) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int CB = chunk_bytes_of(KIND);                         // a ring stage holds one chunk
  constexpr bool Q4 = (KIND == kQ4_1 || KIND == kQ4_K);
  constexpr bool XC = Q4 && !QTR && XCT;                           // may use the x-slice cache
  static_assert(!QTR || (Q4 && MT == 1), "quarters: 4-bit kinds, one token");
  asm volatile("griddepcontrol.launch_dependents;");
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const int m = (MT == 1) ? 1 : a.m;
  const int64_t b = blockIdx.x;
  const int64_t Lc = (a.T * b) / a.grid, Hc = (a.T * (b + 1)) / a.grid;
  const int64_t lo = Lc + ((Hc - Lc) * warp) / nwarps, hi = Lc + ((Hc - Lc) * (warp + 1)) / nwarps;
  const int stages = a.stages;
  // shared memory: ring [warps][stages] chunks | barriers | row slots | counters |
  // x slices [warps][stages][MT] | per-warp scratch [warps][MT], or the x-slice cache
  const uint64_t ring_bytes = static_cast<uint64_t>(nwarps) * stages * CB;
  uint8_t* ring = smem + static_cast<uint64_t>(warp) * stages * CB;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + ring_bytes) + warp * stages;
  uint8_t* p8 = smem + ring_bytes + align16(static_cast<uint64_t>(nwarps) * stages * 8);
  float* slots = reinterpret_cast<float*>(p8);                                   // [nwarps][2][MT][32]
  uint32_t* cnt = reinterpret_cast<uint32_t*>(slots + nwarps * 2 * MT * 32);     // [nwarps][2]
  uint8_t* tail = reinterpret_cast<uint8_t*>(cnt) + align16(static_cast<uint64_t>(nwarps) * 8);
  uint8_t* xsl = tail + static_cast<uint64_t>(warp) * stages * MT * kXSliceBytes;
  const uint32_t tail2 = smem_u32(tail) + nwarps * stages * MT * kXSliceBytes;
  const uint32_t scratch = tail2 + warp * MT * kScratchBytes;
  const uint32_t xcache = tail2;
  const int n = static_cast<int>(hi - lo);                     // chunks of this warp (>= 1)

  Pos cur{}, pre{};                         // chunk being processed / next chunk to fetch
  cur.seek<CB, QTR>(a, lo);
  pre = cur;
  if (lane == 0) {
    for (int s = 0; s < stages; ++s) mbar_init(&bars[s], 1);
    fence_barrier_init();
    // weights never change between launches: fetch the first chunks before
    // waiting on the previous grid; their x slices follow after the wait
    Pos p = pre;
    for (int s = 0; s < stages && s < n; ++s) {
      issue_chunk<KIND, MT, QTR>(a, p, static_cast<uint32_t>(m * kXSliceBytes), ring + s * CB, &bars[s]);
      p.next<CB, QTR>(a);
    }
  }
  if (XC && a.xslots > 0 && threadIdx.x == 32 * (nwarps - 1)) {
    // which (item, tile column) slices the CTA's chunks touch; the cache is
    // used when they fit and each is reused four times on average (below
    // that, filling it costs the short launches more than it saves)
    Pos p0{}, p1{};
    p0.seek<CB, QTR>(a, Lc);
    p1.seek<CB, QTR>(a, Hc - 1);
    int ok = p1.it - p0.it < kXTabItems, total = 0;
    for (int it = p0.it; ok && it <= p1.it; ++it) {
      const GemvItemDev& I = a.items[it];
      const int64_t ca = (Lc > I.cbase ? Lc : I.cbase) - I.cbase;
      const int64_t ce = (Hc < I.cbase + I.nchunks ? Hc : I.cbase + I.nchunks) - I.cbase;
      const bool whole = ce - ca >= I.TC;
      const int ns = whole ? I.TC : static_cast<int>(ce - ca);
      s_xtab[it - p0.it] = make_int4(total, whole ? 0 : static_cast<int>(ca % I.TC), ns, I.TC);
      total += ns;
      ok = total <= a.xslots;
    }
    // (reused at least 4 times for one token; more than twice for several,
    // whose preparation per chunk costs several times more.  Measured on
    // GB300: a reuse of exactly 2 -- Q4_K 9728x2560 against 2 tokens -- lost
    // 4 % to the fill's barrier, 2.5 -- q4_1 12288x4096 -- gained 7 %)
    s_xinfo[0] = ok && (MT == 1 ? Hc - Lc >= 4 * static_cast<int64_t>(total)
                                : Hc - Lc > 2 * static_cast<int64_t>(total));
    s_xinfo[1] = p0.it;
    s_xinfo[2] = total;
    s_xinfo[3] = p1.it - p0.it + 1;
  }
  if (warp == 0 && lane <= nwarps) s_wlo[lane] = static_cast<uint32_t>(((Hc - Lc) * lane) / nwarps);
  if (threadIdx.x == 0) {
    s_range[0] = Lc;
    s_range[1] = Hc;
  }
  if (threadIdx.x == blockDim.x - 1) {
    Pos e{};
    e.seek<CB, QTR>(a, Hc - 1);
    const int64_t r1 = a.items[e.it].cbase + (static_cast<int64_t>(e.tr) + 1) * a.items[e.it].TC;
    s_clast = r1 > Hc ? cta_of(r1 - 1, a.T, a.grid) : b;
  }
  if (lane < 2) cnt[warp * 2 + lane] = 0u;
  if (threadIdx.x == 0) s_top1_key = 0ull;
  __syncwarp();
  // the row counters are zero and the tables written before any warp can
  // count; done before the wait, so that no CTA-wide barrier follows it
  // (except the one after the x-slice cache is filled)
  __syncthreads();
  const bool xc = XC && a.xslots > 0 && s_xinfo[0] != 0;      // this CTA's x slices come from the cache
  const uint32_t xbytes = xc ? 0u : static_cast<uint32_t>(m * kXSliceBytes);   // x bytes with each refill
  asm volatile("griddepcontrol.wait;" ::: "memory");            // x, y and the workspace may be the previous grid's
  // the x slices of the chunks already in flight (unused when the cache
  // serves them); every lane walks `pre`, so that it stays warp-uniform
  for (int s = 0; s < stages && s < n; ++s) {
    if (lane == 0) issue_xslice<KIND, MT>(a, pre, m, xsl + s * MT * kXSliceBytes, &bars[s]);
    pre.next<CB, QTR>(a);
  }
  if (xc) {
    // fill the cache: warp w prepares slices w, w + nwarps, ...; each lane
    // loads its 16 bytes of up to four slices before preparing any
    const int nsl = s_xinfo[2], it0 = s_xinfo[1], nti = s_xinfo[3];
    const int gp = lane & 7, tp = lane >> 3;
    constexpr int kU = MT == 1 ? 4 : 1;              // slices loaded before any is prepared
    for (int s0 = warp; s0 < nsl; s0 += kU * nwarps) {
      uint4 xr[kU][MT];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int sl = s0 + u * nwarps;
        if (sl < nsl) {
          int k = 0;                                  // the touched item holding slot sl
          while (k + 1 < nti && s_xtab[k + 1].x <= sl) ++k;
          const int4 e = s_xtab[k];
          int tc = e.y + (sl - e.x);
          if (tc >= e.w) tc -= e.w;
          const uint8_t* xs0 = a.items[it0 + k].x + static_cast<int64_t>(tc) * kXSliceBytes + gp * 64 + tp * 16;
#pragma unroll
          for (int tok = 0; tok < MT; ++tok)
            if (MT == 1 || tok < m) xr[u][tok] = ld_cg_u4(xs0 + tok * a.x_stride);
        }
      }
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int sl = s0 + u * nwarps;
        if (sl < nsl) xslot_fill<MT>(xr[u], xcache + sl * (MT * kXSlotBytes), m, lane);
      }
    }
    __syncthreads();
  }

  float yacc[MT][8];
#pragma unroll
  for (int tok = 0; tok < MT; ++tok)
#pragma unroll
    for (int i = 0; i < 8; ++i) yacc[tok][i] = 0.f;
  int seg_it = cur.it, seg_tr = cur.tr;
  uint32_t phase = 0;                       // bit s: parity awaited next on stage s
  int s = 0;
  bool failed = false;

  for (int j = 0; j < n; ++j) {
    const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&bars[s], (phase >> s) & 1u));
    if (!ok) { failed = true; break; }
    phase ^= 1u << s;
    if (cur.it != seg_it || cur.tr != seg_tr) {    // the previous segment is complete
      int row;
      float v[MT];
#pragma unroll
      for (int tok = 0; tok < MT; ++tok) v[tok] = finish_rows<KIND>(yacc[tok], lane, row);
      finish_segment<MT>(a, b, warp, nwarps, seg_it, seg_tr, row, v, slots, cnt, lane);
#pragma unroll
      for (int tok = 0; tok < MT; ++tok)
#pragma unroll
        for (int i = 0; i < 8; ++i) yacc[tok][i] = 0.f;
      seg_it = cur.it;
      seg_tr = cur.tr;
    }
    const uint32_t st = smem_u32(ring + s * CB);
    const uint32_t xs = smem_u32(xsl + s * MT * kXSliceBytes);
    // 4-bit chunks: the lanes take their share of the stage into registers,
    // find or prepare the chunk's x (which covers the loads' latency), and
    // the stage is refilled before the arithmetic; Q8: after it
    Q4Lane<Q4 ? KIND : kQ4_1, MT> q4l;
    XGroup G[MT];
    int mode = 0;
    uint32_t src = scratch;
    if constexpr (Q4) {
      q4_read<KIND, MT, QTR>(st, xs, !xc, lane, m, q4l, cur.h);
      if (XC && xc) {
        src = xcache + xslot_of(cur) * (MT * kXSlotBytes);
#pragma unroll
        for (int tok = 0; tok < MT; ++tok) {
          if (MT > 1 && tok >= m) break;
          const uint32_t gr = src + MT * kScratchBytes + tok * kXRecBytes + (lane & 7) * 32;
          const uint4 g0 = lds128(gr), g1 = lds128(gr + 16);
          G[tok].q0 = __uint_as_float(g0.x);
          G[tok].xq[0] = __uint_as_float(g0.y);
          G[tok].xq[1] = __uint_as_float(g0.z);
          G[tok].xq[2] = __uint_as_float(g0.w);
          G[tok].xq[3] = __uint_as_float(g1.x);
          mode = static_cast<int>(g1.y);                        // the slice's mode: uniform over its tokens
        }
      } else {
        mode = q4_prep<KIND, MT>(q4l, scratch, lane, m, G);
      }
    } else {
      q8_chunk<KIND, MT>(st, xs, lane, m, yacc);
    }
    // every lane's reads of the stage are done before it is refilled, and
    // the prepared planes are visible to the warp
    __syncwarp();
    if (j + stages < n) {
      if (lane == 0) {
        issue_chunk<KIND, MT, QTR>(a, pre, xbytes, ring + s * CB, &bars[s]);
        if (!xc) issue_xslice<KIND, MT>(a, pre, m, xsl + s * MT * kXSliceBytes, &bars[s]);
      }
      pre.next<CB, QTR>(a);
    }
    if constexpr (Q4) q4_math<KIND, MT, QTR>(q4l, src, lane, m, mode, G, yacc, cur.h);
    cur.next<CB, QTR>(a);
    if (++s == stages) s = 0;
  }
  if (failed) {
    // A wait gave up: record it and let this warp's copies in flight land.
    if (lane == 0) atomicOr(a.err, 1u);
    for (int t = 0; t < stages; ++t) mbar_wait_bounded(&bars[t], (phase >> t) & 1u, 100000000ull);
  } else {
    int row;
    float v[MT];
#pragma unroll
    for (int tok = 0; tok < MT; ++tok) v[tok] = finish_rows<KIND>(yacc[tok], lane, row);
    finish_segment<MT>(a, b, warp, nwarps, seg_it, seg_tr, row, v, slots, cnt, lane);
  }
  if (MT == 1 && a.top1) {
    // every warp's rows are folded in; the CTA's key goes to the launch's key,
    // and the last CTA to finish writes the index and clears the two words
    __syncthreads();
    if (threadIdx.x == 0) {
      const unsigned long long k = s_top1_key;
      if (k != 0ull) atomicMax(reinterpret_cast<unsigned long long*>(a.top1_key), k);
      // the count is an acquire-release atomic: it orders this CTA's max
      // before its count, and the CTA that counts last sees every CTA's max
      // (two full fences here cost 0.3-0.5 us at the end of the launch)
      uint32_t done;
      asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(done) : "l"(a.top1_done) : "memory");
      if (done == static_cast<uint32_t>(a.grid - 1)) {
        const unsigned long long best = atomicExch(reinterpret_cast<unsigned long long*>(a.top1_key), 0ull);
        if (a.top1_idx) *a.top1_idx = argmax_index(best);
        if (a.top1_key_out) *a.top1_key_out = static_cast<int64_t>(best ^ (1ull << 63));
        *a.top1_done = 0u;
      }
    }
  }
}

// ----------------------------------------------------------------- host ----

// Chunks per SM from which a 4-bit single-token launch runs two CTAs per SM.
constexpr int kTwoCtaChunksPerSm = 128;
// Chunks per SM up to which a 4-bit single-token launch takes quarters of
// chunks as its units.
constexpr int kQuarterChunksPerSm = 8;

static int gemv_max_warps(int kind, int MT) {
  (void)kind;
  (void)MT;
  return 8;
}

bool gemv_plan(int kind, int64_t T, const DeviceInfo& info, GemvPlan* p, int MT, int64_t tc) {
  const int CB = chunk_bytes_of(kind);
  if (CB == 0 || info.sms <= 0 || T <= 0 || MT < 1) return false;
  // ring, barriers, row slots, counters and the per-warp x slices; then the
  // per-warp scratch, or (4-bit kinds) the x-slice cache
  auto base = [&](int w, int st) {
    return static_cast<uint64_t>(w) * st * CB + align16(static_cast<uint64_t>(w) * st * 8) +
           static_cast<uint64_t>(w) * MT * kSlotBytes + align16(static_cast<uint64_t>(w) * kCntBytes) +
           static_cast<uint64_t>(w) * st * MT * kXSliceBytes;
  };
  auto need = [&](int w, int st) { return base(w, st) + static_cast<uint64_t>(w) * MT * kScratchBytes; };
  p->quarter = 0;
  if ((kind == kQ4_1 || kind == kQ4_K) && MT == 1 && T <= static_cast<int64_t>(kQuarterChunksPerSm) * info.sms) {
    // A small one-token 4-bit launch (at most kQuarterChunksPerSm chunks per
    // SM) is latency-bound: a warp's arithmetic on one chunk lies on its
    // critical path.  Its units are quarters of chunks (8 rows each), up to
    // 16 warps per CTA over CTAs of at least 4 chunks, one CTA per SM.
    const uint64_t qcap = static_cast<uint64_t>(info.max_smem_optin) - 512;
    int w = kMaxGemvWarps;
    while (w > 1 && need(w, 2) > qcap) w /= 2;
    if (need(w, 2) > qcap) return false;
    int64_t grid = T / 4;
    if (grid < 1) grid = 1;
    if (grid > info.sms) grid = info.sms;
    if (grid > kMaxCtas) grid = kMaxCtas;
    const int64_t per_cta = 4 * T / grid;          // quarters per CTA; every warp gets at least one
    if (per_cta < w) w = static_cast<int>(per_cta);
    p->warps = w;
    p->stages = 2;
    p->grid = static_cast<int>(grid);
    p->smem = need(w, 2);
    p->xslots = 0;
    p->quarter = 1;
    return true;
  }
  // Eight warps per CTA, each streaming a longer run of chunks, measured best
  // on GB300 against 12 and 16.  4-bit chunks: the CTA stays within half an
  // SM's shared memory, so that the next launch in the stream (programmatic
  // dependent launch) starts its weight copies on the same SMs while this one
  // drains -- back-to-back GEMVs then overlap their start-up latency.  Q8
  // chunks are larger and gain more from a deeper ring than from that overlap.
  // (less 512 bytes for the kernel's static shared memory, 384 bytes today:
  // two CTAs of a two-per-SM launch should both fit.  That is for speed, not
  // for progress: a finisher waits only on higher-indexed CTAs, which post
  // after their first tile row, so in-order dispatch suffices)
  // Several tokens need more registers than two CTAs per SM leave, so those
  // launches take the whole of the shared memory.
  const uint64_t cap =
      static_cast<uint64_t>(CB <= kQ41Bytes && MT == 1 ? info.smem_two_per_sm : info.max_smem_optin) - 512;
  const int max_warps = gemv_max_warps(kind, MT);
  static const int kWarpChoices[] = {12, 8, 6, 4, 2, 1};
  static_assert(12 <= kMaxGemvWarps, "warp table");
  int warps = 0, stages = 0;
  for (int w : kWarpChoices) {
    if (w > max_warps) continue;
    for (int st = 4; st >= 2; --st) {
      if (need(w, st) <= cap) { warps = w; stages = st; break; }
    }
    if (warps) break;
  }
  if (!warps) return false;
  // One CTA per SM; small problems use fewer CTAs of at least ~4 chunks each so
  // that split tile rows are combined inside a CTA rather than across CTAs.
  // Large 4-bit launches (at least kTwoCtaChunksPerSm chunks per SM, ~100 MB)
  // take both half-SM slots of every SM themselves: twice the copies in flight
  // while they stream.  Measured on GB300, back to back: the 196-matrix decode
  // step and a 151936x2560 weight 2.3-2.5 % faster.  The price is paid by the
  // launch after it, which can start its first copies only as this one's CTAs
  // exit: a 4096x12288 GEMV behind a 24576x4096 one (81 chunks per SM) lost
  // 2.3 us that way, more than the 0.5 us the larger launch gained, so
  // launches of that size keep one CTA per SM and leave the second slot to the
  // next launch (below ~60 chunks per SM two CTAs are slower even back to back:
  // 12288x4096 8.4 -> 9.0 us).
  const bool two_per_sm = CB <= kQ41Bytes && MT == 1 && T >= static_cast<int64_t>(kTwoCtaChunksPerSm) * info.sms;
  int64_t grid = T / 4;
  if (grid < 1) grid = 1;
  if (grid > (two_per_sm ? 2 : 1) * static_cast<int64_t>(info.sms)) grid = (two_per_sm ? 2 : 1) * static_cast<int64_t>(info.sms);
  if (grid > kMaxCtas) grid = kMaxCtas;
  const int64_t per_cta = T / grid;                // every warp gets at least one chunk
  if (per_cta < warps) warps = static_cast<int>(per_cta);
  p->warps = warps;
  p->stages = stages;
  p->grid = static_cast<int>(grid);
  p->smem = need(warps, stages);
  p->xslots = 0;
  if ((kind == kQ4_1 || kind == kQ4_K) && MT == 1 && cap > base(warps, stages)) {
    // the x-slice cache takes what the budget leaves: 17 slots in half an SM
    const uint64_t room = (cap - base(warps, stages)) / kXSlotBytes;
    p->xslots = static_cast<int>(room < static_cast<uint64_t>(kMaxXSlots) ? room : kMaxXSlots);
    const uint64_t with_cache = base(warps, stages) + static_cast<uint64_t>(p->xslots) * kXSlotBytes;
    if (with_cache > p->smem) p->smem = with_cache;
  } else if ((kind == kQ4_1 || kind == kQ4_K) && MT > 1 && tc > 0 && tc <= kMaxXSlots &&
             (T + grid - 1) / grid > 2 * tc) {
    // Several tokens (one weight of tc tile columns): a CTA of L chunks
    // touches min(L, tc) slices and caches them when L > 2 tc (the kernel's
    // own test).  Each slice takes MT slots' worth; the ring gives up its
    // fourth stage when the tc slices would not fit beside it, since
    // preparing every token's planes once per chunk costs more than the
    // shallower ring.
    const uint64_t per = static_cast<uint64_t>(MT) * kXSlotBytes;
    auto slots = [&](int st) { return cap > base(warps, st) ? (cap - base(warps, st)) / per : uint64_t{0}; };
    int st = stages;
    if (st > 3 && slots(st) < static_cast<uint64_t>(tc)) --st;
    if (slots(st) >= static_cast<uint64_t>(tc)) {
      const uint64_t room = slots(st);
      p->xslots = static_cast<int>(room < static_cast<uint64_t>(kMaxXSlots) ? room : kMaxXSlots);
      p->stages = st;
      p->smem = need(warps, st);
      const uint64_t with_cache = base(warps, st) + static_cast<uint64_t>(p->xslots) * per;
      if (with_cache > p->smem) p->smem = with_cache;
    }
  }
  return true;
}

uint64_t gemv_workspace_bytes(int64_t total_tile_rows, int64_t total_chunks, int MT) {
  (void)total_chunks;
  (void)total_tile_rows;
  return kWsErrBytes + static_cast<uint64_t>(kMaxCtas) * MT * 32 * 8;
}

template <int KIND, int MAXB, int MT, bool QTR = false, bool XCT = true>
static cudaError_t launch_gemv_t(const GemvArgsT<MAXB>& a, const GemvPlan& p, cudaStream_t s) {
  cudaError_t e = set_max_dynamic_smem(reinterpret_cast<const void*>(gemv_kernel<KIND, MAXB, MT, QTR, XCT>));
  if (e != cudaSuccess) return e;
  // Programmatic dependent launch: SMs freed by the previous grid start this
  // one at once; the kernel waits for the previous grid before touching x, y
  // or the workspace.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.grid);
  cfg.blockDim = dim3(p.warps * 32);
  cfg.dynamicSmemBytes = p.smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, gemv_kernel<KIND, MAXB, MT, QTR, XCT>, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// The item table in units: chunks, or (unit = 4) quarters of chunks.
template <int MAXB>
static void fill_items(GemvArgsT<MAXB>& a, const GemvItem* items, int n, int unit = 1) {
  int64_t T = 0;
  for (int i = 0; i < n; ++i) {
    a.items[i].chunks = static_cast<const uint8_t*>(items[i].chunks);
    a.items[i].x = static_cast<const uint8_t*>(items[i].x);
    a.items[i].y = items[i].y;
    a.items[i].cbase = T;
    a.items[i].nchunks = items[i].TR * items[i].TC * unit;
    a.items[i].TC = static_cast<int32_t>(items[i].TC * unit);
    T += items[i].TR * items[i].TC * unit;
  }
  a.nitems = n;
  a.T = T;
}

// One-token launch of a planned GEMV (item table already in the plan's units).
template <int MAXB>
static cudaError_t launch_one_token(int kind, const GemvArgsT<MAXB>& a, const GemvPlan& p, cudaStream_t s) {
  if (p.quarter) {
    switch (kind) {
      case kQ4_1: return launch_gemv_t<kQ4_1, MAXB, 1, true>(a, p, s);
      case kQ4_K: return launch_gemv_t<kQ4_K, MAXB, 1, true>(a, p, s);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (kind) {
    case kQ4_1: return launch_gemv_t<kQ4_1, MAXB, 1>(a, p, s);
    case kQ4_K: return launch_gemv_t<kQ4_K, MAXB, 1>(a, p, s);
    case kQ8_KR: return launch_gemv_t<kQ8_KR, MAXB, 1>(a, p, s);
    case kQ8_BLK: return launch_gemv_t<kQ8_BLK, MAXB, 1>(a, p, s);
    default: return cudaErrorInvalidValue;
  }
}

template <int MAXB>
static void fill_workspace(GemvArgsT<MAXB>& a, void* workspace) {
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  a.err = reinterpret_cast<uint32_t*>(ws);
  a.top1_done = reinterpret_cast<uint32_t*>(ws + 4);
  a.top1_key = reinterpret_cast<uint64_t*>(ws + 8);
  a.posted = reinterpret_cast<uint64_t*>(ws + kWsErrBytes);
}

struct Top1Out {
  int32_t* idx = nullptr;
  int64_t* key = nullptr;
  uint32_t row_base = 0;
};

template <int MAXB>
static cudaError_t launch_gemv_sized(int kind, const GemvItem* items, int n, int out_f32, void* workspace,
                                     const DeviceInfo& info, const Top1Out* top1, cudaStream_t s) {
  GemvArgsT<MAXB> a;
  fill_items(a, items, n);
  a.out_f32 = out_f32;
  a.m = 1;
  a.x_stride = 0;
  a.y_stride = 0;
  a.top1 = top1 != nullptr;
  a.top1_idx = top1 ? top1->idx : nullptr;
  a.top1_key_out = top1 ? top1->key : nullptr;
  a.top1_row_base = top1 ? top1->row_base : 0u;
  GemvPlan p;
  if (!gemv_plan(kind, a.T, info, &p, 1)) return cudaErrorInvalidValue;
  if (p.quarter) fill_items(a, items, n, 4);
  fill_workspace(a, workspace);
  a.grid = p.grid;
  a.stages = p.stages;
  a.xslots = p.xslots;
  a.out_f32 = out_f32;
  a.m = 1;
  a.x_stride = 0;
  a.y_stride = 0;
  a.top1 = top1 != nullptr;
  a.top1_idx = top1 ? top1->idx : nullptr;
  a.top1_key_out = top1 ? top1->key : nullptr;
  a.top1_row_base = top1 ? top1->row_base : 0u;
  return launch_one_token<MAXB>(kind, a, p, s);
}

cudaError_t launch_gemv_batch(int kind, const GemvItem* items, int n, int out_f32, void* workspace,
                              const DeviceInfo& info, cudaStream_t s) {
  if (n < 1 || n > kMaxBatch) return cudaErrorInvalidValue;
  if (n == 1) return launch_gemv_sized<1>(kind, items, n, out_f32, workspace, info, nullptr, s);
  if (n <= 8) return launch_gemv_sized<8>(kind, items, n, out_f32, workspace, info, nullptr, s);
  return launch_gemv_sized<kMaxBatch>(kind, items, n, out_f32, workspace, info, nullptr, s);
}

cudaError_t launch_gemv_top1(int kind, const GemvItem& item, int32_t* idx, int64_t* key, uint32_t row_base,
                             void* workspace, const DeviceInfo& info, cudaStream_t s) {
  Top1Out t;
  t.idx = idx;
  t.key = key;
  t.row_base = row_base;
  return launch_gemv_sized<1>(kind, &item, 1, 1, workspace, info, &t, s);
}

int gemv_max_tokens(int kind) {
  switch (kind) {
    case kQ4_1: return kGemvTokensQ41;
    case kQ4_K: return kGemvTokensQ4K;
    case kQ8_KR:
    case kQ8_BLK: return kGemvTokensQ8;
    default: return 0;
  }
}

cudaError_t launch_gemv_tokens(int kind, const GemvItem& item, int M, int out_f32, uint32_t* err, void* workspace,
                               const DeviceInfo& info, cudaStream_t s) {
  if (M < 1 || M > gemv_max_tokens(kind)) return cudaErrorInvalidValue;
  const int MT = M == 1 ? 1 : M == 2 ? 2 : 4;
  GemvArgsT<1> a;
  fill_items(a, &item, 1);
  GemvPlan p;
  if (!gemv_plan(kind, a.T, info, &p, MT, item.TC)) return cudaErrorInvalidValue;
  fill_workspace(a, workspace);
  a.err = err;
  a.grid = p.grid;
  a.stages = p.stages;
  a.xslots = p.xslots;
  a.out_f32 = out_f32;
  a.m = M;
  a.x_stride = item.TC * 256 * 2;                 // X rows: cols bf16 each
  a.y_stride = item.TR * 32;                      // Y rows: rows elements each
  a.top1 = 0;
  a.top1_idx = nullptr;
  a.top1_key_out = nullptr;
  a.top1_row_base = 0u;
  if (MT == 1) {                                  // one token: the single-GEMV kernel itself
    if (p.quarter) fill_items(a, &item, 1, 4);
    return launch_one_token<1>(kind, a, p, s);
  }
  const bool xc = p.xslots > 0;
  if (MT == 2) {
    switch (kind) {
      case kQ4_1: return xc ? launch_gemv_t<kQ4_1, 1, 2, false, true>(a, p, s) : launch_gemv_t<kQ4_1, 1, 2, false, false>(a, p, s);
      case kQ4_K: return xc ? launch_gemv_t<kQ4_K, 1, 2, false, true>(a, p, s) : launch_gemv_t<kQ4_K, 1, 2, false, false>(a, p, s);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (kind) {
    case kQ4_1: return xc ? launch_gemv_t<kQ4_1, 1, 4, false, true>(a, p, s) : launch_gemv_t<kQ4_1, 1, 4, false, false>(a, p, s);
    case kQ4_K: return xc ? launch_gemv_t<kQ4_K, 1, 4, false, true>(a, p, s) : launch_gemv_t<kQ4_K, 1, 4, false, false>(a, p, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace q4nx
