// q4nx_gemv.cu -- fused decode + GEMV (one token) over Q4NX chunks, sm_103a.
//
// y[n] = sum_k w[n][k] x[k], weights in the chunk kinds of the "Q4NX chunks"
// section of the 1bit engine "NPU engine" page (chunk-kind table: q4_1
// code*scale+zero, Q4_K S*scale*code+M*min, Q8 d*code in layout KR or BLK).
// One launch runs a batch of independent GEMVs of one chunk kind (a single
// GEMV is a batch of one).
//
// Design (HBM-bound: 0.625 B/weight for q4_1, so the instruction budget is
// about three per weight at full bandwidth):
//  * Persistent grid, one CTA per SM.  The chunks of all items form one index
//    space (item after item, each row-major over its tile grid); every warp is
//    an independent worker owning a contiguous range of it, balanced to within
//    one chunk.  A range is a run of (item, tile row) segments.
//  * Each worker streams its chunks with 1-D bulk async copies (TMA
//    cp.async.bulk) into its own ring of shared-memory stages: the chunk and
//    the 512-byte bf16 slice of x for the chunk's tile column, completing on
//    one mbarrier per stage.  Every wait is bounded.  No CTA-wide barrier.
//  * 4-bit kinds: lane (q = lane>>3, g = lane&7) reads the 16-byte run of 32
//    codes of group g in row 4i+q (a 512-byte conflict-free LDS.128 per warp
//    and i).  Codes become floats with one shift-or-LOP3 each: a nibble moved
//    to bit 15 (even k) or 19 (odd k) of 0x3F800000 is 1 + c*2^-8 or
//    1 + c*2^-4, so with packed FFMA2 over (even, odd) column pairs
//        acc_e = X_e + 2^-8 sum_even c x,   acc_o = X_o + 2^-4 sum_odd c x
//    (X_e, X_o the group's sums of x), and the scale and zero factor out:
//        y_r += s_rg * ((acc_e - X_e) 2^8 + (acc_o - X_o) 2^4) + z_rg (X_e + X_o).
//  * Q8 kinds: lane reads 8 rows x 1 column (LDS.64, conflict-free for both
//    layouts); codes become exact floats through the 2^23 magic number; d_rg
//    scales each lane's (row, group) partial.
//  * Row sums are finished with a warp transpose-reduce.  A tile row split
//    between workers is finished by the last worker to arrive (arrival
//    counter per tile row in the workspace), which adds the partials in
//    worker order, clears them, and resets the counter: results do not depend
//    on timing and the workspace is left zero-filled.
#include "q4nx_device.cuh"
#include "q4nx_kernels.h"

namespace q4nx {

constexpr int kXSliceBytes = 512;            // bf16 x of one tile column
constexpr int kMaxBatch = kMaxGemvItems;

struct GemvItemDev {
  const uint8_t* chunks;
  const uint8_t* x;        // bf16 [K]
  void* y;                 // [N]
  int64_t cbase;           // first chunk of this item in the batch index space
  int64_t nchunks;         // TR * TC
  int32_t TC;
  int32_t trbase;          // first tile row of this item in the batch's counter array
};

// Kernel parameters; MAXB batch slots (instantiated for 1, 8 and 256 items so
// that small launches do not carry a 12 KB parameter block).
template <int MAXB>
struct GemvArgsT {
  GemvItemDev items[MAXB];
  int nitems;
  int workers;
  int stages;
  int out_f32;
  int64_t T;               // chunks in the batch
  uint32_t* err;
  uint32_t* counters;      // [sum TR]
  float* partials;         // [workers][2][32]
};

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

// worker that holds chunk c: the largest w with floor(T*w/W) <= c
__device__ __forceinline__ int64_t worker_of(int64_t c, int64_t T, int64_t W) { return ((c + 1) * W - 1) / T; }

template <class GemvArgs>
__device__ __forceinline__ void store_y(const GemvArgs& a, void* y, int64_t n, float v) {
  if (a.out_f32) static_cast<float*>(y)[n] = v;
  else static_cast<uint16_t*>(y)[n] = f32_to_bf16_bits(v);
}

// Finish the segment (item it, tile row tr) of worker wk, whose range starts
// at lo: `val` is the lane's sum for row `row` of the tile row.
template <class GemvArgs>
__device__ __noinline__ void flush_segment(const GemvArgs& a, int64_t wk, int64_t lo, int64_t hi, int it, int64_t tr,
                                           int row, float val, int lane) {
  const GemvItemDev& item = a.items[it];
  const int64_t row_lo = item.cbase + tr * item.TC, row_hi = row_lo + item.TC;
  const int64_t n = tr * 32 + row;
  if (lo <= row_lo && row_hi <= hi) {               // the whole tile row is ours
    store_y(a, item.y, n, val);
    return;
  }
  const int slot = (lo >= row_lo) ? 0 : 1;          // a worker's first segment uses slot 0
  a.partials[(wk * 2 + slot) * 32 + row] = val;
  __threadfence();
  __syncwarp();
  const int64_t w_first = worker_of(row_lo, a.T, a.workers);
  const int64_t w_last = worker_of(row_hi - 1, a.T, a.workers);
  uint32_t* counter = &a.counters[item.trbase + tr];
  uint32_t old = 0;
  if (lane == 0) old = atomicAdd(counter, 1u);
  old = __shfl_sync(0xffffffffu, old, 0);
  if (old != static_cast<uint32_t>(w_last - w_first)) return;   // not the last to arrive
  __threadfence();
  float sum = 0.f;
  for (int64_t w = w_first; w <= w_last; ++w) {
    const int64_t wlo = (a.T * w) / a.workers;
    float* p = &a.partials[(w * 2 + ((wlo >= row_lo) ? 0 : 1)) * 32 + row];
    sum += ld_cg_f32(p);
    *p = 0.f;                                       // leave the workspace zero-filled
  }
  store_y(a, item.y, n, sum);
  __syncwarp();
  if (lane == 0) *counter = 0u;
}

// ------------------------------------------------------- chunk bodies ----

// q4: sum over one 16-byte run (32 codes of group g, one row) of v * x with
// v = 1 + c 2^-8 (even k) / 1 + c 2^-4 (odd k); xv are (even, odd) x pairs.
__device__ __forceinline__ float2 q4_run(uint4 cw, const float2 (&xv)[16]) {
  const uint32_t w[4] = {cw.x, cw.y, cw.z, cw.w};
  const uint32_t ONE = 0x3F800000u;
  float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const uint32_t a = w[t] << 15, b = w[t] << 7, c = w[t] >> 1, d = w[t] >> 9;
    const float2 v0 = make_float2(__uint_as_float(lop3_and_or(a, 0x00078000u, ONE)),
                                  __uint_as_float(lop3_and_or(a, 0x00780000u, ONE)));
    const float2 v1 = make_float2(__uint_as_float(lop3_and_or(b, 0x00078000u, ONE)),
                                  __uint_as_float(lop3_and_or(b, 0x00780000u, ONE)));
    const float2 v2 = make_float2(__uint_as_float(lop3_and_or(c, 0x00078000u, ONE)),
                                  __uint_as_float(lop3_and_or(c, 0x00780000u, ONE)));
    const float2 v3 = make_float2(__uint_as_float(lop3_and_or(d, 0x00078000u, ONE)),
                                  __uint_as_float(lop3_and_or(d, 0x00780000u, ONE)));
    acc0 = ffma2(v0, xv[4 * t + 0], acc0);
    acc1 = ffma2(v1, xv[4 * t + 1], acc1);
    acc0 = ffma2(v2, xv[4 * t + 2], acc0);
    acc1 = ffma2(v3, xv[4 * t + 3], acc1);
  }
  return fadd2(acc0, acc1);
}

template <int KIND>
__device__ __forceinline__ void q4_chunk(uint32_t st, int lane, float (&yacc)[8]) {
  constexpr int CB = chunk_bytes_of(KIND);
  const int q = lane >> 3, g = lane & 7;
  // x of group g: 32 bf16 = 16 (even, odd) pairs
  float2 xv[16];
  float2 xs = make_float2(0.f, 0.f);
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const uint4 xr = lds128(st + CB + g * 64 + u * 16);
    const uint32_t xw[4] = {xr.x, xr.y, xr.z, xr.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      xv[4 * u + j] = make_float2(__uint_as_float(xw[j] << 16), __uint_as_float(xw[j] & 0xFFFF0000u));
      xs = fadd2(xs, xv[4 * u + j]);
    }
  }
  const float xsum = xs.x + xs.y;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = 4 * i + q;
    const uint4 cw = lds128(st + r * 128 + g * 16);
    float s, z;
    if constexpr (KIND == kQ4_1) {
      s = bf16_bits_to_f32(lds_u16(st + kQ41Scale + (r * 8 + g) * 2));
      z = bf16_bits_to_f32(lds_u16(st + kQ41Zero + (r * 8 + g) * 2));
    } else {
      const float S = bf16_bits_to_f32(lds_u16(st + kQ4KS + r * 2));
      const float M = bf16_bits_to_f32(lds_u16(st + kQ4KM + r * 2));
      s = S * static_cast<float>(lds_u8(st + kQ4KSc + r * 8 + g));
      z = M * static_cast<float>(lds_u8(st + kQ4KMn + r * 8 + g));
    }
    const float2 acc = q4_run(cw, xv);
    const float dot = fmaf(acc.x - xs.x, 256.f, (acc.y - xs.y) * 16.f);
    yacc[i] = fmaf(s, dot, fmaf(z, xsum, yacc[i]));
  }
}

// Q8: lane covers rows 8*qe + (0..7) of columns 8t + kc, t = 0..31.
template <int KIND>
__device__ __forceinline__ void q8_lane_map(int lane, int& qe, int& kc) {
  if constexpr (KIND == kQ8_KR) { qe = lane & 3; kc = lane >> 2; }
  else { qe = ((lane >> 4) << 1) | (lane & 1); kc = (lane >> 1) & 7; }
}

template <int KIND>
__device__ __forceinline__ void q8_chunk(uint32_t st, int lane, float (&yacc)[8]) {
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
    float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
    for (int tt = 0; tt < 4; ++tt) {
      const int kk = 8 * tt + kc;                 // column within the group
      uint32_t off;
      if constexpr (KIND == kQ8_KR) off = (g * 32 + kk) * 32 + qe * 8;
      else off = (qe >> 1) * 4096 + g * 512 + kk * 16 + (qe & 1) * 8;
      const uint2 cw = lds64(st + off);
      const float xk = bf16_bits_to_f32(lds_u16(st + kQ8Bytes + (g * 32 + kk) * 2));
      const float2 xx = make_float2(xk, xk);
      const uint32_t w0 = cw.x ^ 0x80808080u, w1 = cw.y ^ 0x80808080u;
      float2 c01 = fadd2(make_float2(__uint_as_float(prmt(w0, B, 0x7540)), __uint_as_float(prmt(w0, B, 0x7541))), nm);
      float2 c23 = fadd2(make_float2(__uint_as_float(prmt(w0, B, 0x7542)), __uint_as_float(prmt(w0, B, 0x7543))), nm);
      float2 c45 = fadd2(make_float2(__uint_as_float(prmt(w1, B, 0x7540)), __uint_as_float(prmt(w1, B, 0x7541))), nm);
      float2 c67 = fadd2(make_float2(__uint_as_float(prmt(w1, B, 0x7542)), __uint_as_float(prmt(w1, B, 0x7543))), nm);
      acc[0] = ffma2(c01, xx, acc[0]);
      acc[1] = ffma2(c23, xx, acc[1]);
      acc[2] = ffma2(c45, xx, acc[2]);
      acc[3] = ffma2(c67, xx, acc[3]);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t wd = (g >> 1) == 0 ? drow[i].x : (g >> 1) == 1 ? drow[i].y : (g >> 1) == 2 ? drow[i].z : drow[i].w;
      const float d = __uint_as_float((g & 1) ? (wd & 0xFFFF0000u) : (wd << 16));
      const float part = (i & 1) ? acc[i >> 1].y : acc[i >> 1].x;
      yacc[i] = fmaf(d, part, yacc[i]);
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

// Position of a chunk in the batch: item, index inside the item, tile row and
// column.  Workers walk their ranges in order, so positions advance by one
// without divisions.
struct Pos {
  int it;
  int32_t tr, tc;
  int64_t local;
  template <class GemvArgs>
  __device__ __forceinline__ void seek(const GemvArgs& a, int64_t c) {
    int lo = 0, hi = a.nitems - 1;                  // last item with cbase <= c
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (a.items[mid].cbase <= c) lo = mid; else hi = mid - 1;
    }
    it = lo;
    local = c - a.items[it].cbase;
    tr = static_cast<int32_t>(local / a.items[it].TC);
    tc = static_cast<int32_t>(local - static_cast<int64_t>(tr) * a.items[it].TC);
  }
  template <class GemvArgs>
  __device__ __forceinline__ void next(const GemvArgs& a) {
    ++local;
    if (++tc == a.items[it].TC) { tc = 0; ++tr; }
    if (local == a.items[it].nchunks && it + 1 < a.nitems) { ++it; local = 0; tr = 0; tc = 0; }
  }
};

template <int KIND, class GemvArgs>
__device__ __forceinline__ void issue_stage(const GemvArgs& a, const Pos& p, uint8_t* dst, uint64_t* bar) {
  constexpr int CB = chunk_bytes_of(KIND);
  const GemvItemDev& item = a.items[p.it];
  mbar_arrive_expect_tx(bar, CB + kXSliceBytes);
  bulk_g2s(dst, item.chunks + p.local * CB, CB, bar);
  bulk_g2s(dst + CB, item.x + static_cast<int64_t>(p.tc) * kXSliceBytes, kXSliceBytes, bar);
}

template <int KIND, int MAXB>
__global__ void __launch_bounds__(512, 1) gemv_kernel(const __grid_constant__ GemvArgsT<MAXB> a) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int SB = chunk_bytes_of(KIND) + kXSliceBytes;     // stage bytes
  constexpr bool Q4 = (KIND == kQ4_1 || KIND == kQ4_K);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const int64_t wk = static_cast<int64_t>(blockIdx.x) * nwarps + warp;
  if (wk >= a.workers) return;                                 // idle warp of the last CTA
  const int64_t lo = (a.T * wk) / a.workers, hi = (a.T * (wk + 1)) / a.workers;
  const int stages = a.stages;
  uint8_t* ring = smem + static_cast<uint64_t>(warp) * stages * SB;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + static_cast<uint64_t>(nwarps) * stages * SB) + warp * stages;
  const int n = static_cast<int>(hi - lo);                     // chunks of this worker

  Pos cur, pre;                             // chunk being processed / next chunk to fetch
  cur.seek(a, lo);
  pre = cur;
  if (lane == 0) {
    for (int s = 0; s < stages; ++s) mbar_init(&bars[s], 1);
    fence_barrier_init();
    for (int s = 0; s < stages && s < n; ++s) {
      issue_stage<KIND>(a, pre, ring + s * SB, &bars[s]);
      pre.next(a);
    }
  }
  __syncwarp();

  float yacc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) yacc[i] = 0.f;
  int seg_it = cur.it, seg_tr = cur.tr;
  uint32_t phase = 0;                       // bit s: parity awaited next on stage s
  int s = 0;

  for (int j = 0; j < n; ++j) {
    const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&bars[s], (phase >> s) & 1u));
    if (!ok) {
      // A wait gave up: record it, let this worker's copies in flight land, stop.
      if (lane == 0) atomicOr(a.err, 1u);
      for (int t = 0; t < stages; ++t) mbar_wait_bounded(&bars[t], (phase >> t) & 1u, 100000000ull);
      return;
    }
    phase ^= 1u << s;
    if (cur.it != seg_it || cur.tr != seg_tr) {    // the previous segment is complete
      int row;
      const float v = finish_rows<KIND>(yacc, lane, row);
      flush_segment(a, wk, lo, hi, seg_it, seg_tr, row, v, lane);
#pragma unroll
      for (int i = 0; i < 8; ++i) yacc[i] = 0.f;
      seg_it = cur.it;
      seg_tr = cur.tr;
    }
    const uint32_t st = smem_u32(ring + s * SB);
    if constexpr (Q4) q4_chunk<KIND>(st, lane, yacc);
    else q8_chunk<KIND>(st, lane, yacc);
    __syncwarp();
    if (lane == 0 && j + stages < n) {
      issue_stage<KIND>(a, pre, ring + s * SB, &bars[s]);
      pre.next(a);
    }
    cur.next(a);
    if (++s == stages) s = 0;
  }
  int row;
  const float v = finish_rows<KIND>(yacc, lane, row);
  flush_segment(a, wk, lo, hi, seg_it, seg_tr, row, v, lane);
}

// ----------------------------------------------------------------- host ----

bool gemv_plan(int kind, int64_t T, int sms, int max_smem, GemvPlan* p) {
  const int CB = chunk_bytes_of(kind);
  if (CB == 0 || sms <= 0 || T <= 0) return false;
  const uint64_t SB = static_cast<uint64_t>(CB) + kXSliceBytes;
  static const int kWarpChoices[] = {16, 12, 8, 6, 4, 2, 1};
  int warps = 0, stages = 0;
  for (int w : kWarpChoices) {
    const uint64_t need = static_cast<uint64_t>(w) * 2 * (SB + 8);
    if (need <= static_cast<uint64_t>(max_smem)) { warps = w; stages = 2; break; }
  }
  if (!warps) return false;
  if (static_cast<uint64_t>(warps) * 3 * (SB + 8) <= static_cast<uint64_t>(max_smem)) stages = 3;
  // Small problems: spread chunks over SMs before stacking warps.
  const int64_t per_sm = (T + sms - 1) / sms;
  if (per_sm < warps) warps = static_cast<int>(per_sm < 1 ? 1 : per_sm);
  int64_t grid = (T + warps - 1) / warps;
  if (grid > sms) grid = sms;
  int64_t workers = grid * warps;
  if (workers > T) workers = T;                    // every worker gets at least one chunk
  if (workers > kMaxWorkers) workers = kMaxWorkers;
  grid = (workers + warps - 1) / warps;
  p->warps = warps;
  p->stages = stages;
  p->grid = static_cast<int>(grid);
  p->workers = static_cast<int>(workers);
  p->smem = static_cast<uint64_t>(warps) * stages * (SB + 8);
  return true;
}

uint64_t gemv_workspace_bytes(int64_t total_tile_rows, int64_t total_chunks) {
  const int64_t w = total_chunks < kMaxWorkers ? total_chunks : kMaxWorkers;
  return kWsErrBytes + align16(static_cast<uint64_t>(total_tile_rows) * 4) + static_cast<uint64_t>(w) * 2 * 32 * 4;
}

template <int KIND, int MAXB>
static cudaError_t launch_gemv_t(const GemvArgsT<MAXB>& a, const GemvPlan& p, cudaStream_t s) {
  const int slot = KIND + (MAXB == 1 ? 0 : MAXB == 8 ? 4 : 8);
  cudaError_t e = set_max_dynamic_smem(reinterpret_cast<const void*>(gemv_kernel<KIND, MAXB>), slot);
  if (e != cudaSuccess) return e;
  gemv_kernel<KIND, MAXB><<<p.grid, p.warps * 32, p.smem, s>>>(a);
  return cudaGetLastError();
}

template <int MAXB>
static cudaError_t launch_gemv_sized(int kind, const GemvItem* items, int n, int out_f32, void* workspace, int sms,
                                     int max_smem, cudaStream_t s) {
  GemvArgsT<MAXB> a;
  int64_t T = 0, TRsum = 0;
  for (int i = 0; i < n; ++i) {
    a.items[i].chunks = static_cast<const uint8_t*>(items[i].chunks);
    a.items[i].x = static_cast<const uint8_t*>(items[i].x);
    a.items[i].y = items[i].y;
    a.items[i].cbase = T;
    a.items[i].nchunks = items[i].TR * items[i].TC;
    a.items[i].TC = static_cast<int32_t>(items[i].TC);
    a.items[i].trbase = static_cast<int32_t>(TRsum);
    T += items[i].TR * items[i].TC;
    TRsum += items[i].TR;
  }
  GemvPlan p;
  if (!gemv_plan(kind, T, sms, max_smem, &p)) return cudaErrorInvalidValue;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  a.nitems = n;
  a.workers = p.workers;
  a.stages = p.stages;
  a.out_f32 = out_f32;
  a.T = T;
  a.err = reinterpret_cast<uint32_t*>(ws);
  a.counters = reinterpret_cast<uint32_t*>(ws + kWsErrBytes);
  a.partials = reinterpret_cast<float*>(ws + kWsErrBytes + align16(static_cast<uint64_t>(TRsum) * 4));
  switch (kind) {
    case kQ4_1: return launch_gemv_t<kQ4_1, MAXB>(a, p, s);
    case kQ4_K: return launch_gemv_t<kQ4_K, MAXB>(a, p, s);
    case kQ8_KR: return launch_gemv_t<kQ8_KR, MAXB>(a, p, s);
    case kQ8_BLK: return launch_gemv_t<kQ8_BLK, MAXB>(a, p, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_gemv_batch(int kind, const GemvItem* items, int n, int out_f32, void* workspace, int sms,
                              int max_smem, cudaStream_t s) {
  if (n < 1 || n > kMaxBatch) return cudaErrorInvalidValue;
  if (n == 1) return launch_gemv_sized<1>(kind, items, n, out_f32, workspace, sms, max_smem, s);
  if (n <= 8) return launch_gemv_sized<8>(kind, items, n, out_f32, workspace, sms, max_smem, s);
  return launch_gemv_sized<kMaxBatch>(kind, items, n, out_f32, workspace, sms, max_smem, s);
}

}  // namespace q4nx
