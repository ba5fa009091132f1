/*
 * q4nx_oracle.c -- the ORACLE: plain, slow, single-threaded CPU statement of
 * what the Q4NX dequant-GEMV/GEMM path computes.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link or
 * call this file; only the test suite, the smoke check and the CPU-baseline leg
 * of the benchmark do.  It shares no code, header, table or constant with the
 * CUDA library: every offset below is written out here again from the format
 * description.
 *
 * Source of the format: the 1bit engine's "NPU engine" page (docs/npu.md),
 * section "Q4NX chunks" (chunk-kind table and the two Q8 code layouts) and the
 * paragraph after it (decoders, Q4_K -> q4_1 repack and its rounding bound).
 *
 * A weight W[N][K] is a grid of 32-row x 256-column tiles, one chunk per tile,
 * chunks stored row-major over the grid: chunk (tr, tc) starts at byte
 * (tr * (K/256) + tc) * chunk_bytes.
 *
 * The page does not print the byte order inside a chunk.  This file uses the
 * reading fixed for the whole build (every reading is listed in the design
 * notes; parity of this byte order is UNPINNED, because no page shows it):
 *
 *   q4_1  (5120 B)  [codes 4096][scale bf16 [32 r][8 g]][zero bf16 [32 r][8 g]]
 *   Q4_K  (4736 B)  [codes 4096][sc u8 [32][8]][mn u8 [32][8]][S bf16 [32]][M bf16 [32]]
 *   Q8    (8704 B)  [codes int8 8192 in layout KR or BLK][d bf16 [32 r][8 g]]
 *
 *   4-bit code (r, k) sits in byte r*128 + k/2: low nibble for even k,
 *   high nibble for odd k.  g = k/32 is the 32-column group.
 *   Q8 layout KR : code (r, k) at byte k*32 + r                      (page, verbatim)
 *   Q8 layout BLK: (r/16)*4096 + (k/32)*512 + (k%32)*16 + r%16        (page, verbatim)
 *   bf16 fields are little-endian.
 *
 * Weight formulas (page, chunk-kind table):
 *   q4_1: w = code * scale + zero
 *   Q4_K: w = S * scale * code + M * min        (sign of the min term as printed)
 *   Q8  : w = d * code
 *
 * Compile with -O2 -ffp-contract=off: the fp32 decode below must round after
 * every single operation, exactly as written.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

enum { ORC_Q4_1 = 1, ORC_Q4_K = 2, ORC_Q8_KR = 3, ORC_Q8_BLK = 4 };

/* chunk-kind table of the "Q4NX chunks" section */
int64_t oracle_chunk_bytes(int kind)
{
    switch (kind) {
    case ORC_Q4_1: return 5120;
    case ORC_Q4_K: return 4736;
    case ORC_Q8_KR:
    case ORC_Q8_BLK: return 8704;
    default: return 0;
    }
}

/* ---------------------------------------------------------------- bf16 --- */

/* bf16 is the upper half of an IEEE binary32 pattern. */
float oracle_bf16_to_f32(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round a binary32 to the nearest bf16, ties to even (IEEE 754 default
 * rounding applied to an 8-bit significand).  NaN maps to the quiet NaN
 * 0x7FC0 (payload and sign are not part of the contract). */
uint16_t oracle_f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0)
        return 0x7FC0;
    uint32_t low = u & 0xFFFFu;           /* the 16 bits that are dropped */
    uint32_t up = u >> 16;
    if (low > 0x8000u || (low == 0x8000u && (up & 1u)))
        up += 1;                          /* carries into the exponent as needed */
    return (uint16_t)up;
}

static uint16_t rd16(const uint8_t* p) { return (uint16_t)(p[0] | (p[1] << 8)); }

/* ------------------------------------------------------- field readers --- */

static const uint8_t* chunk_at(const uint8_t* base, int kind, int64_t K, int64_t tr, int64_t tc)
{
    int64_t tiles_per_row = K / 256;
    return base + (tr * tiles_per_row + tc) * oracle_chunk_bytes(kind);
}

/* 4-bit code (r, k) of a q4_1 or Q4_K chunk */
static int code4(const uint8_t* ch, int r, int k)
{
    uint8_t b = ch[r * 128 + k / 2];
    return (k % 2 == 0) ? (b & 0x0F) : (b >> 4);
}

/* int8 code (r, k) of a Q8 chunk, in the layout the caller states */
static int code8(const uint8_t* ch, int kind, int r, int k)
{
    int64_t off;
    if (kind == ORC_Q8_KR)
        off = (int64_t)k * 32 + r;
    else
        off = (int64_t)(r / 16) * 4096 + (k / 32) * 512 + (k % 32) * 16 + r % 16;
    return (int)(int8_t)ch[off];
}

/* All fields that determine weight (r, k) of one chunk. */
typedef struct {
    int code;
    float scale, zero;          /* q4_1 */
    int sc, mn;                 /* Q4_K u8 scale and min */
    float S, M;                 /* Q4_K per-row bf16 */
    float d;                    /* Q8 */
} fields_t;

static fields_t read_fields(const uint8_t* ch, int kind, int r, int k)
{
    fields_t f;
    memset(&f, 0, sizeof f);
    int g = k / 32;
    switch (kind) {
    case ORC_Q4_1:
        f.code = code4(ch, r, k);
        f.scale = oracle_bf16_to_f32(rd16(ch + 4096 + (r * 8 + g) * 2));
        f.zero = oracle_bf16_to_f32(rd16(ch + 4608 + (r * 8 + g) * 2));
        break;
    case ORC_Q4_K:
        f.code = code4(ch, r, k);
        f.sc = ch[4096 + r * 8 + g];
        f.mn = ch[4352 + r * 8 + g];
        f.S = oracle_bf16_to_f32(rd16(ch + 4608 + r * 2));
        f.M = oracle_bf16_to_f32(rd16(ch + 4672 + r * 2));
        break;
    default: /* Q8, either layout */
        f.code = code8(ch, kind, r, k);
        f.d = oracle_bf16_to_f32(rd16(ch + 8192 + (r * 8 + g) * 2));
        break;
    }
    return f;
}

/* Weight (n, k) of the whole tensor, its fields */
static fields_t weight_fields(const uint8_t* w, int kind, int64_t K, int64_t n, int64_t k)
{
    const uint8_t* ch = chunk_at(w, kind, K, n / 32, k / 256);
    return read_fields(ch, kind, (int)(n % 32), (int)(k % 256));
}

/* The weight's value in exact arithmetic (binary64 holds every product and
 * sum of these fields exactly for finite inputs of the generators' ranges). */
static double weight_exact(fields_t f, int kind)
{
    switch (kind) {
    case ORC_Q4_1: return (double)f.code * (double)f.scale + (double)f.zero;
    case ORC_Q4_K: return (double)f.S * (double)f.sc * (double)f.code + (double)f.M * (double)f.mn;
    default: return (double)f.d * (double)f.code;
    }
}

/* The weight as the binary32 decode forms it: one operation at a time,
 * rounded after each (no contraction).  Every product here is exact in
 * binary32 (code 4 bits x bf16 8 bits; S 8 bits x sc 8 bits x code 4 bits;
 * M 8 bits x mn 8 bits; d 8 bits x code 8 bits), so the only rounding is the
 * one addition. */
static float weight_f32(fields_t f, int kind)
{
    switch (kind) {
    case ORC_Q4_1: {
        float t = (float)f.code * f.scale;
        return t + f.zero;
    }
    case ORC_Q4_K: {
        float a = f.S * (float)f.sc;
        float t = a * (float)f.code;
        float u = f.M * (float)f.mn;
        return t + u;
    }
    default:
        return f.d * (float)f.code;
    }
}

/* ------------------------------------------------------------ exported --- */

/* Logical fields of every weight, for round-trip checks.
 * code[n*K+k] gets the stored code (0..15 or -128..127). */
void oracle_codes(const uint8_t* w, int kind, int64_t N, int64_t K, int32_t* code)
{
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k)
            code[n * K + k] = weight_fields(w, kind, K, n, k).code;
}

/* Decode to bf16 [N][K] row-major: bf16_rne(weight_f32). */
void oracle_decode(const uint8_t* w, int kind, int64_t N, int64_t K, uint16_t* out)
{
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k)
            out[n * K + k] = oracle_f32_to_bf16(weight_f32(weight_fields(w, kind, K, n, k), kind));
}

/* Decode to binary32 [N][K] (the value before the bf16 rounding). */
void oracle_decode_f32(const uint8_t* w, int kind, int64_t N, int64_t K, float* out)
{
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k)
            out[n * K + k] = weight_f32(weight_fields(w, kind, K, n, k), kind);
}

/* Exact weights in binary64 [N][K]. */
void oracle_weights_f64(const uint8_t* w, int kind, int64_t N, int64_t K, double* out)
{
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k)
            out[n * K + k] = weight_exact(weight_fields(w, kind, K, n, k), kind);
}

/* Y[m][j] = sum_k w(rows[j], k) * X[m][k] in binary64, k ascending, for the
 * nrows output rows listed in rows[] (all rows: rows[j] = j).  X is bf16
 * [M][K] row-major.  A[m][j] = sum_k |w * x|, the scale of the tolerance.
 * Y and A are [M][nrows] row-major. */
void oracle_matmul_rows(const uint8_t* w, int kind, int64_t N, int64_t K,
                        const uint16_t* X, int64_t M,
                        const int64_t* rows, int64_t nrows, double* Y, double* A)
{
    (void)N;
    for (int64_t j = 0; j < nrows; ++j) {
        int64_t n = rows[j];
        for (int64_t m = 0; m < M; ++m) {
            Y[m * nrows + j] = 0.0;
            A[m * nrows + j] = 0.0;
        }
        for (int64_t k = 0; k < K; ++k) {
            double wk = weight_exact(weight_fields(w, kind, K, n, k), kind);
            for (int64_t m = 0; m < M; ++m) {
                double p = wk * (double)oracle_bf16_to_f32(X[m * K + k]);
                Y[m * nrows + j] += p;
                A[m * nrows + j] += fabs(p);
            }
        }
    }
}

/* Q4_K -> q4_1 repack ("NPU engine" page, paragraph after the chunk table):
 * codes unchanged; scale = bf16(S * sc), zero = bf16(M * mn), per (row, group).
 * Each product is exact in binary32 (8 x 8 significant bits), so the rounding
 * to bf16 is the only one.  in: TR*TC Q4_K chunks; out: TR*TC q4_1 chunks. */
void oracle_repack_q4k(const uint8_t* in, int64_t N, int64_t K, uint8_t* out)
{
    int64_t tiles = (N / 32) * (K / 256);
    for (int64_t t = 0; t < tiles; ++t) {
        const uint8_t* src = in + t * 4736;
        uint8_t* dst = out + t * 5120;
        for (int i = 0; i < 4096; ++i)
            dst[i] = src[i];
        for (int r = 0; r < 32; ++r) {
            float S = oracle_bf16_to_f32(rd16(src + 4608 + r * 2));
            float M = oracle_bf16_to_f32(rd16(src + 4672 + r * 2));
            for (int g = 0; g < 8; ++g) {
                uint16_t s = oracle_f32_to_bf16(S * (float)src[4096 + r * 8 + g]);
                uint16_t z = oracle_f32_to_bf16(M * (float)src[4352 + r * 8 + g]);
                dst[4096 + (r * 8 + g) * 2] = (uint8_t)(s & 0xFF);
                dst[4096 + (r * 8 + g) * 2 + 1] = (uint8_t)(s >> 8);
                dst[4608 + (r * 8 + g) * 2] = (uint8_t)(z & 0xFF);
                dst[4608 + (r * 8 + g) * 2 + 1] = (uint8_t)(z >> 8);
            }
        }
    }
}

/* Top-1 of each logits row [M][V]: the first maximum; a NaN counts as larger
 * than every number, so the first NaN wins; +-inf compare as usual. */
void oracle_argmax(const float* logits, int64_t M, int64_t V, int32_t* idx)
{
    for (int64_t m = 0; m < M; ++m) {
        const float* row = logits + m * V;
        int64_t best = 0;
        for (int64_t v = 0; v < V; ++v) {
            if (isnan(row[v])) { best = v; break; }
            if (row[v] > row[best]) best = v;
        }
        idx[m] = (int32_t)best;
    }
}

/* ------------------------------------------------------------------------
 * GGUF-type tensors -> q4_1 chunks ("NPU engine" page, section "From a GGUF",
 * the GGUF-type table):
 *   Q4_0  -> scale d, zero -8d, codes unchanged   (error: bf16 rounding of scale and zero)
 *   Q4_1  -> scale d, zero m,   codes unchanged   (same)
 *   Q8_0, F32, F16, BF16 -> dequantized, then a min/max q4_1 per 32 columns (lossy)
 *
 * The page names the GGUF types but does not print their blocks.  Reading used
 * (the GGUF block structs): a tensor [N][K] is row-major, a row is K/32 blocks
 * of 32 consecutive columns;
 *   Q4_0 block 18 B: fp16 d, 16 code bytes; element i < 16 is the low nibble of
 *        byte i, element i >= 16 the high nibble of byte i - 16; value d*(q - 8)
 *   Q4_1 block 20 B: fp16 d, fp16 m, 16 code bytes (as Q4_0); value d*q + m
 *   Q8_0 block 34 B: fp16 d, 32 int8 codes; value d*q
 *   F32 / F16 / BF16: N*K little-endian values.
 * Min/max q4_1 of 32 values x (reading, made exact in binary32 one operation at
 * a time): lo = min x, hi = max x; scale s = bf16((hi - lo) / 15); zero
 * z = bf16(lo); code = clamp(rint((x - z) / s), 0, 15) with s, z the stored
 * bf16 values (ties to even); every code is 0 when s == 0.  Inputs are finite.
 */
enum { ORC_SRC_Q4_0 = 1, ORC_SRC_Q4_1 = 2, ORC_SRC_Q8_0 = 3, ORC_SRC_F32 = 4, ORC_SRC_F16 = 5, ORC_SRC_BF16 = 6 };

/* IEEE binary16 -> binary32 (exact): 1 sign, 5 exponent (bias 15), 10 fraction bits */
float oracle_f16_to_f32(uint16_t h)
{
    int sign = (h >> 15) & 1, e = (h >> 10) & 31, f = h & 1023;
    float v;
    if (e == 0) v = ldexpf((float)f, -24);                 /* zero and subnormals: f * 2^-24 */
    else if (e == 31) v = f ? NAN : INFINITY;
    else v = ldexpf((float)(f + 1024), e - 25);            /* (1 + f/1024) * 2^(e-15) */
    return sign ? -v : v;
}

static void put16(uint8_t* p, uint16_t v) { p[0] = (uint8_t)(v & 0xFF); p[1] = (uint8_t)(v >> 8); }

/* value of element (n, k) of a dense or Q8_0 source, in binary32 */
static float src_value(const uint8_t* src, int type, int64_t K, int64_t n, int64_t k)
{
    if (type == ORC_SRC_F32) { float v; memcpy(&v, src + (n * K + k) * 4, 4); return v; }
    if (type == ORC_SRC_F16) return oracle_f16_to_f32(rd16(src + (n * K + k) * 2));
    if (type == ORC_SRC_BF16) return oracle_bf16_to_f32(rd16(src + (n * K + k) * 2));
    /* Q8_0 */
    const uint8_t* blk = src + (n * (K / 32) + k / 32) * 34;
    float d = oracle_f16_to_f32(rd16(blk));
    int8_t q = (int8_t)blk[2 + k % 32];
    return (float)q * d;                                    /* exact: 8 x 11 significant bits */
}

/* out: TR*TC q4_1 chunks of the N x K tensor `src` of GGUF type `type` */
void oracle_pack_q4_1(const uint8_t* src, int type, int64_t N, int64_t K, uint8_t* out)
{
    int64_t TC = K / 256;
    for (int64_t n = 0; n < N; ++n) {
        int64_t tr = n / 32;
        int r = (int)(n % 32);
        for (int64_t b = 0; b < K / 32; ++b) {          /* one 32-column group of row n */
            int64_t tc = b / 8;
            int g = (int)(b % 8);
            uint8_t* ch = out + (tr * TC + tc) * 5120;
            int q[32];
            uint16_t s_bits, z_bits;
            if (type == ORC_SRC_Q4_0 || type == ORC_SRC_Q4_1) {
                int bs = type == ORC_SRC_Q4_0 ? 18 : 20;
                const uint8_t* blk = src + (n * (K / 32) + b) * bs;
                float d = oracle_f16_to_f32(rd16(blk));
                const uint8_t* qs = blk + (type == ORC_SRC_Q4_0 ? 2 : 4);
                for (int i = 0; i < 32; ++i) q[i] = i < 16 ? (qs[i] & 15) : (qs[i - 16] >> 4);
                s_bits = oracle_f32_to_bf16(d);
                if (type == ORC_SRC_Q4_0) z_bits = oracle_f32_to_bf16(-8.0f * d);   /* exact product */
                else z_bits = oracle_f32_to_bf16(oracle_f16_to_f32(rd16(blk + 2)));
            } else {
                float x[32], lo, hi;
                for (int i = 0; i < 32; ++i) x[i] = src_value(src, type, K, n, b * 32 + i);
                lo = hi = x[0];
                for (int i = 1; i < 32; ++i) {
                    if (x[i] < lo) lo = x[i];
                    if (x[i] > hi) hi = x[i];
                }
                float range = hi - lo;
                float step = range / 15.0f;
                s_bits = oracle_f32_to_bf16(step);
                z_bits = oracle_f32_to_bf16(lo);
                float s = oracle_bf16_to_f32(s_bits), z = oracle_bf16_to_f32(z_bits);
                for (int i = 0; i < 32; ++i) {
                    if (s == 0.0f) { q[i] = 0; continue; }
                    float t = x[i] - z;
                    float u = t / s;
                    float c = rintf(u);                     /* nearest, ties to even */
                    q[i] = c < 0.0f ? 0 : (c > 15.0f ? 15 : (int)c);
                }
            }
            for (int j = 0; j < 16; ++j)                    /* code (r, k) in byte r*128 + k/2, low nibble even k */
                ch[r * 128 + g * 16 + j] = (uint8_t)(q[2 * j] | (q[2 * j + 1] << 4));
            put16(ch + 4096 + (r * 8 + g) * 2, s_bits);
            put16(ch + 4608 + (r * 8 + g) * 2, z_bits);
        }
    }
}
