/*
 * q4nx.h -- C ABI of libq4nx.so: Q4NX dequant-GEMV / GEMM on one GB300 (sm_103a).
 *
 * Operations come from the 1bit engine page "NPU engine" (docs/npu.md),
 * section "Q4NX chunks": a weight W[N][K] is a grid of 32-row x 256-column
 * tiles, one chunk per tile, chunks row-major over the grid; three chunk kinds
 * (chunk-kind table), two Q8 code layouts, decoders for all kinds, and the
 * Q4_K -> q4_1 repack.
 *
 * Byte order inside a chunk (the page does not print it; this library fixes it):
 *   q4_1  5120 B: codes 4096 | scale bf16 [32 r][8 g] | zero bf16 [32 r][8 g]
 *   Q4_K  4736 B: codes 4096 | sc u8 [32][8] | mn u8 [32][8] | S bf16 [32] | M bf16 [32]
 *   Q8    8704 B: codes int8 8192 (layout KR or BLK) | d bf16 [32 r][8 g]
 *   4-bit code (r, k): byte r*128 + k/2, low nibble for even k, high for odd k.
 *   g = k/32.  All bf16 fields little-endian.
 *
 * Conventions for every entry point
 *   - Pointers named *_dev are device pointers (cudaMalloc'd or from a
 *     framework allocator); the caller owns them.  The library allocates
 *     nothing, frees nothing and keeps no pointer after a call returns.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Work is enqueued on it; nothing synchronises.
 *   - Arguments are validated before anything is enqueued.  A non-zero status
 *     means nothing was launched and no output byte was written, except
 *     Q4NX_E_CUDA (the launch itself failed; outputs undefined).
 *   - Device buffers must start on 16-byte boundaries (Q4NX_E_ALIGN).
 *   - No exception crosses this boundary; there is no global error state.
 *   - Calls are thread-safe.  Two calls that share a workspace must not
 *     overlap on the GPU.
 */
#ifndef Q4NX_H
#define Q4NX_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Chunk kinds ("Q4NX chunks", chunk-kind table; Q8 layouts from the paragraph below it). */
enum q4nx_kind {
    Q4NX_Q4_1 = 1,    /* 5120 B: w = code*scale + zero                               */
    Q4NX_Q4_K = 2,    /* 4736 B: w = S*sc*code + M*mn                                */
    Q4NX_Q8_KR = 3,   /* 8704 B: w = d*code, code (r,k) at byte k*32 + r             */
    Q4NX_Q8_BLK = 4   /* 8704 B: code (r,k) at (r/16)*4096+(k/32)*512+(k%32)*16+r%16 */
};

/* Status codes. */
enum q4nx_status {
    Q4NX_OK = 0,
    Q4NX_E_NULL = 1,            /* a required pointer is NULL                          */
    Q4NX_E_KIND = 2,            /* unknown chunk kind                                  */
    Q4NX_E_SHAPE = 3,           /* rows % 32, cols % 256, or a size <= 0               */
    Q4NX_E_SHORT = 4,           /* a buffer is shorter than its layout needs           */
    Q4NX_E_ALIGN = 5,           /* a device buffer is not 16-byte aligned              */
    Q4NX_E_M = 6,               /* M outside 1..64                                     */
    Q4NX_E_WORKSPACE = 7,       /* workspace NULL or smaller than the *_workspace size */
    Q4NX_E_UNSUPPORTED = 8,     /* valid kind, but not for this operation / size       */
    Q4NX_E_CUDA = 9,            /* a CUDA call failed (launch error)                   */
    Q4NX_E_DEVICE_TIMEOUT = 10, /* a bounded in-kernel wait gave up (see q4nx_check)   */
    Q4NX_E_DTYPE = 11           /* unknown output dtype                                */
};

/* Output element type of the products. */
enum q4nx_out { Q4NX_OUT_BF16 = 0, Q4NX_OUT_F32 = 1 };

/* A Q4NX weight: `rows` x `cols` (N x K), TR = rows/32 tile rows by TC = cols/256
 * tile columns, chunk (tr, tc) at byte (tr*TC + tc) * chunk_bytes(kind).
 * A contiguous range of tile rows of a larger weight is itself a weight
 * (chunks_dev advanced by tr0*TC*chunk_bytes, rows = count*32). */
typedef struct q4nx_weight {
    const void* chunks_dev;   /* device, 16-byte aligned                          */
    uint64_t bytes;           /* length of the chunk buffer                       */
    int32_t kind;             /* enum q4nx_kind                                   */
    int32_t reserved;         /* must be 0                                        */
    int64_t rows;             /* N, multiple of 32                                */
    int64_t cols;             /* K, multiple of 256                               */
} q4nx_weight;

/* Bytes of one chunk of `kind` (5120, 4736, 8704, 8704), 0 for an unknown kind. */
uint64_t q4nx_chunk_bytes(int kind);

/* A static, human-readable name of a status code. */
const char* q4nx_status_str(int status);

/* Library ABI version (bumped on any signature change). */
int q4nx_abi_version(void);

/* Decode a whole weight to bf16 ("Q4NX chunks", decoders paragraph).
 * out_dev: bf16 [rows][cols] row-major, rows*cols*2 bytes.
 * Each weight is formed in binary32 one operation at a time (no contraction):
 *   q4_1 (code*scale) + zero;  Q4_K ((S*sc)*code) + (M*mn);  Q8 d*code,
 * then rounded to bf16 to nearest-even.  Every product is exact in binary32,
 * so the result is bf16(fl32(exact)).  All four kinds. */
int q4nx_decode(const q4nx_weight* w, void* out_dev, uint64_t out_bytes, void* stream);

/* Fused decode + GEMV, one token:  y[n] = sum_k w[n][k] * x[k]  (fp32 accumulation).
 * x_dev: bf16 [cols].  y_dev: [rows] of out_dtype (bf16 rounds to nearest-even;
 * fp32 is meant for lm_head logits).  All four kinds, any cols.
 * workspace_dev: device scratch of at least q4nx_gemv_workspace(w) bytes, 16-byte
 * aligned, ZERO-FILLED before its first use; every call leaves it zero-filled
 * again (after Q4NX_E_DEVICE_TIMEOUT it must be zero-filled anew).  It holds
 * an error word and the partial sums of tile rows split between CTAs, each
 * posted with a ready flag (16 B + 256 KiB for any weight).
 * Non-finite activations give each row the IEEE outcome of the sum (+-Inf,
 * or NaN for 0*Inf or a NaN activation); chunks whose scale or zero fields
 * are non-finite give non-finite rows, but not necessarily the per-weight
 * pattern of Inf and NaN (decode such chunks with q4nx_decode instead).
 * Results are deterministic: partials are added in a fixed order.  A tile row
 * split between CTAs is finished by the CTA that holds its first chunk once
 * the later CTAs (at most two per SM) have posted; they get SMs as soon as
 * any frees, and a wait that still runs out reports Q4NX_E_DEVICE_TIMEOUT
 * through q4nx_check. */
int q4nx_gemv(const q4nx_weight* w, const void* x_dev, void* y_dev, int out_dtype,
              void* workspace_dev, uint64_t workspace_bytes, void* stream);
uint64_t q4nx_gemv_workspace(const q4nx_weight* w);

/* lm_head GEMV fused with top-1 (greedy decoding: the serving section of the
 * "NPU engine" page and onw's TECHNICAL.md take only the argmax of the logits):
 * *idx_dev = argmax over n of y[n], y = w * x_dev computed exactly as
 * q4nx_gemv with Q4NX_OUT_F32 computes it.  Ties go to the lowest row; a NaN
 * output wins (the first one).  The logits are never written to memory.
 * idx_dev: device int32, 4-byte aligned.  Workspace: q4nx_gemv_workspace(w)
 * bytes under the same zero-fill rule (the launch uses bytes 4..15 of it and
 * leaves them zero). */
int q4nx_gemv_top1(const q4nx_weight* w, const void* x_dev, int32_t* idx_dev, void* workspace_dev,
                   uint64_t workspace_bytes, void* stream);

/* Vocabulary-sharded lm_head top-1 (the sharding of the lm_head rows over
 * GPUs, each GPU holding a contiguous range of rows): the GEMV of this shard
 * fused with top-1 as q4nx_gemv_top1 computes it, written as one 64-bit key
 * instead of an index, so that the shards' winners combine with a single MAX
 * reduction of int64 values (an all-reduce, or a max on the host):
 *   key = (ord(v) << 32 | (0xFFFFFFFF - (row_base + n))) XOR (1 << 63)
 * where v is the shard's largest fp32 output, n its row within the shard (the
 * lowest of equal maxima; a NaN output counts as the largest, the first one
 * winning) and ord maps fp32 to uint32 preserving order (-0 as +0, NaN to
 * 0xFFFFFFFF).  The flipped top bit makes the signed int64 order equal the
 * unsigned key order.  The global row of a combined key is
 * 0xFFFFFFFF - (key & 0xFFFFFFFF).
 * row_base: the shard's first global row, 0 <= row_base <= INT32_MAX - rows
 * (Q4NX_E_SHAPE otherwise).  key_dev: device int64, 8-byte aligned.
 * Workspace as for q4nx_gemv_top1. */
int q4nx_gemv_top1_key(const q4nx_weight* w, const void* x_dev, int64_t row_base, int64_t* key_dev,
                       void* workspace_dev, uint64_t workspace_bytes, void* stream);

/* One GEMV of a batch: y_dev[rows] = w * x_dev[cols]. */
typedef struct q4nx_gemv_item {
    q4nx_weight w;
    const void* x_dev;        /* bf16 [w.cols], 16-byte aligned */
    void* y_dev;              /* [w.rows] of the batch's out_dtype, 16-byte aligned */
} q4nx_gemv_item;

/* Up to Q4NX_MAX_BATCH independent GEMVs of ONE chunk kind in one launch: the
 * chunks of all items are spread evenly over the GPU, so many small matrices
 * (a decode layer's projections) stream at the bandwidth of one large one.
 * `items` is a HOST array (read during the call only).  Each item behaves as
 * q4nx_gemv; the workspace is q4nx_gemv_batch_workspace(items, count) bytes
 * under the same zero-fill rule.  Q4NX_E_KIND if the kinds differ,
 * Q4NX_E_SHAPE if count is outside 1..Q4NX_MAX_BATCH. */
#define Q4NX_MAX_BATCH 256
int q4nx_gemv_batch(const q4nx_gemv_item* items, int count, int out_dtype,
                    void* workspace_dev, uint64_t workspace_bytes, void* stream);
uint64_t q4nx_gemv_batch_workspace(const q4nx_gemv_item* items, int count);

/* Fused decode + GEMM for a block of 1..64 tokens on the tcgen05 tensor cores:
 *   Y[m][n] = sum_k X[m][k] * w[n][k],  m < M.
 * X_dev: bf16 [M][cols] row-major.  Y_dev: [M][rows] row-major of out_dtype.
 * A few tokens run on the CUDA cores (M = 1 for every kind, as q4nx_gemv;
 * M = 2 for q4_1; M <= 4 for Q4_K): each chunk is read once and its codes
 * enter exact integer dot products with every token.  Larger M runs on
 * the tensor cores: weights are decoded to bf16 (code*scale + zero for q4_1,
 * rounded once; d*code for Q8, exactly the standalone decode) into tensor
 * memory and multiplied with fp32 accumulation there; kinds q4_1, Q8_KR,
 * Q8_BLK, while Q4_K returns Q4NX_E_UNSUPPORTED (repack it with
 * q4nx_repack_q4k first, which keeps the codes).  The tensor-core launch
 * expects its CTAs (at most one per SM) to be resident together, as they are
 * when no other kernel occupies the GPU; a stalled launch gives up after a
 * bounded wait and reports it through q4nx_check.
 * Accuracy: CUDA-core outputs as q4nx_gemv; tensor-core outputs multiply
 * bf16-rounded weights, each within 2^-9 of itself, so an output may differ
 * from the exact sum by that much of sum_k |w x| beyond the fp32 rounding.
 * workspace_dev: at least q4nx_gemm_workspace(w, M) bytes (the same for every
 * M), zero-filled before first use and again after Q4NX_E_DEVICE_TIMEOUT; it
 * holds the error word, and calls may leave partial sums in it, so it is not
 * shared with the GEMV entry points. */
int q4nx_gemm_m64(const q4nx_weight* w, const void* X_dev, int M, void* Y_dev, int out_dtype,
                  void* workspace_dev, uint64_t workspace_bytes, void* stream);
uint64_t q4nx_gemm_workspace(const q4nx_weight* w, int M);

/* Q4_K -> q4_1 repack ("Q4NX chunks", decoders paragraph): codes copied byte for
 * byte; scale = bf16(S*sc), zero = bf16(M*mn) per (row, group), nearest-even.
 * in_dev: TR*TC Q4_K chunks (in_bytes >= TR*TC*4736).  out_dev: TR*TC q4_1
 * chunks (out_bytes >= TR*TC*5120).  rows, cols as for a weight. */
int q4nx_repack_q4k(const void* in_dev, uint64_t in_bytes, int64_t rows, int64_t cols,
                    void* out_dev, uint64_t out_bytes, void* stream);

/* GGUF-type tensor -> q4_1 chunks ("NPU engine" page, section "From a GGUF",
 * GGUF-type table).  Q4NX_SRC_Q4_0 becomes scale d, zero -8d and Q4NX_SRC_Q4_1
 * scale d, zero m, codes unchanged: the only error is the bf16 rounding of
 * scale and zero.  Q4NX_SRC_Q8_0, _F32, _F16 and _BF16 are dequantized and
 * quantized to a min/max q4_1 per 32 columns (lossy): lo, hi of the 32 values
 * (the first of equal minima / maxima), scale = bf16((hi - lo) / 15),
 * zero = bf16(lo), code = clamp(rint((x - zero) / scale), 0, 15) with the
 * stored scale and zero (ties to even; 0 when scale is 0), each step one IEEE
 * binary32 operation.  Inputs must be finite.
 * src_dev: the rows x cols tensor, row-major, as GGUF blocks of 32 columns
 * (Q4_0: 18 B = fp16 d + 16 code bytes, element i < 16 in the low nibble of
 * byte i and i >= 16 in the high nibble of byte i - 16; Q4_1: 20 B = fp16 d,
 * fp16 m + those 16 bytes; Q8_0: 34 B = fp16 d + 32 int8) or dense values
 * (4 / 2 / 2 bytes each); 16-byte aligned; at least rows * cols/32 blocks.
 * out_dev: (rows/32)*(cols/256)*5120 bytes, 16-byte aligned. */
enum { Q4NX_SRC_Q4_0 = 1, Q4NX_SRC_Q4_1 = 2, Q4NX_SRC_Q8_0 = 3, Q4NX_SRC_F32 = 4, Q4NX_SRC_F16 = 5, Q4NX_SRC_BF16 = 6 };
int q4nx_pack_q4_1(int src_type, const void* src_dev, uint64_t src_bytes, int64_t rows, int64_t cols, void* out_dev,
                   uint64_t out_bytes, void* stream);

/* Top-1 of each row of fp32 logits [M][V] (greedy decoding, "Serving" section):
 * idx_dev[m] = index of the first maximum; a NaN counts above every number and
 * the first NaN wins; +0 and -0 are equal.  1 <= M <= 65535, 1 <= V < 2^31. */
int q4nx_argmax(const float* logits_dev, int M, int64_t V, int32_t* idx_dev, void* stream);

/* GEMV without any allocation, for callers that may not allocate device memory
 * at all: code that runs under a strict no-allocation policy once set up (for
 * example a real-time decode loop, or a plug-in inside a framework that owns
 * every device allocation and hands out only inputs and outputs).  The pages
 * have no counterpart of this entry point; it is q4nx_gemv with its scratch
 * memory (error word, posted partial sums) taken from a 1 MiB array compiled
 * into the library, which every GPU that loads the library keeps until the
 * process exits.
 * The caller passes inputs and outputs only, exactly as for q4nx_gemv; the
 * arguments are checked as q4nx_gemv checks them (same statuses, same order;
 * there is no workspace to check).  Every call looks up the current device's
 * copy of the array (cudaGetSymbolAddress, a host-side lookup); the first call
 * on a device also loads the library's device code there, so make it before
 * any stream capture.  Every call clears the scratch it uses before its
 * launch, so a call never depends on what an earlier call left behind; but all
 * calls on a device share the one array, so calls that can overlap on the GPU
 * (different streams, or concurrent graph branches) race and must be
 * serialised by the caller.  The scratch a call needs does not grow with the
 * weight, so every weight that q4nx_gemv accepts fits
 * q4nx_noalloc_scratch_bytes().  A bounded in-kernel wait that gives up
 * (see q4nx_gemv) is reported by q4nx_check_noalloc, not by the call.  Calls
 * no cudaMalloc or cudaFree. */
int q4nx_gemv_noalloc(const q4nx_weight* w, const void* x_dev, void* y_dev, int out_dtype, void* stream);
uint64_t q4nx_noalloc_scratch_bytes(void);

/* The error word of q4nx_gemv_noalloc's built-in scratch on the current
 * device: read it after the calls to check (synchronises `stream`) and before
 * the next call, which clears it.  Q4NX_OK, or Q4NX_E_DEVICE_TIMEOUT if a
 * bounded wait of an earlier call gave up (that call's outputs are invalid);
 * the array is then cleared.  Q4NX_E_CUDA if the lookup or the copy fails. */
int q4nx_check_noalloc(void* stream);

/* Read and clear the error word of a workspace (synchronises `stream`).
 * Returns Q4NX_OK, or Q4NX_E_DEVICE_TIMEOUT if a bounded in-kernel wait of a
 * call that used this workspace gave up (its outputs are then invalid, and
 * the workspace must be zero-filled before it is used again: the calls that
 * gave up may have left counters and posted sums in it). */
int q4nx_check(void* workspace_dev, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* Q4NX_H */
