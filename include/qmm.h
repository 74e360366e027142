/*
 * qmm.h -- C ABI of the B300 (sm_103a) GGML block-quantized linear layer.
 *
 * What it computes.  The mistral.rs documentation page "Quantization types"
 * describes in-situ quantization (ISQ): unquantized (bf16) weights are
 * quantized at load time (opening section, `--isq N`), and on CUDA the
 * shorthand 8 resolves to Q8_0 and 4 to Q4K (section "Numeric shorthands";
 * widths in tables "Legacy GGML types" and "Q*K family").  This library
 * provides that step and the linear layer that consumes it:
 *
 *   qmm_quantize    bf16 (or fp32) weights W[rows x cols] -> packed blocks
 *   qmm_dequantize  packed blocks -> fp32 W^[rows x cols] (exact)
 *   qmm_matmul      Y[M x N] = X[M x K] * W^[N x K]^T   (fp32 out, bf16 X)
 *   qmm_embedding   rows ids[] of a packed [V x D] table -> fp32 / bf16
 *
 * Formats: Q8_0 and Q4_K (the CUDA targets of `--isq 8` / `--isq 4`) and
 * FP8 E4M3 with row scales (W8A16) for the linear layers, and Q6_K
 * (`--isq 6`), which the page's section
 * "Sensitive tensor precision" gives to the token embeddings and the output
 * head of a Q4K model (Q8_0 for Q5K / Q6K / Q8_0 models; see
 * qmm_embedding_format).
 *
 * The pages give names and widths only.  The byte layouts and the quantizer
 * used here (the library's reading, GGUF-shaped) are:
 *
 *   Q8_0  32 weights -> 34 bytes: binary16 d = fp16(max|x| / 127), then
 *         int8 q_i = clamp(round_half_away(x_i / d), -127, 127).
 *         Dequantized weight: d * q.
 *   Q4_K  256 weights -> 144 bytes: binary16 d, binary16 dmin, 12 bytes of
 *         eight 6-bit sub-block scale codes sc_j and eight 6-bit min codes
 *         mc_j, 128 bytes of 4-bit codes q (byte 32c+l: weight l of sub-block
 *         2c in the low nibble, of sub-block 2c+1 in the high nibble).
 *         Per 32-weight sub-block: s_j = (max - min(0, min)) / 15,
 *         m_j = -min(0, min); d = fp16(max_j s_j / 63), dmin = fp16(max_j
 *         m_j / 63); sc_j, mc_j = round(s_j / d), round(m_j / dmin) in 0..63;
 *         q = round((x + dmin*mc_j) / (d*sc_j)) in 0..15.
 *         Dequantized weight: (d*sc_j) * q - dmin*mc_j.
 *   Scale bytes of Q4_K, j = 0..3: byte j = sc_j | (sc_{j+4} >> 4) << 6;
 *   byte j+4 = mc_j | (mc_{j+4} >> 4) << 6; byte j+8 = (sc_{j+4} & 15) |
 *   (mc_{j+4} & 15) << 4.
 *   Q6_K  256 weights -> 210 bytes: 16 sub-blocks of 16.  s_j = max|x| / 31;
 *         d = fp16(max_j s_j / 127); sc_j = round(s_j / d) in 0..127 (int8);
 *         c = clamp(round(x / (d*sc_j)), -32, 31), stored as q = c + 32.
 *         Dequantized weight: (d*sc_j) * c.  Bytes 0-127 ql (low 4 bits of
 *         q), 128-191 qh (high 2 bits), 192-207 sc[16], 208-209 d; weight
 *         w = 128h + 32s + l (h < 2, s < 4, l < 32) has its low bits in ql
 *         byte 64h + 32(s & 1) + l (high nibble when s >= 2) and its high
 *         bits in bits 2s, 2s+1 of qh byte 32h + l.  Superblocks are only
 *         2-byte aligned inside a packed row.
 *   Q5_K  256 weights -> 176 bytes: Q4_K's quantizer with 5-bit codes
 *         (s_j = (max - min(0, min)) / 31, q in 0..31).  Bytes 0-1 d, 2-3
 *         dmin, 4-15 the scale bytes (Q4_K's packing), 16-47 qh, 48-175 qs:
 *         byte 48+32c+l holds the low 4 bits of weight l of sub-block 2c
 *         (low nibble) and 2c+1 (high nibble); bit j of qh byte 16+l is bit 4
 *         of weight l of sub-block j.  Value (d*sc_j) * q - dmin*mc_j.
 *   Q3_K  256 weights -> 110 bytes, 16 sub-blocks of 16, symmetric:
 *         s_j = max|x| / 3; d = fp16(max_j s_j / 31); sc_j = round(s_j / d)
 *         in 0..31; c = clamp(round(x / (d*sc_j)), -4, 3), q = c + 4.  Bytes
 *         0-31 hmask, 32-95 qs, 96-107 sixteen 6-bit fields sc_j + 32 (low 4
 *         bits of field j in byte j mod 8, high nibble for j >= 8; high 2 bits
 *         at bit 2 (j div 4) of byte 8 + j mod 4), 108-109 d.  Weight w =
 *         128h + 32s + l: bits 0-1 of q at bit 2s of qs byte 32h + l, bit 2 at
 *         bit 4h + s of hmask byte l.  Value (d*sc_j) * c (exact).
 *   Q2_K  256 weights -> 84 bytes, 16 sub-blocks of 16, affine: s_j =
 *         (max - min(0, min)) / 3, m_j = -min(0, min); d, dmin = fp16(max_j
 *         s_j / 15), fp16(max_j m_j / 15); sc_j, mc_j in 0..15; q in 0..3.
 *         Bytes 0-15 scales (sc_j | mc_j << 4), 16-79 qs (weight w = 128h +
 *         32s + l at bit 2s of byte 16 + 32h + l), 80-81 d, 82-83 dmin.  Value
 *         (d*sc_j) * q - dmin*mc_j.
 *   Q5_K / Q3_K / Q2_K are the page's q5k / q3k / q2k (table "Q*K family";
 *         `--isq 5 / 3 / 2` on CUDA).  Q5_K superblocks are 16-byte aligned
 *         and its matmul runs the row-tile decode kernel and the tiled
 *         tensor-core kernel; Q3_K and Q2_K superblocks are only 2- or 4-byte
 *         aligned inside a row, and the library serves them with CUDA-core
 *         kernels (see qmm_matmul).
 *   FP8_E4M3  (W8A16; the page's section "FP8": E4M3 produced by ISQ,
 *         symmetric weights with channel scales): one fp32 scale per row,
 *         s = max|x| / 448; code = E4M3(x / s), round to nearest even,
 *         saturating at +-448 (E4M3: 1 sign, 4 exponent bits with bias 7, 3
 *         fraction bits, no infinities).  Dequantized weight: E4M3 value * s.
 *         A packed row is the K codes, s (fp32), 12 zero bytes: K + 16.
 *
 * A packed matrix is row-major in blocks: row n holds cols/32 Q8_0 blocks
 * (cols/32*34 bytes), cols/256 K-quant superblocks (cols/256 * 144 / 210 /
 * 176 / 110 / 84 bytes for Q4_K / Q6_K / Q5_K / Q3_K / Q2_K) or the FP8 codes
 * and row scale (cols + 16 bytes), rows back to back.
 *
 * Conventions for every call:
 *  - Pointers are DEVICE pointers owned by the caller.  The library allocates
 *    nothing and never synchronises; work is enqueued on `stream` (NULL = the
 *    legacy default stream) and completes asynchronously.
 *  - Row-major, contiguous, 16-byte aligned buffers; buffers must not alias.
 *  - cols (K) must be a positive multiple of 256 for both formats (this makes
 *    every packed row a multiple of 16 bytes).  rows / N / M may be 0 (nothing
 *    is launched) or any positive value.
 *  - Arguments are checked on the host before anything is launched; on an
 *    error nothing is enqueued and the status says why.  A launch failure
 *    reported by the CUDA runtime maps to QMM_ERR_CUDA.  Faults during the
 *    asynchronous execution surface at the caller's next synchronisation.
 *  - NaN or infinite inputs give unspecified (but memory-safe) results.
 *  - qmm_matmul feeds binary16 operands to the tensor cores (see its
 *    declaration for the exact accuracy contract): |x| must stay below 65504.
 *  - No C++ exception crosses this interface.
 */
#ifndef QMM_H
#define QMM_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define QMM_API __attribute__((visibility("default")))
#else
#define QMM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream (cudaStream_t); declared here so that this header does not
 * need the CUDA headers. */
struct CUstream_st;
typedef struct CUstream_st *qmm_stream_t;

/* Block formats; the values mirror the ISQ shorthands `--isq 8 / 6 / 5 / 4 /
 * 3 / 2` (mistral.rs "Quantization types", section "Numeric shorthands":
 * Q8_0, Q6K, Q5K, Q4K, Q3K, Q2K on CUDA). */
typedef enum {
    QMM_Q8_0 = 8,
    QMM_Q4_K = 4,
    QMM_Q6_K = 6,
    QMM_Q5_K = 5,
    QMM_Q3_K = 3,
    QMM_Q2_K = 2,
    QMM_FP8_E4M3 = 80
} qmm_format;

/* Element type of an embedding lookup's output. */
typedef enum { QMM_OUT_F32 = 0, QMM_OUT_BF16 = 1 } qmm_out_dtype;

/* Element type of the unquantized source of qmm_quantize.  BF16 is the ISQ
 * source (model weights); F32 lets tests feed values that bf16 cannot hold. */
typedef enum { QMM_SRC_BF16 = 0, QMM_SRC_F32 = 1 } qmm_src_dtype;

typedef enum {
    QMM_OK = 0,
    QMM_ERR_INVALID_ARG = -1, /* NULL pointer, negative size, unknown enum  */
    QMM_ERR_UNSUPPORTED = -2, /* valid request this build does not handle   */
    QMM_ERR_SHAPE = -3,       /* cols / K not a positive multiple of 256     */
    QMM_ERR_ALIGNMENT = -4,   /* a pointer is not 16-byte aligned            */
    QMM_ERR_WORKSPACE = -5,   /* workspace missing or smaller than required  */
    QMM_ERR_CUDA = -6,        /* the CUDA runtime reported an error          */
    QMM_ERR_DEVICE = -7       /* a kernel recorded an internal error (below) */
} qmm_status;

/* Bytes of a packed [rows x cols] matrix; 0 if the format is unknown, a size
 * is negative, or cols is not a multiple of the format's block (32 / 256). */
QMM_API size_t qmm_packed_bytes(qmm_format fmt, int64_t rows, int64_t cols);

/* ISQ: quantize src[rows x cols] (bf16 bit patterns or fp32, per `st`) into
 * dst_packed (qmm_packed_bytes(fmt, rows, cols) bytes).  Bit-exact and
 * deterministic: the same bytes as the plain CPU definition above (IEEE
 * single arithmetic without contraction, round-half-away codes, binary16
 * round-to-nearest-even scales).  One kernel launch. */
QMM_API qmm_status qmm_quantize(qmm_format fmt, qmm_src_dtype st, const void *src, void *dst_packed,
                        int64_t rows, int64_t cols, qmm_stream_t stream);

/* dst[rows x cols] (fp32) = the dequantized weights of src_packed: Q8_0
 * d * q, Q4_K (d*sc_j) * q - dmin*mc_j (formulas above).  The pages fix only
 * what the formats are (mistral.rs "Quantization types", tables "Q*K family"
 * and "Legacy GGML types"); the values are those of the layouts above.  Every
 * value is exact except the single rounding of Q4_K's final subtraction.
 * src_packed: qmm_packed_bytes(fmt, rows, cols) bytes; dst: rows * cols fp32.
 * One kernel launch. */
QMM_API qmm_status qmm_dequantize(qmm_format fmt, const void *src_packed, float *dst, int64_t rows,
                          int64_t cols, qmm_stream_t stream);

/* Embedding lookup (mistral.rs "Quantization types", section "Sensitive
 * tensor precision": quantized embedding kernels, Q8_0 the common target):
 * out[t][0 .. D) = the dequantized row ids[t] of the packed table
 * table_packed[V x D], for t < T, as fp32 (the exact dequantized values) or
 * bf16 (those values rounded to nearest even).  ids: T int64 token ids in
 * device memory (8-byte aligned); D a positive multiple of 256; table and
 * out 16-byte aligned.  The ids are not read on the host: an id outside
 * 0 .. V-1 writes zeros for that token and records
 * QMM_DEVERR_EMBEDDING_ID (see qmm_device_error_take).  One kernel launch. */
QMM_API qmm_status qmm_embedding(qmm_format fmt, const void *table_packed, const int64_t *ids, int64_t T,
                                 int64_t V, int64_t D, void *out, qmm_out_dtype out_dtype,
                                 qmm_stream_t stream);

/* The format the page's section "Sensitive tensor precision" gives the token
 * embeddings and output head of a model quantized to model_fmt: QMM_Q6_K for
 * Q2_K, Q3_K and Q4_K models, QMM_Q8_0 for Q5_K, Q6_K and Q8_0 models; 0 for
 * any other format.  Host only. */
QMM_API qmm_format qmm_embedding_format(qmm_format model_fmt);

/* Workspace qmm_matmul needs for this problem, in bytes (0 = none; then
 * workspace may be NULL). */
QMM_API size_t qmm_matmul_workspace_bytes(qmm_format fmt, int64_t M, int64_t N, int64_t K);

/* Y[M x N] (fp32, row-major) = X[M x K] (bf16 bit patterns, row-major) times
 * the transpose of the packed weights W[N x K] (qmm_packed_bytes(fmt, N, K)
 * bytes).  The split follows mistral.rs "Quantization types", section
 * "NVFP4" (a dedicated matrix-vector kernel for small decode batches, tiled
 * matrix multiplication for larger ones), and the large-batch kernel converts
 * each weight tile inside the GEMM as that page's section "FP8" describes for
 * W8A16.  M <= 16 runs a decode kernel (except on long rows, K >= 12288,
 * where FP8 and Q5_K from M = 9 and Q8_0 from M = 12 run the tiled kernel,
 * measured faster there): persistent CTAs over 16-row tiles
 * when the tiles fill the GPU (each tile's partial sums added in a fixed
 * order), otherwise split-K over a thread-block cluster reduced in
 * distributed shared memory in a fixed order; both are deterministic.
 * FP8 runs the row-tile decode kernel for M <= 16 (codes converted
 * exactly to binary16 in the MMA fragments, the row scale applied to the
 * finished sums) and the tiled kernel above that (each weight tile converted
 * to binary16 inside the GEMM, the row scale applied in the epilogue).
 * Q5_K runs the row-tile decode kernel for M <= 16 (5-bit codes exactly in
 * the MMA fragments, Q4_K's scale and min handling) and the tiled kernel
 * above.  Q6_K (output heads) runs a CUDA-core kernel for every M: a warp
 * per weight row, exact integer codes times the activations, the sub-block
 * scale applied per superblock, fp32 sums.  Q3_K and Q2_K run a CUDA-core
 * kernel: a warp per weight row, exact codes with the sub-block scale and
 * min applied once per superblock at one token, each weight dequantized
 * exactly (one fp32 rounding, as qmm_dequantize gives it) for more tokens,
 * fp32 products with the activations exact (no binary16 rounding).  For
 * Q8_0 / Q4_K / Q5_K, larger M runs
 * the tiled kernel (tcgen05 tensor cores, TMEM accumulators):
 * token tiles of 32, 64, 128 or 256 (the smallest of 32 / 64 / 128 that holds
 * M, else 256).  When the output tiles are fewer than the SMs, K is split:
 * 256-token tiles into two halves added onto a zeroed Y, smaller tiles into
 * parts whose partial tiles the last part to finish adds in part order.  From
 * four waves of 256-token tiles, each CTA takes an equal run of K work and a
 * tile cut between two CTAs is the sum of both parts on a zeroed Y.  Two
 * additions onto zero commute, so every result is deterministic.
 *
 * Accuracy, per element, with w^ the dequantized weights:
 *   |y - y_exact| <= 1e-3 * sum_k |w^_k x_k| + 1e-6 + 2^-25 * T,
 * where T = sum over k of |x_k| for the weights with |w^_k| < 2^-14 (prefill
 * path, M > 16, only) plus |w^_k| for the activations with |x_k| < 2^-14 (both
 * paths; the CUDA-core kernels of Q6_K, Q3_K and Q2_K have no T term).  Both paths round each activation to binary16
 * once, and the prefill path also rounds each dequantized weight to
 * binary16 once: a relative error
 * of at most 2^-11 for values in binary16's normal range, an absolute error
 * of at most 2^-25 below it.  T is 0 when no such values occur; for the
 * synthetic weights and activations of the tests it is negligible.
 * `workspace` must hold qmm_matmul_workspace_bytes(fmt, M, N, K) bytes (or be
 * NULL when that is 0): the tiled path keeps the binary16 copy of X there
 * and, with a K split, the partial tiles and their tickets (cleared by the
 * call itself).  The size depends on the current device's SM count.  It is
 * only read and written by this call's kernels. */
QMM_API qmm_status qmm_matmul(qmm_format fmt, const void *W_packed, const uint16_t *X_bf16, float *Y,
                      int64_t M, int64_t N, int64_t K, void *workspace, size_t workspace_bytes,
                      qmm_stream_t stream);

/* Prefill matmul (M > 16) that allocates nothing, for callers that cannot
 * allocate device memory: code handed only raw tensor pointers by a host
 * framework, engines whose pool owns all device memory, loops that must not
 * call cudaMalloc because it can synchronise the device.  It computes what
 * qmm_matmul computes, with the same kernels, but its scratch (the binary16
 * copy of X and, with a K split, the partial tiles) lives in a fixed 64 MiB
 * device array inside this library, held by every GPU that loads the library
 * until the process exits.  The pages
 * describe no counterpart of this call; it is an interface convenience.
 *  - Requires qmm_matmul_workspace_bytes(fmt, M, N, K) <= 64 MiB (M * K
 *    somewhat below 32 Mi); larger problems return QMM_ERR_WORKSPACE and
 *    launch nothing.  M <= 16 and Q6_K return QMM_ERR_UNSUPPORTED:
 *    those paths need no scratch, call qmm_matmul with a NULL workspace.
 *  - Every call looks up the array's address in the current device's
 *    context (cudaGetSymbolAddress), so it stays valid after a device reset.
 *    The first call on a device may load the library's device code: make
 *    that first call before any stream capture.
 *  - All calls share the one array: calls whose executions overlap on the
 *    GPU (different streams, or different host threads on one device) race
 *    on it.  Serialise them, e.g. on one stream.  Nothing in the array needs
 *    to start at zero. */
QMM_API qmm_status qmm_matmul_prefill_static(qmm_format fmt, const void *W_packed,
                                             const uint16_t *X_bf16, float *Y, int64_t M,
                                             int64_t N, int64_t K, qmm_stream_t stream);

/* Static description of a status code (never NULL). */
QMM_API const char *qmm_status_string(qmm_status s);

/* Codes a kernel records in the device error word (qmm_device_error_take). */
typedef enum {
    QMM_DEVERR_NONE = 0,
    QMM_DEVERR_GEMV_FULL_WAIT = 101,   /* decode: waited too long for a stage */
    QMM_DEVERR_GEMV_EMPTY_WAIT = 102,  /* decode: waited too long for a free slot */
    QMM_DEVERR_GEMM_WAIT = 201,        /* prefill: a pipeline wait ran out */
    QMM_DEVERR_EMBEDDING_ID = 301,     /* qmm_embedding: an id outside 0 .. V-1 */
    QMM_DEVERR_SELFTEST_TIMEOUT = 901, /* qmm_selftest_bounded_wait: expected */
    QMM_DEVERR_SELFTEST_UNEXPECTED = 902
} qmm_device_error;

/* Kernels never trap.  A wait inside a kernel that exceeds its time limit
 * (about two seconds; it can only happen through a bug) makes the kernel
 * record a nonzero code (qmm_device_error; the first one recorded is kept) in
 * a device word and return early.  This call synchronises the current device,
 * returns that code (0 = none) and clears it; -1 if the synchronisation or
 * the copy of the word failed. */
QMM_API int qmm_device_error_take(void);

/* Diagnostic (no counterpart on the pages): runs the bounded-wait path that
 * every kernel's pipeline waits use, on one warp: a wait on a completed
 * barrier (must succeed) and then one on a barrier that nothing arrives on,
 * which must give up after limit_ns nanoseconds (1 .. 1e8), record
 * QMM_DEVERR_SELFTEST_TIMEOUT and return.  Nothing faults and no copy is in
 * flight.  The next qmm_device_error_take() then returns 901 and the device
 * stays usable.  Returns QMM_ERR_INVALID_ARG for a limit out of range. */
QMM_API qmm_status qmm_selftest_bounded_wait(int64_t limit_ns, qmm_stream_t stream);

/* Library version, e.g. "qmm 0.2.0 sm_103a". */
QMM_API const char *qmm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* QMM_H */
