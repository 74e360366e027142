// qmm_api.cu -- the C ABI declared in include/qmm.h: argument checks on the
// host, kernel selection and launch.  Nothing here allocates or synchronises
// (except qmm_device_error_take, which is documented to synchronise).
#include <atomic>
#include <cstdint>
#include <cstring>

#include "common.cuh"
#include "qmm.h"

namespace qmm {

cudaError_t launch_quantize(int fmt, int src_f32, const void *src, void *dst, int64_t nweights,
                            int sms, cudaStream_t stream);
cudaError_t launch_dequantize(int fmt, const void *src, float *dst, int64_t nweights, int sms,
                              cudaStream_t stream);
cudaError_t launch_gemv(int fmt, const void *W, const uint16_t *X, float *Y, int M, int N, int K,
                        int sms, cudaStream_t stream);
cudaError_t launch_gemv_rows(int fmt, const void *W, const uint16_t *X, float *Y, int M, int N,
                             int K, int sms, cudaStream_t stream);
cudaError_t launch_gemm(int fmt, const void *W, const uint16_t *X, float *Y, int M, int N, int K,
                        void *workspace, size_t workspace_bytes, int sms, cudaStream_t stream);
size_t gemm_workspace_bytes(int fmt, int M, int N, int K, int sms);
cudaError_t launch_q6k_quantize(int src_f32, const void *src, void *dst, int64_t nweights, int sms,
                                cudaStream_t stream);
cudaError_t launch_q6k_dequantize(const void *src, float *dst, int64_t nweights, int sms, cudaStream_t stream);
cudaError_t launch_q6k_matmul(const void *W, const uint16_t *X, float *Y, int M, int N, int K, int sms,
                              cudaStream_t stream);
cudaError_t launch_embedding(int fmt, const void *table, const int64_t *ids, void *out, int bf16, int64_t T,
                             int64_t V, int64_t D, int sms, cudaStream_t stream);
cudaError_t launch_fp8_quantize(int src_f32, const void *src, void *dst, int64_t rows, int64_t K, int sms,
                                cudaStream_t stream);
cudaError_t launch_fp8_dequantize(const void *src, float *dst, int64_t rows, int64_t K, int sms,
                                  cudaStream_t stream);
cudaError_t launch_kq_quantize(int fmt, int src_f32, const void *src, void *dst, int64_t nweights, int sms,
                               cudaStream_t stream);
cudaError_t launch_kq_dequantize(int fmt, const void *src, float *dst, int64_t nweights, int sms,
                                 cudaStream_t stream);
cudaError_t launch_kq_matmul(int fmt, const void *W, const uint16_t *X, float *Y, int M, int N, int K, int sms,
                             cudaStream_t stream);
cudaError_t launch_kq_embedding(int fmt, const void *table, const int64_t *ids, void *out, int bf16, int64_t T,
                                int64_t V, int64_t D, int sms, cudaStream_t stream);
bool sbrows_supported(int fmt, int M, int K);
cudaError_t launch_sbrows(int fmt, const void *W, const uint16_t *X, float *Y, int N, int K, int sms,
                          cudaStream_t stream);

constexpr int kMaxDecodeM = 16;

// The tiled (tcgen05) kernel's batches: above 16 tokens, and from 9 tokens
// on long rows (K >= 12288, where 9-16 tokens of activations no longer stay
// resident in a decode CTA) for FP8 and Q5_K, from 12 for Q8_0 (4096 x 14336
// on a B300: the tiled kernel 25.6 / 30.7 / 26.3 us against the decode
// kernels' 29.5-40.3 / 37.1-57.6 / 30.2 at 9-16 tokens).  Q4_K stays on the
// decode kernels (even there); Q6_K, Q3_K, Q2_K have no tiled kernel.
static bool tiled_batch(qmm_format fmt, int64_t M, int64_t K) {
    if (fmt == QMM_Q6_K || fmt == QMM_Q3_K || fmt == QMM_Q2_K) return false;
    if (M > kMaxDecodeM) return true;
    if (K < 12288) return false;
    if (fmt == QMM_FP8_E4M3 || fmt == QMM_Q5_K) return M >= 9;
    return fmt == QMM_Q8_0 && M >= 12;
}
// Largest dimension accepted (keeps every 32-bit index in the kernels exact).
constexpr int64_t kMaxDim = (int64_t)1 << 30;

// SMs of the current device, looked up once per device (calls may come
// from several host threads: the cache is atomic).
static int sm_count() {
    static std::atomic<int> cached[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    if (dev < 0 || dev >= 64) return 148;
    int n = cached[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 148;
        cached[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

#ifndef QMM_ROWS_MAX_M
#define QMM_ROWS_MAX_M 16
#endif
#ifndef QMM_ROWS_MIN_CTAS_PER_SM  // in 1/4 CTA per SM
#define QMM_ROWS_MIN_CTAS_PER_SM 4
#endif
// Decode kernel choice: 16-row CTAs over the whole K (no cluster) when the
// tokens are few and the rows alone give every SM enough CTAs; otherwise the
// 64-row tile with a cluster split-K.
// The persistent row-tile kernel when its 16-row tiles fill the SMs; with
// more than 8 tokens only while the activations stay resident in shared
// memory (M * K / 256 <= 256: restaging 16 token rows per tile costs more
// than the cluster kernel's windows).
static bool use_rows_kernel(int M, int N, int K, int sms) {
    if (M > QMM_ROWS_MAX_M || (M > 8 && (int64_t)M * (K / 256) > 256)) return false;
    const int64_t tiles = (N + 15) / 16;
    if (tiles * 4 >= (int64_t)sms * QMM_ROWS_MIN_CTAS_PER_SM) return true;
    // with 1-2 tokens, tiles on a quarter of the SMs still beat the cluster
    // kernel's fixed costs (1024 x 4096: 4.4 -> 3.7 us at M = 1)
    return M <= 2 && tiles * 4 >= (int64_t)sms;
}

static bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
static bool known_fmt(qmm_format f) {
    return f == QMM_Q8_0 || f == QMM_Q4_K || f == QMM_Q6_K || f == QMM_FP8_E4M3 || f == QMM_Q5_K || f == QMM_Q3_K ||
           f == QMM_Q2_K;
}
// Q5_K / Q3_K / Q2_K: the CUDA-core kernels of kquant.cu
static bool is_kq(qmm_format f) { return f == QMM_Q5_K || f == QMM_Q3_K || f == QMM_Q2_K; }
static int64_t block_weights(qmm_format f) { return f == QMM_Q8_0 ? kQ8Weights : 256; }
static int64_t block_bytes(qmm_format f) {
    switch (f) {
    case QMM_Q8_0: return kQ8Bytes;
    case QMM_Q4_K: return kQ4Bytes;
    case QMM_Q5_K: return 176;
    case QMM_Q3_K: return 110;
    case QMM_Q2_K: return 84;
    default: return 210;  // Q6_K
    }
}

static qmm_status from_cuda(cudaError_t e) { return e == cudaSuccess ? QMM_OK : QMM_ERR_CUDA; }

// Self-test of the bounded-wait path that every kernel's mbarrier waits use:
// one warp waits on a barrier that has completed (must succeed) and then on
// one that nothing ever arrives on (must give up after limit_ns, record
// kErrSelftestTimeout and return).  No copy is in flight, nothing faults.
__global__ void __launch_bounds__(32) qmm_selftest_wait_kernel(uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bars[2];
    const uint32_t done = smem_addr(&bars[0]), never = smem_addr(&bars[1]);
    if (threadIdx.x == 0) {
        mbar_init(done, 1);
        mbar_init(never, 1);
        fence_mbar_init();
        mbar_arrive(done);  // completes phase 0 of `done`
    }
    __syncwarp();
    if (threadIdx.x == 0) {
        if (mbar_wait_limit(done, 0, kErrSelftestUnexpected, limit_ns))
            mbar_wait_limit(never, 0, kErrSelftestTimeout, limit_ns);
    }
}

}  // namespace qmm

using namespace qmm;

extern "C" {

size_t qmm_packed_bytes(qmm_format fmt, int64_t rows, int64_t cols) {
    if (!known_fmt(fmt) || rows < 0 || cols < 0) return 0;
    if (rows > kMaxDim || cols > kMaxDim) return 0;
    if (fmt == QMM_FP8_E4M3)  // K codes, the fp32 row scale, 12 zero bytes
        return cols % kGroup == 0 && cols > 0 ? (size_t)(rows * (cols + kFp8RowPad)) : 0;
    const int64_t qk = block_weights(fmt);
    const int64_t bb = block_bytes(fmt);
    if (cols % qk != 0) return 0;
    return (size_t)(rows * (cols / qk) * bb);
}

qmm_status qmm_quantize(qmm_format fmt, qmm_src_dtype st, const void *src, void *dst_packed,
                        int64_t rows, int64_t cols, qmm_stream_t stream) {
    if (!known_fmt(fmt) || (st != QMM_SRC_BF16 && st != QMM_SRC_F32)) return QMM_ERR_INVALID_ARG;
    if (rows < 0 || cols < 0 || rows > kMaxDim || cols > kMaxDim) return QMM_ERR_INVALID_ARG;
    if (cols == 0 || cols % kGroup != 0) return QMM_ERR_SHAPE;
    if (rows == 0) return QMM_OK;
    if (src == nullptr || dst_packed == nullptr) return QMM_ERR_INVALID_ARG;
    if (!aligned16(src) || !aligned16(dst_packed)) return QMM_ERR_ALIGNMENT;
    if (fmt == QMM_Q6_K)
        return from_cuda(launch_q6k_quantize(st == QMM_SRC_F32, src, dst_packed, rows * cols, sm_count(),
                                             reinterpret_cast<cudaStream_t>(stream)));
    if (fmt == QMM_FP8_E4M3)
        return from_cuda(launch_fp8_quantize(st == QMM_SRC_F32, src, dst_packed, rows, cols, sm_count(),
                                             reinterpret_cast<cudaStream_t>(stream)));
    if (is_kq(fmt))
        return from_cuda(launch_kq_quantize((int)fmt, st == QMM_SRC_F32, src, dst_packed, rows * cols, sm_count(),
                                            reinterpret_cast<cudaStream_t>(stream)));
    return from_cuda(launch_quantize((int)fmt, st == QMM_SRC_F32, src, dst_packed, rows * cols,
                                     sm_count(), reinterpret_cast<cudaStream_t>(stream)));
}

qmm_status qmm_dequantize(qmm_format fmt, const void *src_packed, float *dst, int64_t rows,
                          int64_t cols, qmm_stream_t stream) {
    if (!known_fmt(fmt)) return QMM_ERR_INVALID_ARG;
    if (rows < 0 || cols < 0 || rows > kMaxDim || cols > kMaxDim) return QMM_ERR_INVALID_ARG;
    if (cols == 0 || cols % kGroup != 0) return QMM_ERR_SHAPE;
    if (rows == 0) return QMM_OK;
    if (src_packed == nullptr || dst == nullptr) return QMM_ERR_INVALID_ARG;
    if (!aligned16(src_packed) || !aligned16(dst)) return QMM_ERR_ALIGNMENT;
    if (fmt == QMM_Q6_K)
        return from_cuda(launch_q6k_dequantize(src_packed, dst, rows * cols, sm_count(),
                                               reinterpret_cast<cudaStream_t>(stream)));
    if (fmt == QMM_FP8_E4M3)
        return from_cuda(launch_fp8_dequantize(src_packed, dst, rows, cols, sm_count(),
                                               reinterpret_cast<cudaStream_t>(stream)));
    if (is_kq(fmt))
        return from_cuda(launch_kq_dequantize((int)fmt, src_packed, dst, rows * cols, sm_count(),
                                              reinterpret_cast<cudaStream_t>(stream)));
    return from_cuda(launch_dequantize((int)fmt, src_packed, dst, rows * cols, sm_count(),
                                       reinterpret_cast<cudaStream_t>(stream)));
}

size_t qmm_matmul_workspace_bytes(qmm_format fmt, int64_t M, int64_t N, int64_t K) {
    if (!known_fmt(fmt) || M <= 0 || !tiled_batch(fmt, M, K) || N <= 0 || K <= 0 || M > kMaxDim ||
        N > kMaxDim || K > kMaxDim || K % kGroup != 0)
        return 0;
    return gemm_workspace_bytes((int)fmt, (int)M, (int)N, (int)K, sm_count());
}

qmm_status qmm_matmul(qmm_format fmt, const void *W_packed, const uint16_t *X_bf16, float *Y,
                      int64_t M, int64_t N, int64_t K, void *workspace, size_t workspace_bytes,
                      qmm_stream_t stream) {
    if (!known_fmt(fmt)) return QMM_ERR_INVALID_ARG;
    if (M < 0 || N < 0 || K < 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim)
        return QMM_ERR_INVALID_ARG;
    if (K == 0 || K % kGroup != 0) return QMM_ERR_SHAPE;
    if (M == 0 || N == 0) return QMM_OK;
    if (W_packed == nullptr || X_bf16 == nullptr || Y == nullptr) return QMM_ERR_INVALID_ARG;
    if (!aligned16(W_packed) || !aligned16(X_bf16) || !aligned16(Y)) return QMM_ERR_ALIGNMENT;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // one token, Q6_K / Q3_K / Q2_K: TMA-fed CUDA-core kernel where the rows
    // are 16-byte multiples; otherwise direct loads
    if (sbrows_supported((int)fmt, (int)M, (int)K))
        return from_cuda(launch_sbrows((int)fmt, W_packed, X_bf16, Y, (int)N, (int)K, sm_count(), s));
    if (fmt == QMM_Q6_K)
        return from_cuda(launch_q6k_matmul(W_packed, X_bf16, Y, (int)M, (int)N, (int)K, sm_count(), s));
    // Q5_K runs the row-tile decode kernel and the tiled kernel (its
    // superblocks are 16-byte aligned, so TMA boxes fit); Q3_K / Q2_K on CUDA cores
    const bool tiled = tiled_batch(fmt, M, K);
    if (fmt == QMM_Q5_K && !tiled)
        return from_cuda(launch_gemv_rows((int)fmt, W_packed, X_bf16, Y, (int)M, (int)N, (int)K, sm_count(), s));
    if (fmt == QMM_Q3_K || fmt == QMM_Q2_K)
        return from_cuda(launch_kq_matmul((int)fmt, W_packed, X_bf16, Y, (int)M, (int)N, (int)K, sm_count(), s));
    if (!tiled) {
        // FP8 has only the row-tile decode kernel
        if (fmt == QMM_FP8_E4M3 || use_rows_kernel((int)M, (int)N, (int)K, sm_count()))
            return from_cuda(launch_gemv_rows((int)fmt, W_packed, X_bf16, Y, (int)M, (int)N, (int)K,
                                              sm_count(), s));
        return from_cuda(launch_gemv((int)fmt, W_packed, X_bf16, Y, (int)M, (int)N, (int)K,
                                     sm_count(), s));
    }
    const size_t need = gemm_workspace_bytes((int)fmt, (int)M, (int)N, (int)K, sm_count());
    if (need > 0 && (workspace == nullptr || workspace_bytes < need)) return QMM_ERR_WORKSPACE;
    if (need > 0 && !aligned16(workspace)) return QMM_ERR_ALIGNMENT;
    return from_cuda(launch_gemm((int)fmt, W_packed, X_bf16, Y, (int)M, (int)N, (int)K, workspace,
                                 workspace_bytes, sm_count(), s));
}

const char *qmm_status_string(qmm_status s) {
    switch (s) {
    case QMM_OK: return "ok";
    case QMM_ERR_INVALID_ARG: return "invalid argument (null pointer, negative size or unknown enum)";
    case QMM_ERR_UNSUPPORTED: return "unsupported request";
    case QMM_ERR_SHAPE: return "cols / K / D must be a positive multiple of 256";
    case QMM_ERR_ALIGNMENT: return "pointers must be 16-byte aligned";
    case QMM_ERR_WORKSPACE: return "workspace missing or too small";
    case QMM_ERR_CUDA: return "CUDA runtime error";
    case QMM_ERR_DEVICE: return "a kernel recorded an internal error";
    }
    return "unknown status";
}

int qmm_device_error_take(void) {
    if (cudaDeviceSynchronize() != cudaSuccess) return -1;
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(int)) != cudaSuccess) return -1;
    if (v != 0) {
        const int zero = 0;
        if (cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int)) != cudaSuccess) return -1;
    }
    return v;
}

qmm_status qmm_embedding(qmm_format fmt, const void *table_packed, const int64_t *ids, int64_t T, int64_t V,
                         int64_t D, void *out, qmm_out_dtype out_dtype, qmm_stream_t stream) {
    if (!known_fmt(fmt) || (out_dtype != QMM_OUT_F32 && out_dtype != QMM_OUT_BF16)) return QMM_ERR_INVALID_ARG;
    if (T < 0 || V < 0 || D < 0 || T > kMaxDim || V > kMaxDim || D > kMaxDim) return QMM_ERR_INVALID_ARG;
    if (D == 0 || D % kGroup != 0) return QMM_ERR_SHAPE;
    if (T == 0) return QMM_OK;
    if (V == 0 || table_packed == nullptr || ids == nullptr || out == nullptr) return QMM_ERR_INVALID_ARG;
    if (!aligned16(table_packed) || !aligned16(out) || (reinterpret_cast<uintptr_t>(ids) & 7u) != 0)
        return QMM_ERR_ALIGNMENT;
    if (is_kq(fmt))
        return from_cuda(launch_kq_embedding((int)fmt, table_packed, ids, out, out_dtype == QMM_OUT_BF16, T, V, D,
                                             sm_count(), reinterpret_cast<cudaStream_t>(stream)));
    return from_cuda(launch_embedding((int)fmt, table_packed, ids, out, out_dtype == QMM_OUT_BF16, T, V, D,
                                      sm_count(), reinterpret_cast<cudaStream_t>(stream)));
}

qmm_format qmm_embedding_format(qmm_format model_fmt) {
    // "Sensitive tensor precision": Q2K-Q4K models keep their embeddings and
    // output head in Q6K, Q5K / Q6K / Q8_0 models in Q8_0
    if (model_fmt == QMM_Q2_K || model_fmt == QMM_Q3_K || model_fmt == QMM_Q4_K) return QMM_Q6_K;
    if (model_fmt == QMM_Q5_K || model_fmt == QMM_Q6_K || model_fmt == QMM_Q8_0) return QMM_Q8_0;
    return (qmm_format)0;
}

qmm_status qmm_selftest_bounded_wait(int64_t limit_ns, qmm_stream_t stream) {
    if (limit_ns <= 0 || limit_ns > 100000000) return QMM_ERR_INVALID_ARG;
    qmm_selftest_wait_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>((uint64_t)limit_ns);
    return from_cuda(cudaGetLastError());
}

const char *qmm_version(void) { return "qmm 0.3.0 sm_103a"; }

}  // extern "C"
