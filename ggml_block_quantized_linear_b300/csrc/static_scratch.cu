// static_scratch.cu -- qmm_matmul_prefill_static: the prefill matmul for
// callers that cannot allocate device memory.
//
// qmm_matmul's prefill path needs a scratch buffer (the binary16 copy of the
// activations) that the caller normally passes as `workspace`.  Some callers
// cannot provide one: code that runs with no access to a device allocator
// (plugins handed only raw tensor pointers by a host framework), engines
// whose memory pool owns all device memory and forbids side allocations, and
// latency-critical loops that must not call cudaMalloc because it can
// synchronise the device.  This entry point runs the same kernels with the
// scratch in a fixed, file-scope device array instead, so it allocates
// nothing at call time.
#include "common.cuh"
#include "qmm.h"

namespace qmm {

// 64 MiB: enough for M * K <= 32 Mi activations (e.g. 2048 tokens x 14336).
// Every GPU that loads this library holds the array until the process exits.
constexpr size_t kStaticScratchBytes = (size_t)64 << 20;
static __device__ __align__(256) uint8_t g_prefill_scratch[kStaticScratchBytes];

// Device address of g_prefill_scratch in the current device's context (in
// host code the symbol is only a host-side stand-in).  It is looked up on
// every call, not cached: after a device reset the module is loaded again
// and the array may move.
static void *static_scratch_for_current_device(cudaError_t *err) {
    void *p = nullptr;
    *err = cudaGetSymbolAddress(&p, g_prefill_scratch);
    return *err == cudaSuccess ? p : nullptr;
}

}  // namespace qmm

using namespace qmm;

extern "C" qmm_status qmm_matmul_prefill_static(qmm_format fmt, const void *W_packed,
                                                const uint16_t *X_bf16, float *Y, int64_t M,
                                                int64_t N, int64_t K, qmm_stream_t stream) {
    if (!known_fmt(fmt)) return QMM_ERR_INVALID_ARG;
    if (M < 0 || N < 0 || K < 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim)
        return QMM_ERR_INVALID_ARG;
    if (K == 0 || K % kGroup != 0) return QMM_ERR_SHAPE;
    if (M == 0 || N == 0) return QMM_OK;
    // decode (and every Q6_K, Q3_K, Q2_K product) needs no scratch: use qmm_matmul
    if (M <= kMaxDecodeM || fmt == QMM_Q6_K || fmt == QMM_Q3_K || fmt == QMM_Q2_K) return QMM_ERR_UNSUPPORTED;
    if (W_packed == nullptr || X_bf16 == nullptr || Y == nullptr) return QMM_ERR_INVALID_ARG;
    if (!aligned16(W_packed) || !aligned16(X_bf16) || !aligned16(Y)) return QMM_ERR_ALIGNMENT;
    const size_t need = gemm_workspace_bytes((int)fmt, (int)M, (int)N, (int)K, sm_count());
    if (need > kStaticScratchBytes) return QMM_ERR_WORKSPACE;
    cudaError_t e = cudaSuccess;
    void *scratch = static_scratch_for_current_device(&e);
    if (scratch == nullptr) return QMM_ERR_CUDA;
    return from_cuda(launch_gemm((int)fmt, W_packed, X_bf16, Y, (int)M, (int)N, (int)K, scratch,
                                 kStaticScratchBytes, sm_count(),
                                 reinterpret_cast<cudaStream_t>(stream)));
}
