// gemm.cu -- prefill-shaped quantized matmul (M > 16).  Placeholder until the
// tcgen05 kernel lands: reports "not supported".
#include "common.cuh"

namespace qmm {

size_t gemm_workspace_bytes(int fmt, int M, int N, int K) {
    (void)fmt; (void)M; (void)N; (void)K;
    return 0;
}

cudaError_t launch_gemm(int fmt, const void *W, const uint16_t *X, float *Y, int M, int N, int K,
                        void *workspace, size_t workspace_bytes, int sms, cudaStream_t stream) {
    (void)fmt; (void)W; (void)X; (void)Y; (void)M; (void)N; (void)K; (void)workspace;
    (void)workspace_bytes; (void)sms; (void)stream;
    return cudaErrorNotSupported;
}

}  // namespace qmm
