// fp8.cu -- FP8 E4M3 weights with a scale per row: ISQ and dequantization.
//
// mistral.rs, "Quantization types", section "FP8": E4M3 FP8 can be produced
// with ISQ, and W8A16 keeps the E4M3 weights resident and converts each
// weight tile to BF16 / F16 inside the GEMM (the tiled kernel in gemm.cu
// does that; the decode kernel in gemv_rows.cu converts its MMA fragments).
// The scale layout is this library's reading of the page's "channel" weight
// scales: one fp32 scale per output row, s = max |x| / 448, codes
// E4M3(x / s) rounded to nearest even and saturated at +-448.  A packed row
// is K codes, s, 12 zero bytes (K + 16 bytes, so rows stay 16-byte aligned).
#include "common.cuh"

namespace qmm {

constexpr int kFp8Threads = 256;

// Four floats -> four E4M3 codes (round to nearest even, saturating).
__device__ __forceinline__ uint32_t f32x4_to_e4m3x4(float a, float b, float c, float d) {
    const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
    const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
    return (lo & 0xFFFFu) | (hi << 16);
}

template <bool kSrcF32>
__device__ __forceinline__ void fp8_load8(const void *src, int64_t idx, float (&x)[8]) {
    if constexpr (kSrcF32) {
        const float4 *p = reinterpret_cast<const float4 *>(static_cast<const float *>(src) + idx);
        const float4 v0 = __ldg(p), v1 = __ldg(p + 1);
        x[0] = v0.x; x[1] = v0.y; x[2] = v0.z; x[3] = v0.w;
        x[4] = v1.x; x[5] = v1.y; x[6] = v1.z; x[7] = v1.w;
    } else {
        const uint4 v = __ldg(reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(src) + idx));
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            x[2 * e] = __uint_as_float(w[e] << 16);
            x[2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
        }
    }
}

// One CTA per row (grid-stride): the row's largest magnitude, then the codes.
template <bool kSrcF32>
__global__ void __launch_bounds__(kFp8Threads) qmm_quantize_fp8_kernel(const void *__restrict__ src,
                                                                       uint8_t *__restrict__ dst, int64_t rows,
                                                                       int64_t K) {
    __shared__ float red[kFp8Threads / 32];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t rb = K + kFp8RowPad;
    for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
        float amax = 0.f;
        for (int64_t k = 8 * (int64_t)tid; k < K; k += 8 * kFp8Threads) {
            float x[8];
            fp8_load8<kSrcF32>(src, r * K + k, x);
#pragma unroll
            for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(x[e]));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        if (lane == 0) red[warp] = amax;
        __syncthreads();
        amax = red[0];
#pragma unroll
        for (int w = 1; w < kFp8Threads / 32; ++w) amax = fmaxf(amax, red[w]);
        __syncthreads();  // red is rewritten for the next row
        const float s = __fdiv_rn(amax, 448.0f);
        uint8_t *out = dst + r * rb;
        for (int64_t k = 8 * (int64_t)tid; k < K; k += 8 * kFp8Threads) {
            float x[8];
            fp8_load8<kSrcF32>(src, r * K + k, x);
            uint2 q = make_uint2(0u, 0u);
            if (s > 0.f) {
                float y[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) y[e] = __fdiv_rn(x[e], s);
                q = make_uint2(f32x4_to_e4m3x4(y[0], y[1], y[2], y[3]), f32x4_to_e4m3x4(y[4], y[5], y[6], y[7]));
            }
            *reinterpret_cast<uint2 *>(out + k) = q;
        }
        if (tid == 0) *reinterpret_cast<uint4 *>(out + K) = make_uint4(__float_as_uint(s), 0u, 0u, 0u);
    }
}

// 8 weights per thread: value * row scale (one fp32 rounding).
__global__ void __launch_bounds__(kFp8Threads) qmm_dequantize_fp8_kernel(const uint8_t *__restrict__ src,
                                                                         float *__restrict__ dst, int64_t rows,
                                                                         int64_t K) {
    const int64_t per_row = K / 8, total = rows * per_row;
    const int64_t rb = K + kFp8RowPad;
    for (int64_t i = (int64_t)blockIdx.x * kFp8Threads + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * kFp8Threads) {
        const int64_t r = i / per_row, k = 8 * (i - r * per_row);
        const uint8_t *row = src + r * rb;
        const float s = __ldg(reinterpret_cast<const float *>(row + K));
        const uint2 q = __ldg(reinterpret_cast<const uint2 *>(row + k));
        const uint32_t w[2] = {q.x, q.y};
        float v[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const uint32_t h2 = e4m3x2_to_h2(w[e >> 1] >> (16 * (e & 1)));
            v[2 * e] = __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu))) * s;
            v[2 * e + 1] = __half2float(__ushort_as_half((unsigned short)(h2 >> 16))) * s;
        }
        float4 *y = reinterpret_cast<float4 *>(dst + r * K + k);
        y[0] = make_float4(v[0], v[1], v[2], v[3]);
        y[1] = make_float4(v[4], v[5], v[6], v[7]);
    }
}

static int fp8_grid(int64_t units, int sms) {
    const int64_t cap = (int64_t)sms * 8;
    int64_t g = units < cap ? units : cap;
    return g < 1 ? 1 : (int)g;
}

cudaError_t launch_fp8_quantize(int src_f32, const void *src, void *dst, int64_t rows, int64_t K, int sms,
                                cudaStream_t stream) {
    const int grid = fp8_grid(rows, sms);
    uint8_t *d = static_cast<uint8_t *>(dst);
    if (src_f32)
        qmm_quantize_fp8_kernel<true><<<grid, kFp8Threads, 0, stream>>>(src, d, rows, K);
    else
        qmm_quantize_fp8_kernel<false><<<grid, kFp8Threads, 0, stream>>>(src, d, rows, K);
    return cudaGetLastError();
}

cudaError_t launch_fp8_dequantize(const void *src, float *dst, int64_t rows, int64_t K, int sms,
                                  cudaStream_t stream) {
    const int grid = fp8_grid((rows * (K / 8) + kFp8Threads - 1) / kFp8Threads, sms);
    qmm_dequantize_fp8_kernel<<<grid, kFp8Threads, 0, stream>>>(static_cast<const uint8_t *>(src), dst, rows, K);
    return cudaGetLastError();
}

}  // namespace qmm
