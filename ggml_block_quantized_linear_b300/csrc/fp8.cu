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
#include <atomic>

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

// E4M3 codes of x / s for 8 weights (s > 0, rs = rcp_approx(s)), identical
// to converting the IEEE quotient RN(x / s): y = RN(x rs) is within
// 2^-22 |y| of it (rs within an ulp of 1 / s, two roundings), so RN(x / s)
// lies between y (1 - 2^-21) and y (1 + 2^-21).  The conversion (round to
// nearest even, saturating) is monotone, so when both ends give the same
// code that is the code; otherwise (an E4M3 rounding boundary within the
// interval) the pair is converted from the IEEE quotient.
__device__ __forceinline__ uint32_t fp8_codes4(const float (&x)[8], int o, float s, float rs) {
    uint32_t out = 0;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const float a = x[o + 2 * h], b = x[o + 2 * h + 1];
        const float ya = __fmul_rn(a, rs), yb = __fmul_rn(b, rs);
        const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(__fmul_rn(ya, 0.99999952316284180f),
                                                                 __fmul_rn(yb, 0.99999952316284180f)),
                                                     __NV_SATFINITE, __NV_E4M3);
        const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(__fmul_rn(ya, 1.00000047683715820f),
                                                                 __fmul_rn(yb, 1.00000047683715820f)),
                                                     __NV_SATFINITE, __NV_E4M3);
        uint32_t c = lo & 0xFFFFu;
        if (c != (hi & 0xFFFFu))
            c = __nv_cvt_float2_to_fp8x2(make_float2(__fdiv_rn(a, s), __fdiv_rn(b, s)), __NV_SATFINITE, __NV_E4M3) &
                0xFFFFu;
        out |= c << (16 * h);
    }
    return out;
}

// Rows staged in shared memory: each CTA takes rows b, b + G, ...; one bulk
// copy brings a whole row (K bf16 or fp32 values) into one of nbuf buffers
// while the rows before it are quantized from the others, so every weight is
// read from memory once and nbuf - 1 row copies stay in flight.
template <bool kSrcF32>
__global__ void __launch_bounds__(kFp8Threads) qmm_quantize_fp8_staged_kernel(const void *__restrict__ src,
                                                                              uint8_t *__restrict__ dst,
                                                                              int64_t rows, int64_t K, int nbuf) {
    constexpr int kE = kSrcF32 ? 4 : 2;
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ float red[kFp8Threads / 32];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t rowb = (uint32_t)(K * kE);
    const uint32_t bar0 = smem_addr(smem + nbuf * rowb);
    const int64_t rb = K + kFp8RowPad;
    const char *srcb = static_cast<const char *>(src);
    if (tid == 0) {
        for (int b = 0; b < nbuf; ++b) mbar_init(bar0 + 8u * b, 1);
        fence_mbar_init();
    }
    __syncthreads();
    // the first nbuf - 1 rows
    if (tid == 0)
        for (int j = 0; j < nbuf - 1; ++j) {
            const int64_t rj = blockIdx.x + (int64_t)j * gridDim.x;
            if (rj >= rows) break;
            mbar_arrive_expect_tx(bar0 + 8u * j, rowb);
            bulk_g2s(smem_addr(smem + j * rowb), srcb + rj * rowb, rowb, bar0 + 8u * j);
        }
    bool ok = true;
    int i = 0;
    for (int64_t r = blockIdx.x; r < rows; r += gridDim.x, ++i) {
        const int b = i % nbuf;
        // the buffer of row i - 1 was last read in the previous iteration
        // (closed by its final __syncthreads): bring row i + nbuf - 1 there
        const int64_t rn = r + (int64_t)(nbuf - 1) * gridDim.x;
        if (tid == 0 && rn < rows) {
            const int bn = (i + nbuf - 1) % nbuf;
            mbar_arrive_expect_tx(bar0 + 8u * bn, rowb);
            bulk_g2s(smem_addr(smem + bn * rowb), srcb + rn * rowb, rowb, bar0 + 8u * bn);
        }
        if (ok) ok = mbar_wait(bar0 + 8u * b, (i / nbuf) & 1, kErrGemvFullWait);
        const uint8_t *row = smem + b * rowb;
        auto load8 = [&](int64_t k, float (&x)[8]) {
            if constexpr (kSrcF32) {
                const float4 v0 = *reinterpret_cast<const float4 *>(row + 4 * k);
                const float4 v1 = *reinterpret_cast<const float4 *>(row + 4 * k + 16);
                x[0] = v0.x; x[1] = v0.y; x[2] = v0.z; x[3] = v0.w;
                x[4] = v1.x; x[5] = v1.y; x[6] = v1.z; x[7] = v1.w;
            } else {
                const uint4 v = *reinterpret_cast<const uint4 *>(row + 2 * k);
                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    x[2 * e] = __uint_as_float(w[e] << 16);
                    x[2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
                }
            }
        };
        float amax = 0.f;
        if (ok)
            for (int64_t k = 8 * (int64_t)tid; k < K; k += 8 * kFp8Threads) {
                float x[8];
                load8(k, x);
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
        const float s = __fdiv_rn(amax, 448.0f);
        const float rs = s > 0.f ? rcp_approx(s) : 0.f;
        uint8_t *out = dst + r * rb;
        if (ok)
            for (int64_t k = 8 * (int64_t)tid; k < K; k += 8 * kFp8Threads) {
                float x[8];
                load8(k, x);
                uint2 q = make_uint2(0u, 0u);
                if (s > 0.f) q = make_uint2(fp8_codes4(x, 0, s, rs), fp8_codes4(x, 4, s, rs));
                *reinterpret_cast<uint2 *>(out + k) = q;
            }
        if (tid == 0) *reinterpret_cast<uint4 *>(out + K) = make_uint4(__float_as_uint(s), 0u, 0u, 0u);
        __syncthreads();  // buffer b and red are reused
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
    uint8_t *d = static_cast<uint8_t *>(dst);
    // two row buffers (and their barriers) in shared memory, while they fit;
    // more buffers measured slower (fewer resident CTAs: the per-row
    // reduction chain, not the copies, sets the pace)
    const int64_t rowb = K * (src_f32 ? 4 : 2);
    const int nbuf = 2;
    const int64_t smem = nbuf * rowb + 8 * nbuf;
    constexpr int kMaxSmem = 200 * 1024 + 32;  // the attribute covers every size this path launches
    if (smem <= kMaxSmem) {
        static std::atomic<uint64_t> done_f{0}, done_b{0};
        const void *fn = src_f32 ? reinterpret_cast<const void *>(qmm_quantize_fp8_staged_kernel<true>)
                                 : reinterpret_cast<const void *>(qmm_quantize_fp8_staged_kernel<false>);
        cudaError_t e = set_smem_limit_once(fn, kMaxSmem, src_f32 ? done_f : done_b);
        if (e != cudaSuccess) return e;
        int occ = 0;
        e = src_f32 ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, qmm_quantize_fp8_staged_kernel<true>,
                                                                     kFp8Threads, (size_t)smem)
                    : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, qmm_quantize_fp8_staged_kernel<false>,
                                                                     kFp8Threads, (size_t)smem);
        if (e != cudaSuccess) return e;
        const int64_t cap = (int64_t)sms * (occ < 1 ? 1 : occ);
        const int grid = (int)(rows < cap ? rows : cap);
        if (src_f32)
            qmm_quantize_fp8_staged_kernel<true><<<grid, kFp8Threads, (size_t)smem, stream>>>(src, d, rows, K, nbuf);
        else
            qmm_quantize_fp8_staged_kernel<false><<<grid, kFp8Threads, (size_t)smem, stream>>>(src, d, rows, K, nbuf);
        return cudaGetLastError();
    }
    const int grid = fp8_grid(rows, sms);
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
