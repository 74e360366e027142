// quantize.cu -- ISQ (in-situ quantization) of bf16 / fp32 weights into Q8_0
// and Q4_K blocks, and exact dequantization back to fp32.
//
// ISQ is the load-time quantization of the mistral.rs documentation page
// "Quantization types" (opening section; CUDA resolves `--isq 8` to Q8_0 and
// `--isq 4` to Q4K, section "Numeric shorthands").  The block formulas and
// byte layouts are the library's reading given in include/qmm.h.
//
// Both formats are processed in groups of 256 consecutive weights of the
// flattened row-major matrix (cols is a multiple of 256, so a group never
// straddles two rows): 8 Q8_0 blocks -> 272 bytes, or one Q4_K superblock
// -> 144 bytes.  One warp handles one group per iteration: every lane loads
// 8 consecutive weights with 16-byte loads, block statistics are reduced
// with warp shuffles, the packed group is assembled in shared memory and
// written back with coalesced 16-byte stores.  The kernels are HBM-bound:
// per weight they move 2 bytes in and 1.0625 (Q8_0) or 0.5625 (Q4_K) out.
//
// Bit-exactness: every floating-point step is an explicit IEEE single
// operation (__fdiv_rn, __fadd_rn, __fsub_rn, __fmul_rn: no contraction),
// codes use round-half-away (roundf), scales use binary16 round-to-nearest-
// even (__float2half_rn).  Signed zeros cannot change a byte: the maxima
// that feed a scale are forced to +0 when they are zero.
#include "common.cuh"

namespace qmm {

constexpr int kQuantThreads = 256;
constexpr int kQuantWarps = kQuantThreads / 32;

template <bool kSrcF32>
__device__ __forceinline__ void load8(const void *src, int64_t elem, float (&x)[8]) {
    if (kSrcF32) {
        const float4 *p = reinterpret_cast<const float4 *>(static_cast<const float *>(src) + elem);
        float4 a = __ldg(p), b = __ldg(p + 1);
        x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
        x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
    } else {
        uint4 v = __ldg(reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(src) + elem));
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            x[2 * i] = __uint_as_float(w[i] << 16);
            x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
    }
}

__device__ __forceinline__ float clamp_f(float v, float lo, float hi) {
    return v < lo ? lo : (v > hi ? hi : v);
}

// ------------------------------------------------------------------ Q8_0
template <bool kSrcF32>
__global__ void __launch_bounds__(kQuantThreads)
quantize_q8_0_kernel(const void *__restrict__ src, uint8_t *__restrict__ dst, int64_t ngroups) {
    __shared__ __align__(16) uint8_t stage[kQuantWarps][kQ8GroupBytes];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int blk = lane >> 2, part = lane & 3;
    uint8_t *st = stage[warp];
    const int64_t nwarps = (int64_t)gridDim.x * kQuantWarps;
    for (int64_t g = (int64_t)blockIdx.x * kQuantWarps + warp; g < ngroups; g += nwarps) {
        float x[8];
        load8<kSrcF32>(src, g * kGroup + lane * 8, x);
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(x[i]));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
        const float d = __fdiv_rn(amax, 127.0f);
        const __half dh = __float2half_rn(d);
        const float df = __half2float(dh);
        uint32_t packed[2] = {0u, 0u};
        if (df != 0.0f) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float q = clamp_f(roundf(__fdiv_rn(x[i], df)), -127.0f, 127.0f);
                packed[i >> 2] |= (uint32_t)((uint8_t)(int8_t)(int)q) << (8 * (i & 3));
            }
        }
        // 8 codes at byte 34*blk + 2 + 8*part (2-byte aligned)
        uint16_t *q16 = reinterpret_cast<uint16_t *>(st + kQ8Bytes * blk + 2 + 8 * part);
        q16[0] = (uint16_t)packed[0];
        q16[1] = (uint16_t)(packed[0] >> 16);
        q16[2] = (uint16_t)packed[1];
        q16[3] = (uint16_t)(packed[1] >> 16);
        if (part == 0) *reinterpret_cast<uint16_t *>(st + kQ8Bytes * blk) = __half_as_ushort(dh);
        __syncwarp();
        if (lane < kQ8GroupBytes / 16)
            reinterpret_cast<uint4 *>(dst + g * kQ8GroupBytes)[lane] =
                reinterpret_cast<const uint4 *>(st)[lane];
        __syncwarp();
    }
}

__global__ void __launch_bounds__(kQuantThreads)
dequantize_q8_0_kernel(const uint8_t *__restrict__ src, float *__restrict__ dst, int64_t ngroups) {
    __shared__ __align__(16) uint8_t stage[kQuantWarps][kQ8GroupBytes];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int blk = lane >> 2, part = lane & 3;
    uint8_t *st = stage[warp];
    const int64_t nwarps = (int64_t)gridDim.x * kQuantWarps;
    for (int64_t g = (int64_t)blockIdx.x * kQuantWarps + warp; g < ngroups; g += nwarps) {
        if (lane < kQ8GroupBytes / 16)
            reinterpret_cast<uint4 *>(st)[lane] =
                __ldg(reinterpret_cast<const uint4 *>(src + g * kQ8GroupBytes) + lane);
        __syncwarp();
        const float df =
            __half2float(__ushort_as_half(*reinterpret_cast<const uint16_t *>(st + kQ8Bytes * blk)));
        const uint16_t *q16 = reinterpret_cast<const uint16_t *>(st + kQ8Bytes * blk + 2 + 8 * part);
        float y[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint16_t h = q16[i];
            y[2 * i] = __fmul_rn(df, (float)(int8_t)(h & 0xFF));
            y[2 * i + 1] = __fmul_rn(df, (float)(int8_t)(h >> 8));
        }
        __syncwarp();
        float4 *out = reinterpret_cast<float4 *>(dst + g * kGroup + lane * 8);
        out[0] = make_float4(y[0], y[1], y[2], y[3]);
        out[1] = make_float4(y[4], y[5], y[6], y[7]);
    }
}

// ------------------------------------------------------------------ Q4_K
template <bool kSrcF32>
__global__ void __launch_bounds__(kQuantThreads)
quantize_q4_k_kernel(const void *__restrict__ src, uint8_t *__restrict__ dst, int64_t ngroups) {
    __shared__ __align__(16) uint8_t stage[kQuantWarps][kQ4Bytes];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int sub = lane >> 2, part = lane & 3;  // sub-block j, 8-weight slice
    uint8_t *st = stage[warp];
    const int64_t nwarps = (int64_t)gridDim.x * kQuantWarps;
    for (int64_t g = (int64_t)blockIdx.x * kQuantWarps + warp; g < ngroups; g += nwarps) {
        float x[8];
        load8<kSrcF32>(src, g * kGroup + lane * 8, x);
        float mx = x[0], mn = 0.0f;  // max_i x_i and min(0, min_i x_i)
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            mx = fmaxf(mx, x[i]);
            mn = fminf(mn, x[i]);
        }
#pragma unroll
        for (int o = 1; o <= 2; o <<= 1) {
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
        }
        const float s = __fdiv_rn(__fsub_rn(mx, mn), 15.0f);
        const float m = __fsub_rn(0.0f, mn);
        float smax = s, mmax = m;
#pragma unroll
        for (int o = 4; o <= 16; o <<= 1) {
            smax = fmaxf(smax, __shfl_xor_sync(0xffffffffu, smax, o));
            mmax = fmaxf(mmax, __shfl_xor_sync(0xffffffffu, mmax, o));
        }
        smax = smax > 0.0f ? smax : 0.0f;
        mmax = mmax > 0.0f ? mmax : 0.0f;
        const __half dh = __float2half_rn(__fdiv_rn(smax, 63.0f));
        const __half dminh = __float2half_rn(__fdiv_rn(mmax, 63.0f));
        const float df = __half2float(dh), dminf = __half2float(dminh);
        const int sc = df > 0.0f ? (int)clamp_f(roundf(__fdiv_rn(s, df)), 0.0f, 63.0f) : 0;
        const int mc = dminf > 0.0f ? (int)clamp_f(roundf(__fdiv_rn(m, dminf)), 0.0f, 63.0f) : 0;
        const float S = __fmul_rn(df, (float)sc);
        const float Mn = __fmul_rn(dminf, (float)mc);
        uint32_t w[2] = {0u, 0u};
        if (S > 0.0f) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float q = clamp_f(roundf(__fdiv_rn(__fadd_rn(x[i], Mn), S)), 0.0f, 15.0f);
                w[i >> 2] |= (uint32_t)(int)q << (8 * (i & 3));
            }
        }
        // sub-block 2c (low nibbles) and 2c+1 (high nibbles) share chunk c
        const uint32_t h0 = __shfl_xor_sync(0xffffffffu, w[0], 4);
        const uint32_t h1 = __shfl_xor_sync(0xffffffffu, w[1], 4);
        if ((sub & 1) == 0) {
            uint2 v = make_uint2(w[0] | (h0 << 4), w[1] | (h1 << 4));
            *reinterpret_cast<uint2 *>(st + 16 + 32 * (sub >> 1) + 8 * part) = v;
        }
        // gather the eight (sc, mc) pairs into lane 0 and pack the header
        uint32_t code = (uint32_t)sc | ((uint32_t)mc << 8);
        uint32_t codes[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) codes[j] = __shfl_sync(0xffffffffu, code, 4 * j);
        if (lane == 0) {
            uint8_t sb[12];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint32_t scj = codes[j] & 0xFF, mcj = codes[j] >> 8;
                const uint32_t sch = codes[j + 4] & 0xFF, mch = codes[j + 4] >> 8;
                sb[j] = (uint8_t)(scj | ((sch >> 4) << 6));
                sb[j + 4] = (uint8_t)(mcj | ((mch >> 4) << 6));
                sb[j + 8] = (uint8_t)((sch & 15) | ((mch & 15) << 4));
            }
            uint4 hdr;
            hdr.x = (uint32_t)__half_as_ushort(dh) | ((uint32_t)__half_as_ushort(dminh) << 16);
            hdr.y = sb[0] | (sb[1] << 8) | (sb[2] << 16) | ((uint32_t)sb[3] << 24);
            hdr.z = sb[4] | (sb[5] << 8) | (sb[6] << 16) | ((uint32_t)sb[7] << 24);
            hdr.w = sb[8] | (sb[9] << 8) | (sb[10] << 16) | ((uint32_t)sb[11] << 24);
            *reinterpret_cast<uint4 *>(st) = hdr;
        }
        __syncwarp();
        if (lane < kQ4Bytes / 16)
            reinterpret_cast<uint4 *>(dst + g * kQ4Bytes)[lane] =
                reinterpret_cast<const uint4 *>(st)[lane];
        __syncwarp();
    }
}

// 6-bit scale / min codes of sub-block j from the 12 scale bytes s[].
__device__ __forceinline__ void q4k_codes(const uint8_t *s, int j, int &sc, int &mc) {
    if (j < 4) {
        sc = s[j] & 63;
        mc = s[j + 4] & 63;
    } else {
        sc = (s[j + 4] & 15) | ((s[j - 4] >> 6) << 4);
        mc = (s[j + 4] >> 4) | ((s[j] >> 6) << 4);
    }
}

__global__ void __launch_bounds__(kQuantThreads)
dequantize_q4_k_kernel(const uint8_t *__restrict__ src, float *__restrict__ dst, int64_t ngroups) {
    __shared__ __align__(16) uint8_t stage[kQuantWarps][kQ4Bytes];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int sub = lane >> 2, part = lane & 3;
    uint8_t *st = stage[warp];
    const int64_t nwarps = (int64_t)gridDim.x * kQuantWarps;
    for (int64_t g = (int64_t)blockIdx.x * kQuantWarps + warp; g < ngroups; g += nwarps) {
        if (lane < kQ4Bytes / 16)
            reinterpret_cast<uint4 *>(st)[lane] =
                __ldg(reinterpret_cast<const uint4 *>(src + g * kQ4Bytes) + lane);
        __syncwarp();
        const uint32_t dd = *reinterpret_cast<const uint32_t *>(st);
        const float df = __half2float(__ushort_as_half((uint16_t)(dd & 0xFFFF)));
        const float dminf = __half2float(__ushort_as_half((uint16_t)(dd >> 16)));
        int sc, mc;
        q4k_codes(st + 4, sub, sc, mc);
        const float S = __fmul_rn(df, (float)sc);
        const float Mn = __fmul_rn(dminf, (float)mc);
        const uint2 qv = *reinterpret_cast<const uint2 *>(st + 16 + 32 * (sub >> 1) + 8 * part);
        const int shift = 4 * (sub & 1);
        float y[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t word = i < 4 ? qv.x : qv.y;
            const int q = (word >> (8 * (i & 3) + shift)) & 15;
            y[i] = __fsub_rn(__fmul_rn(S, (float)q), Mn);
        }
        __syncwarp();
        float4 *out = reinterpret_cast<float4 *>(dst + g * kGroup + lane * 8);
        out[0] = make_float4(y[0], y[1], y[2], y[3]);
        out[1] = make_float4(y[4], y[5], y[6], y[7]);
    }
}

// ------------------------------------------------------------- launchers
static int grid_for(int64_t ngroups, int sms) {
    int64_t want = (ngroups + kQuantWarps - 1) / kQuantWarps;
    int64_t cap = (int64_t)sms * 8;  // 8 resident CTAs of 256 threads per SM
    return (int)(want < cap ? (want > 0 ? want : 1) : cap);
}

cudaError_t launch_quantize(int fmt, int src_f32, const void *src, void *dst, int64_t nweights,
                            int sms, cudaStream_t stream) {
    const int64_t ngroups = nweights / kGroup;
    if (ngroups == 0) return cudaSuccess;
    const int grid = grid_for(ngroups, sms);
    uint8_t *d = static_cast<uint8_t *>(dst);
    if (fmt == 8) {
        if (src_f32)
            quantize_q8_0_kernel<true><<<grid, kQuantThreads, 0, stream>>>(src, d, ngroups);
        else
            quantize_q8_0_kernel<false><<<grid, kQuantThreads, 0, stream>>>(src, d, ngroups);
    } else {
        if (src_f32)
            quantize_q4_k_kernel<true><<<grid, kQuantThreads, 0, stream>>>(src, d, ngroups);
        else
            quantize_q4_k_kernel<false><<<grid, kQuantThreads, 0, stream>>>(src, d, ngroups);
    }
    return cudaGetLastError();
}

cudaError_t launch_dequantize(int fmt, const void *src, float *dst, int64_t nweights, int sms,
                              cudaStream_t stream) {
    const int64_t ngroups = nweights / kGroup;
    if (ngroups == 0) return cudaSuccess;
    const int grid = grid_for(ngroups, sms);
    const uint8_t *s = static_cast<const uint8_t *>(src);
    if (fmt == 8)
        dequantize_q8_0_kernel<<<grid, kQuantThreads, 0, stream>>>(s, dst, ngroups);
    else
        dequantize_q4_k_kernel<<<grid, kQuantThreads, 0, stream>>>(s, dst, ngroups);
    return cudaGetLastError();
}

}  // namespace qmm
