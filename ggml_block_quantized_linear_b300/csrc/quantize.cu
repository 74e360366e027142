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
// -> 144 bytes.  ISQ gives each lane one 32-weight (sub-)block, loaded with
// 16-byte loads; Q4_K superblock statistics are reduced over 8 lanes with
// shuffles; the packed output is assembled in shared memory and written
// back with coalesced 16-byte stores.  Dequantization runs one warp per
// 256-weight group.  The kernels are HBM-bound:
// per weight they move 2 bytes in and 1.0625 (Q8_0) or 0.5625 (Q4_K) out.
//
// Bit-exactness: every floating-point step is an explicit IEEE single
// operation (__fdiv_rn, __fadd_rn, __fsub_rn, __fmul_rn: no contraction),
// codes use round-half-away (roundf), scales use binary16 round-to-nearest-
// even (__float2half_rn).  Divisions by the constants 15, 63, 127 use an
// FMA-corrected product that equals the IEEE quotient (div_const); a
// quotient that is only rounded to an integer (a weight code, a 6-bit scale
// code) uses an approximate reciprocal and falls back to the IEEE division
// only next to a rounding tie (round_quotient), which gives the same codes.
// Signed zeros cannot change a byte: the maxima that feed a scale are
// forced to +0 when they are zero.
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

// roundf(x / D) for D > 0, bit-identical to roundf(__fdiv_rn(x, D)), from
// a reciprocal r of D within 1 ulp (the hardware approximation rcp_approx).
// t = x * r (rounded) is within (2^-23 + 2^-24) |Q| of Q = x / D, and the
// correctly rounded quotient within 2^-24 |Q|; roundf only jumps at
// half-integers, so the nearest integer k of t is the answer unless t lies
// within 4 * 2^-24 * 128 < 2^-14 of a half-integer (|Q| <= 128), where the
// exact division decides.  Callers clamp the result to a range inside
// [-128, 128]: beyond it, both ways clamp to the same code.
//
// The block quantizers apply this per block: every code takes the fast
// path, the largest |t - k| of the block is kept, and only a block where it
// reaches 0.5 - 2^-14 (a possible tie) is recomputed with exact divisions --
// one branch per block instead of one per weight.
__device__ __forceinline__ float rcp_approx(float d) {
    float r;
    asm("rcp.approx.f32 %0, %1;" : "=f"(r) : "f"(d));
    return r;
}

// x / c for a constant c > 0 and x >= 0, correctly rounded: Markstein's
// correction of the product with the rounded reciprocal r = RN(1/c)
// (P. Markstein, IBM J. Res. Dev. 34(1), 1990): q0 = x r, e = x - c q0
// (exact by fma), q = q0 + e r rounded once.  Checked bit for bit against
// the IEEE division for every non-negative finite float and c = 15, 63, 127.
template <int kC>
__device__ __forceinline__ float div_const(float x) {
    constexpr float c = (float)kC;
    constexpr float r = 1.0f / (float)kC;
    const float q0 = __fmul_rn(x, r);
    const float q = __fmaf_rn(__fmaf_rn(-q0, c, x), r, q0);
    return isinf(q0) ? q0 : q;  // x = inf: the residual would be inf - inf
}

constexpr float kTieGuard = 0.49993896484375f;  // 0.5 - 2^-14
__device__ __forceinline__ float rint_quotient(float x, float r, float &dev) {
    const float t = __fmul_rn(x, r);
    const float k = rintf(t);
    dev = fmaxf(dev, fabsf(__fsub_rn(t, k)));
    return k;
}
__device__ __forceinline__ float round_quotient(float x, float D, float r) {
    const float t = __fmul_rn(x, r);
    const float k = rintf(t);
    if (fabsf(__fsub_rn(t, k)) >= kTieGuard) return roundf(__fdiv_rn(x, D));
    return k;
}

// Byte of an integral float in [-128, 127] (two's complement): adding
// 1.5 * 2^23 moves the integer into the low mantissa bits.
__device__ __forceinline__ uint32_t int_byte(float v) {
    return __float_as_uint(__fadd_rn(v, 12582912.0f)) & 0xFFu;
}
// Four integral floats in [-128, 127] -> one word of bytes (v0 lowest).
__device__ __forceinline__ uint32_t pack4_bytes(float v0, float v1, float v2, float v3) {
    const uint32_t a = __float_as_uint(__fadd_rn(v0, 12582912.0f));
    const uint32_t b = __float_as_uint(__fadd_rn(v1, 12582912.0f));
    const uint32_t c = __float_as_uint(__fadd_rn(v2, 12582912.0f));
    const uint32_t d = __float_as_uint(__fadd_rn(v3, 12582912.0f));
    return prmt(prmt(a, b, 0x0040u), prmt(c, d, 0x0040u), 0x5410u);
}

template <bool kSrcF32>
__device__ __forceinline__ void load32(const void *src, int64_t elem, float (&x)[32]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float v[8];
        load8<kSrcF32>(src, elem + 8 * i, v);
#pragma unroll
        for (int e = 0; e < 8; ++e) x[8 * i + e] = v[e];
    }
}

// ------------------------------------------------------------------ Q8_0
// One lane quantizes one 32-weight block; a warp covers 32 consecutive
// blocks (1024 weights, 1088 packed bytes) per iteration, assembled in
// shared memory and stored with coalesced 16-byte writes.
template <bool kSrcF32>
__global__ void __launch_bounds__(kQuantThreads)
quantize_q8_0_kernel(const void *__restrict__ src, uint8_t *__restrict__ dst, int64_t nblocks) {
    __shared__ __align__(16) uint8_t stage[kQuantWarps][32 * kQ8Bytes];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint8_t *st = stage[warp];
    const int64_t nwarps = (int64_t)gridDim.x * kQuantWarps;
    for (int64_t b0 = ((int64_t)blockIdx.x * kQuantWarps + warp) * 32; b0 < nblocks; b0 += nwarps * 32) {
        const int64_t blk = b0 + lane;
        const int nvalid = (int)min((int64_t)32, nblocks - b0);  // a multiple of 8
        if (blk < nblocks) {
            float x[32];
            load32<kSrcF32>(src, blk * kQ8Weights, x);
            float amax = 0.0f;
#pragma unroll
            for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(x[i]));
            const __half dh = __float2half_rn(div_const<127>(amax));
            const float df = __half2float(dh);
            uint32_t w[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) w[i] = 0u;
            if (df >= 6.103515625e-05f) {
                // normal binary16 scale: |x / d16| <= 127 (1 + 2^-11) < 127.5,
                // so round(x / d16) never needs the clamp
                const float r = rcp_approx(df);
                float dev = 0.0f;
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    w[i] = pack4_bytes(rint_quotient(x[4 * i], r, dev), rint_quotient(x[4 * i + 1], r, dev),
                                       rint_quotient(x[4 * i + 2], r, dev), rint_quotient(x[4 * i + 3], r, dev));
                if (dev >= kTieGuard) {  // a possible tie: exact divisions for the block
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        w[i] = pack4_bytes(roundf(__fdiv_rn(x[4 * i], df)), roundf(__fdiv_rn(x[4 * i + 1], df)),
                                           roundf(__fdiv_rn(x[4 * i + 2], df)), roundf(__fdiv_rn(x[4 * i + 3], df)));
                }
            } else if (df != 0.0f) {  // subnormal scale: the quotient may pass 127.5
                const float r = rcp_approx(df);
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const float q = clamp_f(round_quotient(x[i], df, r), -127.0f, 127.0f);
                    w[i >> 2] |= int_byte(q) << (8 * (i & 3));
                }
            }
            uint16_t *o = reinterpret_cast<uint16_t *>(st + kQ8Bytes * lane);
            o[0] = __half_as_ushort(dh);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                o[1 + 2 * i] = (uint16_t)w[i];
                o[2 + 2 * i] = (uint16_t)(w[i] >> 16);
            }
        }
        __syncwarp();
        const int nvec = nvalid * kQ8Bytes / 16;
        uint4 *out = reinterpret_cast<uint4 *>(dst + b0 * kQ8Bytes);
        for (int v = lane; v < nvec; v += 32) out[v] = reinterpret_cast<const uint4 *>(st)[v];
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
// ------------------------------------------------------------------ Q4_K
// One lane quantizes one 32-weight sub-block; 8 lanes make a superblock and
// a warp covers 4 superblocks (1024 weights, 576 packed bytes) per
// iteration.
#ifndef QMM_Q4_QUANT_MIN_BLOCKS  // resident CTAs per SM the register budget must allow
#define QMM_Q4_QUANT_MIN_BLOCKS 4
#endif
template <bool kSrcF32>
__global__ void __launch_bounds__(kQuantThreads, QMM_Q4_QUANT_MIN_BLOCKS)
quantize_q4_k_kernel(const void *__restrict__ src, uint8_t *__restrict__ dst, int64_t nsuper) {
    __shared__ __align__(16) uint8_t stage[kQuantWarps][4 * kQ4Bytes];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int sj = lane & 7, sbl = lane >> 3;  // sub-block j, superblock in the warp tile
    uint8_t *st = stage[warp] + sbl * kQ4Bytes;
    const int64_t nwarps = (int64_t)gridDim.x * kQuantWarps;
    for (int64_t s0 = ((int64_t)blockIdx.x * kQuantWarps + warp) * 4; s0 < nsuper; s0 += nwarps * 4) {
        const int64_t sb = s0 + sbl;
        const bool valid = sb < nsuper;  // uniform over each group of 8 lanes
        const int nvalid = (int)min((int64_t)4, nsuper - s0);
        float x[32];
        float mx, mn;  // max_i x_i and min(0, min_i x_i)
        if constexpr (kSrcF32) {
            if (valid) load32<kSrcF32>(src, sb * kQ4Weights + sj * 32, x);
            else {
#pragma unroll
                for (int i = 0; i < 32; ++i) x[i] = 0.0f;
            }
            mx = x[0];
            mn = 0.0f;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                mx = fmaxf(mx, x[i]);
                mn = fminf(mn, x[i]);
            }
        } else {
            // bf16 source: the extremes on packed pairs (exact, NaN-skipping
            // like fmaxf / fminf), then the conversion to fp32
            uint32_t raw[16];
            const uint4 *src4 = reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(src) +
                                                                sb * kQ4Weights + sj * 32);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint4 v = valid ? __ldg(src4 + i) : make_uint4(0u, 0u, 0u, 0u);
                raw[4 * i] = v.x;
                raw[4 * i + 1] = v.y;
                raw[4 * i + 2] = v.z;
                raw[4 * i + 3] = v.w;
            }
            __nv_bfloat162 vmax = *reinterpret_cast<const __nv_bfloat162 *>(&raw[0]), vmin = vmax;
#pragma unroll
            for (int i = 1; i < 16; ++i) {
                const __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162 *>(&raw[i]);
                vmax = __hmax2(vmax, v);
                vmin = __hmin2(vmin, v);
            }
            mx = fmaxf(__low2float(vmax), __high2float(vmax));
            mn = fminf(0.0f, fminf(__low2float(vmin), __high2float(vmin)));
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                x[2 * i] = __uint_as_float(raw[i] << 16);
                x[2 * i + 1] = __uint_as_float(raw[i] & 0xFFFF0000u);
            }
        }
        const float s = div_const<15>(__fsub_rn(mx, mn));
        const float m = __fsub_rn(0.0f, mn);
        float smax = s, mmax = m;
#pragma unroll
        for (int o = 1; o <= 4; o <<= 1) {
            smax = fmaxf(smax, __shfl_xor_sync(0xffffffffu, smax, o));
            mmax = fmaxf(mmax, __shfl_xor_sync(0xffffffffu, mmax, o));
        }
        smax = smax > 0.0f ? smax : 0.0f;
        mmax = mmax > 0.0f ? mmax : 0.0f;
        const __half dh = __float2half_rn(div_const<63>(smax));
        const __half dminh = __float2half_rn(div_const<63>(mmax));
        const float df = __half2float(dh), dminf = __half2float(dminh);
        // 6-bit codes of the scale and the min: s / d16 and m / dmin16 are at
        // most ~64, so the reciprocal quotient with the tie check applies
        float tsc = 0.0f, tmc = 0.0f, sdev = 0.0f;
        if (df > 0.0f) tsc = rint_quotient(s, rcp_approx(df), sdev);
        if (dminf > 0.0f) tmc = rint_quotient(m, rcp_approx(dminf), sdev);
        if (sdev >= kTieGuard) {
            tsc = df > 0.0f ? roundf(__fdiv_rn(s, df)) : 0.0f;
            tmc = dminf > 0.0f ? roundf(__fdiv_rn(m, dminf)) : 0.0f;
        }
        const int sc = (int)clamp_f(tsc, 0.0f, 63.0f);
        const int mc = (int)clamp_f(tmc, 0.0f, 63.0f);
        const float S = __fmul_rn(df, (float)sc);
        const float Mn = __fmul_rn(dminf, (float)mc);
        uint32_t w[8];  // 4-bit codes, one per byte
#pragma unroll
        for (int i = 0; i < 8; ++i) w[i] = 0u;
        if (S > 0.0f) {
            const float r = rcp_approx(S);
            float dev = 0.0f;
            auto code = [&](int i) { return clamp_f(rint_quotient(__fadd_rn(x[i], Mn), r, dev), 0.0f, 15.0f); };
#pragma unroll
            for (int i = 0; i < 8; ++i)
                w[i] = pack4_bytes(code(4 * i), code(4 * i + 1), code(4 * i + 2), code(4 * i + 3));
            if (dev >= kTieGuard) {  // a possible tie: exact divisions for the sub-block
                auto exact = [&](int i) { return clamp_f(roundf(__fdiv_rn(__fadd_rn(x[i], Mn), S)), 0.0f, 15.0f); };
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    w[i] = pack4_bytes(exact(4 * i), exact(4 * i + 1), exact(4 * i + 2), exact(4 * i + 3));
            }
        }
        // sub-block 2c (low nibbles) and 2c+1 (high nibbles) share chunk c
        uint32_t hw[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) hw[i] = __shfl_xor_sync(0xffffffffu, w[i], 1);
        // scale bytes: j < 4 writes s[j], s[j+4], s[j+8] with the codes of j+4
        const int sc4 = __shfl_down_sync(0xffffffffu, sc, 4);
        const int mc4 = __shfl_down_sync(0xffffffffu, mc, 4);
        if (valid) {
            if ((sj & 1) == 0) {
                uint4 *o = reinterpret_cast<uint4 *>(st + 16 + 32 * (sj >> 1));
                o[0] = make_uint4(w[0] | (hw[0] << 4), w[1] | (hw[1] << 4), w[2] | (hw[2] << 4),
                                  w[3] | (hw[3] << 4));
                o[1] = make_uint4(w[4] | (hw[4] << 4), w[5] | (hw[5] << 4), w[6] | (hw[6] << 4),
                                  w[7] | (hw[7] << 4));
            }
            if (sj < 4) {
                st[4 + sj] = (uint8_t)(sc | ((sc4 >> 4) << 6));
                st[8 + sj] = (uint8_t)(mc | ((mc4 >> 4) << 6));
                st[12 + sj] = (uint8_t)((sc4 & 15) | ((mc4 & 15) << 4));
            }
            if (sj == 0)
                *reinterpret_cast<uint32_t *>(st) =
                    (uint32_t)__half_as_ushort(dh) | ((uint32_t)__half_as_ushort(dminh) << 16);
        }
        __syncwarp();
        const int nvec = nvalid * kQ4Bytes / 16;
        uint4 *out = reinterpret_cast<uint4 *>(dst + s0 * kQ4Bytes);
        for (int v = lane; v < nvec; v += 32) out[v] = reinterpret_cast<const uint4 *>(stage[warp])[v];
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
static int grid_for(int64_t items, int per_cta, int sms) {
    int64_t want = (items + per_cta - 1) / per_cta;
    int64_t cap = (int64_t)sms * 8;  // 8 resident CTAs of 256 threads per SM
    return (int)(want < cap ? (want > 0 ? want : 1) : cap);
}

cudaError_t launch_quantize(int fmt, int src_f32, const void *src, void *dst, int64_t nweights,
                            int sms, cudaStream_t stream) {
    if (nweights == 0) return cudaSuccess;
    uint8_t *d = static_cast<uint8_t *>(dst);
    if (fmt == 8) {
        const int64_t nblocks = nweights / kQ8Weights;
        const int grid = grid_for(nblocks, 32 * kQuantWarps, sms);
        if (src_f32)
            quantize_q8_0_kernel<true><<<grid, kQuantThreads, 0, stream>>>(src, d, nblocks);
        else
            quantize_q8_0_kernel<false><<<grid, kQuantThreads, 0, stream>>>(src, d, nblocks);
    } else {
        const int64_t nsuper = nweights / kQ4Weights;
        const int grid = grid_for(nsuper, 4 * kQuantWarps, sms);
        if (src_f32)
            quantize_q4_k_kernel<true><<<grid, kQuantThreads, 0, stream>>>(src, d, nsuper);
        else
            quantize_q4_k_kernel<false><<<grid, kQuantThreads, 0, stream>>>(src, d, nsuper);
    }
    return cudaGetLastError();
}

cudaError_t launch_dequantize(int fmt, const void *src, float *dst, int64_t nweights, int sms,
                              cudaStream_t stream) {
    const int64_t ngroups = nweights / kGroup;
    if (ngroups == 0) return cudaSuccess;
    const int grid = grid_for(ngroups, kQuantWarps, sms);
    const uint8_t *s = static_cast<const uint8_t *>(src);
    if (fmt == 8)
        dequantize_q8_0_kernel<<<grid, kQuantThreads, 0, stream>>>(s, dst, ngroups);
    else
        dequantize_q4_k_kernel<<<grid, kQuantThreads, 0, stream>>>(s, dst, ngroups);
    return cudaGetLastError();
}

}  // namespace qmm
