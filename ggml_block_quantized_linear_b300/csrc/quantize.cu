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
// operation (__fdiv_rn, __fadd_rn, __fsub_rn, __fmul_rn or their .f32x2
// pair forms: no contraction), codes use round-half-away (roundf), scales
// use binary16 round-to-nearest-even (__float2half_rn).  Divisions by the
// constants 15, 63, 127 use an FMA-corrected product that equals the IEEE
// quotient (div_const); a quotient that is only rounded to an integer (a
// weight code, a 6-bit scale code) uses an approximate reciprocal and an
// exact division only for the weights next to a rounding tie (round2,
// rint_quotient), which gives the same codes.  Signed zeros cannot change a
// byte: the maxima that feed a scale are forced to +0 when they are zero.
#include "common.cuh"

namespace qmm {

constexpr int kQuantThreads = 256;
constexpr int kQuantWarps = kQuantThreads / 32;

__device__ __forceinline__ float clamp_f(float v, float lo, float hi) {
    return v < lo ? lo : (v > hi ? hi : v);
}

// Reciprocal within 1 ulp (the hardware approximation): for the exact
// product, |x r - x / D| <= 2^-23 |x / D|.
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

// Byte of an integral float in [-128, 127] (two's complement): adding
// 1.5 * 2^23 moves the integer into the low mantissa bits.
constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23
__device__ __forceinline__ uint32_t int_byte(float v) { return __float_as_uint(__fadd_rn(v, kMagic)) & 0xFFu; }

// Byte j (0..3) of word w replaced by the low byte of b.
__device__ __forceinline__ uint32_t set_byte(uint32_t w, int j, uint32_t b) {
    return prmt(w, b, j == 0 ? 0x3214u : j == 1 ? 0x3240u : j == 2 ? 0x3410u : 0x4210u);
}

// roundf(RN(a / D)), D > 0, for a quotient next to the half-step
// h = k + sign(d) / 2, where k is the integer nearest an approximation of
// a / D and d that approximation minus k (|d| close to 1/2; the quotient
// within 1/2 of h).  roundf(q) is the integer on |h|'s far side from zero
// exactly when |q| >= |h|, and RN(|a| / D) >= |h| exactly when |a| / D
// passes the midpoint m between |h| and its float predecessor.  m has an
// odd 25-bit significand, so D m (exact in double: 24 + 25 bits) is never a
// float and the comparison with |a| is strict and exact: no division.
__device__ __forceinline__ float tie_code(float a, float D, float k, float d) {
    const float h = k + copysignf(0.5f, d);                            // exact
    const float ah = fabsf(h);
    const float ulp = ah - __uint_as_float(__float_as_uint(ah) - 1u);  // exact
    const double m = (double)ah - 0.5 * (double)ulp;                   // exact
    const bool far = (double)fabsf(a) > (double)D * m;
    return copysignf(far ? ah + 0.5f : ah - 0.5f, h);
}

// roundf(x / D) for D > 0 and |x / D| <= 128, bit-identical to
// roundf(__fdiv_rn(x, D)): t = RN(x r) is within (2^-23 + 2^-24) |x / D|
// < 2^-15 of x / D, so the nearest integer k of t is the answer unless t
// lies within 2^-14 of a half-integer, where tie_code decides.
constexpr float kTieGuard = 0.49993896484375f;  // 0.5 - 2^-14
__device__ __forceinline__ float round_div(float x, float D) {
    const float t = __fmul_rn(x, rcp_approx(D));
    const float k = rintf(t);
    const float d = __fsub_rn(t, k);
    return fabsf(d) >= kTieGuard ? tie_code(x, D, k, d) : k;
}

// bf16 pair (low half first) -> fp32 pair
__device__ __forceinline__ uint64_t f2_from_bf16x2(uint32_t w) {
    return f2_pack(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

// Weight codes two at a time.  For a quotient Q = a / D and r =
// rcp_approx(D), v = RN(a r + 1.5 * 2^23) is 1.5 * 2^23 plus the integer k
// nearest to the exact product a r, held in the low mantissa bits of v, and
// d = RN(a r - k) is within 2^-25 of a r - k.  A block keeps the codes k
// unless some |d| reaches its guard 0.5 - g; then each flagged weight is
// decided by tie_code (recheck_ties).  Unflagged, |Q - k| < 2^-23 |Q| +
// 2^-25 + 0.5 - g, which is below 0.5 when 2^-23 |Q| + 2^-25 <= g, so k is
// the nearest integer of Q and no rounding tie (where roundf and the
// nearest-even k may differ) goes unflagged.  Q8_0 codes matter for
// |Q| <= 127.5 and Q4_K codes for |Q| <= 15.5 (beyond, both ways clamp to
// the same code): g = 2^-15 and 2^-18.
constexpr float kTieGuardQ8 = 0.499969482421875f;     // 0.5 - 2^-15
constexpr float kTieGuardQ4 = 0.499996185302734375f;  // 0.5 - 2^-18
__device__ __forceinline__ uint64_t round2(uint64_t a, uint64_t r2, float &dev) {
    const uint64_t m2 = f2_pack(kMagic, kMagic);
    const uint64_t v = f2_fma(a, r2, m2);
    const uint64_t d = f2_fma(a, r2, f2_sub(m2, v));  // a r - k
    float d0, d1;
    f2_unpack(d, d0, d1);
    dev = fmaxf(dev, fmaxf(fabsf(d0), fabsf(d1)));
    return v;
}
// Low bytes of the integers carried by two pairs from round2 -> one word
// (first pair's low lane lowest).
__device__ __forceinline__ uint32_t pack4_magic(uint64_t v01, uint64_t v23) {
    return prmt(prmt((uint32_t)v01, (uint32_t)(v01 >> 32), 0x0040u),
                prmt((uint32_t)v23, (uint32_t)(v23 >> 32), 0x0040u), 0x5410u);
}
// Clamp the integers carried by a round2 pair to [lo, hi].
__device__ __forceinline__ uint64_t clamp2(uint64_t v, float lo, float hi) {
    float v0, v1;
    f2_unpack(v, v0, v1);
    return f2_pack(fminf(fmaxf(v0, kMagic + lo), kMagic + hi), fminf(fmaxf(v1, kMagic + lo), kMagic + hi));
}

// The code of weight a / D (D > 0, r = rcp_approx(D)) with round2's
// arithmetic in scalar form (the same correctly rounded operations, so the
// same k), and tie_code where round2 would flag it.
__device__ __forceinline__ float exact_code(float a, float D, float r, float guard) {
    const float k = __fsub_rn(__fmaf_rn(a, r, kMagic), kMagic);
    const float d = __fmaf_rn(a, r, -k);
    return fabsf(d) >= guard ? tie_code(a, D, k, d) : k;
}

// The 32 weights of one lane.  fp32 sources keep 32 floats; bf16 sources
// keep the 16 loaded words (bf16 pairs, lower index in the low half), half
// the registers, and widen a weight or a pair where it is used.
template <bool kSrcF32> struct Lane32;
template <> struct Lane32<true> {
    float x[32];
    __device__ __forceinline__ void load(const void *src, int64_t elem, bool valid) {
        const float4 *p = reinterpret_cast<const float4 *>(static_cast<const float *>(src) + elem);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float4 v = valid ? __ldg(p + i) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            x[4 * i] = v.x;
            x[4 * i + 1] = v.y;
            x[4 * i + 2] = v.z;
            x[4 * i + 3] = v.w;
        }
    }
    __device__ __forceinline__ uint64_t pair(int i) const { return f2_pack(x[i], x[i + 1]); }
    // weight elem + j read from memory (j known only at run time)
    static __device__ __forceinline__ float reload(const void *src, int64_t elem, int j) {
        return __ldg(static_cast<const float *>(src) + elem + j);
    }
    // max_i x_i and min_i x_i (NaN-skipping, like fmaxf / fminf)
    __device__ __forceinline__ void extremes(float &mx, float &mn) const {
        mx = x[0];
        mn = x[0];
#pragma unroll
        for (int i = 1; i < 32; ++i) {
            mx = fmaxf(mx, x[i]);
            mn = fminf(mn, x[i]);
        }
    }
};
template <> struct Lane32<false> {
    uint32_t w[16];
    __device__ __forceinline__ void load(const void *src, int64_t elem, bool valid) {
        const uint4 *p = reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(src) + elem);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint4 v = valid ? __ldg(p + i) : make_uint4(0u, 0u, 0u, 0u);
            w[4 * i] = v.x;
            w[4 * i + 1] = v.y;
            w[4 * i + 2] = v.z;
            w[4 * i + 3] = v.w;
        }
    }
    __device__ __forceinline__ uint64_t pair(int i) const { return f2_from_bf16x2(w[i >> 1]); }
    static __device__ __forceinline__ float reload(const void *src, int64_t elem, int j) {
        return __uint_as_float((uint32_t)__ldg(static_cast<const unsigned short *>(src) + elem + j) << 16);
    }
    // extremes on packed bf16 pairs (exact; NaN-skipping like fmaxf / fminf)
    __device__ __forceinline__ void extremes(float &mx, float &mn) const {
        __nv_bfloat162 vmax = *reinterpret_cast<const __nv_bfloat162 *>(&w[0]), vmin = vmax;
#pragma unroll
        for (int i = 1; i < 16; ++i) {
            const __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162 *>(&w[i]);
            vmax = __hmax2(vmax, v);
            vmin = __hmin2(vmin, v);
        }
        mx = fmaxf(__low2float(vmax), __high2float(vmax));
        mn = fminf(__low2float(vmin), __high2float(vmin));
    }
};

// ------------------------------------------------------------------ Q8_0
// One lane quantizes one 32-weight block; a warp covers 32 consecutive
// blocks (1024 weights, 1088 packed bytes) per iteration, assembled in
// shared memory and stored with coalesced 16-byte writes.
template <bool kSrcF32>
__global__ void __launch_bounds__(kQuantThreads, kSrcF32 ? 3 : 4)
qmm_quantize_q8_0_kernel(const void *__restrict__ src, uint8_t *__restrict__ dst, int64_t nblocks) {
    __shared__ __align__(16) uint8_t stage[kQuantWarps][32 * kQ8Bytes];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint8_t *st = stage[warp];
    const int64_t nwarps = (int64_t)gridDim.x * kQuantWarps;
    // bf16 sources: the next iteration's weights are loaded before this
    // one's are used (fp32 sources have no registers to spare for that)
    const int64_t step = nwarps * 32;
    int64_t b0 = ((int64_t)blockIdx.x * kQuantWarps + warp) * 32;
    Lane32<kSrcF32> Ln;
    if (!kSrcF32 && b0 + lane < nblocks) Ln.load(src, (b0 + lane) * kQ8Weights, true);
    for (; b0 < nblocks; b0 += step) {
        const int64_t blk = b0 + lane;
        const int nvalid = (int)min((int64_t)32, nblocks - b0);  // a multiple of 8
        float df = 0.0f, r = 0.0f;
        bool normal = true, tie = false;
        Lane32<kSrcF32> L;
        if constexpr (kSrcF32) {
            if (blk < nblocks) L.load(src, blk * kQ8Weights, true);
        } else {
            L = Ln;
            if (blk + step < nblocks) Ln.load(src, (blk + step) * kQ8Weights, true);
        }
        if (blk < nblocks) {
            float mx, mn;
            L.extremes(mx, mn);
            float amax = fmaxf(mx, -mn);
            amax = amax > 0.0f ? amax : 0.0f;  // +0 for an all-zero block
            const __half dh = __float2half_rn(div_const<127>(amax));
            df = __half2float(dh);
            uint32_t w[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) w[i] = 0u;
            if (df != 0.0f) {
                // a normal binary16 scale keeps |x / d16| <= 127 (1 + 2^-11)
                // < 127.5, so round(x / d16) needs no clamp; a subnormal one
                // may pass 127.5
                normal = df >= 6.103515625e-05f;
                r = rcp_approx(df);
                const uint64_t r2 = f2_pack(r, r);
                float dev = 0.0f;
                if (normal) {
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        w[i] = pack4_magic(round2(L.pair(4 * i), r2, dev), round2(L.pair(4 * i + 2), r2, dev));
                } else {
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        w[i] = pack4_magic(clamp2(round2(L.pair(4 * i), r2, dev), -127.0f, 127.0f),
                                           clamp2(round2(L.pair(4 * i + 2), r2, dev), -127.0f, 127.0f));
                }
                tie = dev >= kTieGuardQ8;
            }
            // the 34-byte block at byte 34 * lane: an even lane's block starts
            // on a 4-byte boundary, an odd lane's 2 bytes past one; either
            // way 8 aligned words and one 2-byte store
            const bool odd = lane & 1;
            const uint32_t dbits = __half_as_ushort(dh);
            uint8_t *base = st + kQ8Bytes * lane;
            uint32_t *wb = reinterpret_cast<uint32_t *>(base + (odd ? 2 : 0));
            const uint32_t sel = odd ? 0x7654u : 0x5432u;
            uint32_t prev = dbits << 16;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                wb[i] = prmt(prev, w[i], sel);
                prev = w[i];
            }
            *reinterpret_cast<uint16_t *>(base + (odd ? 0 : 32)) = (uint16_t)(odd ? dbits : (w[7] >> 16));
        }
        __syncwarp();
        // blocks with a possible tie: the warp recomputes them one at a time,
        // lane j taking weight j, and overwrites their codes
        for (uint32_t fl = __ballot_sync(0xffffffffu, tie); fl != 0; fl &= fl - 1) {
            const int l = __ffs(fl) - 1;
            const float D = __shfl_sync(0xffffffffu, df, l), rl = __shfl_sync(0xffffffffu, r, l);
            const bool nl = __shfl_sync(0xffffffffu, normal, l);
            float c = exact_code(Lane32<kSrcF32>::reload(src, (b0 + l) * kQ8Weights, lane), D, rl, kTieGuardQ8);
            if (!nl) c = clamp_f(c, -127.0f, 127.0f);
            st[kQ8Bytes * l + 2 + lane] = (uint8_t)int_byte(c);
        }
        __syncwarp();
        const int nvec = nvalid * kQ8Bytes / 16;
        uint4 *out = reinterpret_cast<uint4 *>(dst + b0 * kQ8Bytes);
        for (int v = lane; v < nvec; v += 32) out[v] = reinterpret_cast<const uint4 *>(st)[v];
        __syncwarp();
    }
}

__global__ void __launch_bounds__(kQuantThreads)
qmm_dequantize_q8_0_kernel(const uint8_t *__restrict__ src, float *__restrict__ dst, int64_t ngroups) {
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
// One lane quantizes one 32-weight sub-block; 8 lanes make a superblock and
// a warp covers 4 superblocks (1024 weights, 576 packed bytes) per
// iteration.
#ifndef QMM_Q4_QUANT_MIN_BLOCKS  // resident CTAs per SM the register budget must allow
#define QMM_Q4_QUANT_MIN_BLOCKS 3
#endif
template <bool kSrcF32>
__global__ void __launch_bounds__(kQuantThreads, QMM_Q4_QUANT_MIN_BLOCKS)
qmm_quantize_q4_k_kernel(const void *__restrict__ src, uint8_t *__restrict__ dst, int64_t nsuper) {
    __shared__ __align__(16) uint8_t stage[kQuantWarps][4 * kQ4Bytes];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int sj = lane & 7, sbl = lane >> 3;  // sub-block j, superblock in the warp tile
    uint8_t *st = stage[warp] + sbl * kQ4Bytes;
    const int64_t nwarps = (int64_t)gridDim.x * kQuantWarps;
    // bf16 sources: the next iteration's weights are loaded before this
    // one's are used (fp32 sources have no registers to spare for that)
    const int64_t step = nwarps * 4;
    int64_t s0 = ((int64_t)blockIdx.x * kQuantWarps + warp) * 4;
    Lane32<kSrcF32> Ln;
    if (!kSrcF32) Ln.load(src, (s0 + sbl) * kQ4Weights + sj * 32, s0 + sbl < nsuper);
    for (; s0 < nsuper; s0 += step) {
        const int64_t sb = s0 + sbl;
        const bool valid = sb < nsuper;  // uniform over each group of 8 lanes
        const int nvalid = (int)min((int64_t)4, nsuper - s0);
        Lane32<kSrcF32> L;
        if constexpr (kSrcF32) {
            L.load(src, sb * kQ4Weights + sj * 32, valid);
        } else {
            L = Ln;
            Ln.load(src, (sb + step) * kQ4Weights + sj * 32, sb + step < nsuper);
        }
        float mx, mn;  // max_i x_i and min(0, min_i x_i)
        L.extremes(mx, mn);
        mn = fminf(0.0f, mn);
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
        // most ~64
        const float tsc = df > 0.0f ? round_div(s, df) : 0.0f;
        const float tmc = dminf > 0.0f ? round_div(m, dminf) : 0.0f;
        const int sc = (int)clamp_f(tsc, 0.0f, 63.0f);
        const int mc = (int)clamp_f(tmc, 0.0f, 63.0f);
        const float S = __fmul_rn(df, (float)sc);
        const float Mn = __fmul_rn(dminf, (float)mc);
        uint32_t w[8];  // 4-bit codes, one per byte
#pragma unroll
        for (int i = 0; i < 8; ++i) w[i] = 0u;
        float r = 0.0f;
        bool tie = false;
        if (S > 0.0f) {
            r = rcp_approx(S);
            const uint64_t r2 = f2_pack(r, r), mn2 = f2_pack(Mn, Mn);
            float dev = 0.0f;
            // u = x + Mn rounded as its own step, then the code of u / S.  The
            // codes are monotone in x: when those of the sub-block's extremes
            // lie well inside int16, every code's low 16 bits are the code and
            // the clamp to [0, 15] runs on 16-bit pairs (max(min(c, 15), 0) in
            // one instruction); otherwise it runs on the floats.
            const float khi = __fmul_rn(__fadd_rn(mx, Mn), r), klo = __fmul_rn(__fadd_rn(mn, Mn), r);
            if (khi < 30000.0f && klo > -30000.0f) {
                auto code2 = [&](int i) {
                    const uint64_t v = round2(f2_add(L.pair(i), mn2), r2, dev);
                    return __vimin_s16x2_relu(prmt((uint32_t)v, (uint32_t)(v >> 32), 0x5410u), 0x000F000Fu);
                };
#pragma unroll
                for (int i = 0; i < 8; ++i) w[i] = prmt(code2(4 * i), code2(4 * i + 2), 0x6420u);
            } else {
                auto code2 = [&](int i) { return clamp2(round2(f2_add(L.pair(i), mn2), r2, dev), 0.0f, 15.0f); };
#pragma unroll
                for (int i = 0; i < 8; ++i) w[i] = pack4_magic(code2(4 * i), code2(4 * i + 2));
            }
            tie = valid && dev >= kTieGuardQ4;
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
        // sub-blocks with a possible tie: the warp recomputes them one at a
        // time, lane j taking weight j, and overwrites their nibbles
        for (uint32_t fl = __ballot_sync(0xffffffffu, tie); fl != 0; fl &= fl - 1) {
            const int l = __ffs(fl) - 1, jl = l & 7;
            const float Sl = __shfl_sync(0xffffffffu, S, l), rl = __shfl_sync(0xffffffffu, r, l);
            const float Ml = __shfl_sync(0xffffffffu, Mn, l);
            const float u = __fadd_rn(Lane32<kSrcF32>::reload(src, (s0 + (l >> 3)) * kQ4Weights + jl * 32, lane), Ml);
            const uint32_t c = int_byte(clamp_f(exact_code(u, Sl, rl, kTieGuardQ4), 0.0f, 15.0f));
            uint8_t *q = stage[warp] + (l >> 3) * kQ4Bytes + 16 + 32 * (jl >> 1) + lane;
            *q = (uint8_t)((jl & 1) ? ((*q & 0x0Fu) | (c << 4)) : ((*q & 0xF0u) | c));
            __syncwarp();
        }
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
qmm_dequantize_q4_k_kernel(const uint8_t *__restrict__ src, float *__restrict__ dst, int64_t ngroups) {
    __shared__ __align__(16) uint8_t stage[kQuantWarps][kQ4Bytes];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int sub = lane >> 2, part = lane & 3;
    uint8_t *st = stage[warp];
    const int64_t nwarps = (int64_t)gridDim.x * kQuantWarps;
    // the next group's bytes are loaded before this one is converted
    constexpr int kVec = kQ4Bytes / 16;
    int64_t g = (int64_t)blockIdx.x * kQuantWarps + warp;
    uint4 nx = make_uint4(0u, 0u, 0u, 0u);
    if (g < ngroups && lane < kVec) nx = __ldg(reinterpret_cast<const uint4 *>(src + g * kQ4Bytes) + lane);
    for (; g < ngroups; g += nwarps) {
        if (lane < kVec) reinterpret_cast<uint4 *>(st)[lane] = nx;
        if (g + nwarps < ngroups && lane < kVec)
            nx = __ldg(reinterpret_cast<const uint4 *>(src + (g + nwarps) * kQ4Bytes) + lane);
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
            qmm_quantize_q8_0_kernel<true><<<grid, kQuantThreads, 0, stream>>>(src, d, nblocks);
        else
            qmm_quantize_q8_0_kernel<false><<<grid, kQuantThreads, 0, stream>>>(src, d, nblocks);
    } else {
        const int64_t nsuper = nweights / kQ4Weights;
        const int grid = grid_for(nsuper, 4 * kQuantWarps, sms);
        if (src_f32)
            qmm_quantize_q4_k_kernel<true><<<grid, kQuantThreads, 0, stream>>>(src, d, nsuper);
        else
            qmm_quantize_q4_k_kernel<false><<<grid, kQuantThreads, 0, stream>>>(src, d, nsuper);
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
        qmm_dequantize_q8_0_kernel<<<grid, kQuantThreads, 0, stream>>>(s, dst, ngroups);
    else
        qmm_dequantize_q4_k_kernel<<<grid, kQuantThreads, 0, stream>>>(s, dst, ngroups);
    return cudaGetLastError();
}

}  // namespace qmm
