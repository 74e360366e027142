// kquant.cu -- the K-quants Q5_K, Q3_K and Q2_K: ISQ, dequantization, the
// linear layer and their rows of the embedding lookup.
//
// mistral.rs, "Quantization types": the table "Q*K family" lists q5k, q3k and
// q2k at 5, 3 and 2 bits, and section "Numeric shorthands" resolves `--isq 5`,
// `3` and `2` to Q5K, Q3K and Q2K on CUDA.  The byte layouts (GGUF-shaped)
// and the quantizers are this library's reading, stated in include/qmm.h:
//   Q5_K  176 bytes: d, dmin, 12 scale bytes (Q4_K's packing), qh[32], qs[128];
//         affine, 8 sub-blocks of 32, 5-bit codes.
//   Q3_K  110 bytes: hmask[32], qs[64], 12 bytes of sixteen 6-bit scale fields
//         (each sc + 32), d; symmetric, 16 sub-blocks of 16, 3-bit codes c + 4.
//   Q2_K  84 bytes: scales[16] (sc | mc << 4), qs[64], d, dmin; affine, 16
//         sub-blocks of 16, 2-bit codes.
// ISQ takes quantize.cu's word-level structure (one lane per sub-block,
// codes four to a word, superblocks assembled in shared memory): the plain
// definition's fp32 steps in its order (IEEE division or a correctly rounded
// constant division for the scales, round half away for the codes, binary16
// round-to-nearest-even for d and dmin), so the bytes are bit-identical; a
// quotient that is only rounded to an integer (a weight code, a scale code)
// comes from the approximate reciprocal with an exact decision next to a
// rounding tie (round2 / exact_code / round_div), which gives the integer
// that roundf of the IEEE quotient gives.
// Dequantization, the embedding rows and the direct-load linear layer give
// lane l of a warp the weights 8l .. 8l + 7 of a superblock: each weight is
// dequantized exactly as the plain definition does (one fp32 rounding of
// S q - Mn) and multiplied in fp32.  That linear layer serves Q3_K / Q2_K
// above one token or with rows that are not 16-byte multiples (one token runs
// sbrows.cu); Q5_K runs the row-tile decode kernel (gemv_rows.cu) and the
// tiled kernel (gemm.cu).
#include "common.cuh"

namespace qmm {

constexpr int kKqThreads = 256;  // 8 warps

__host__ __device__ constexpr int kq_bytes(int fmt) { return fmt == 5 ? 176 : fmt == 3 ? 110 : 84; }

__device__ __forceinline__ float h2f_at(const uint8_t *p) {
    return __half2float(__ushort_as_half(*reinterpret_cast<const uint16_t *>(p)));
}

// ------------------------------------------------------------ decoding
// The 6-bit scale / min codes of sub-block j of a Q4_K / Q5_K scale area.
__device__ __forceinline__ void kq_scale_min_k4(const uint8_t *s12, int j, int &sc, int &mc) {
    if (j < 4) {
        sc = s12[j] & 63;
        mc = s12[j + 4] & 63;
    } else {
        sc = (s12[j + 4] & 15) | ((s12[j - 4] >> 6) << 4);
        mc = (s12[j + 4] >> 4) | ((s12[j] >> 6) << 4);
    }
}

// Q3_K scale field j (0..15): low 4 bits in byte j mod 8 (high nibble for
// j >= 8), high 2 bits at bit 2 (j div 4) of byte 8 + j mod 4.
__device__ __forceinline__ int kq_q3_field(const uint8_t *s12, int j) {
    return ((s12[j & 7] >> (j < 8 ? 0 : 4)) & 15) | (((s12[8 + (j & 3)] >> (2 * (j >> 2))) & 3) << 4);
}

// The bytes lane l needs from a superblock for its weights 8l .. 8l + 7,
// loaded with the widest loads the superblock's alignment allows (Q5_K 16,
// Q2_K 4, Q3_K 2 bytes): first all loads, then the decoding, so that a
// caller can put several superblocks' loads in flight before using any.
struct KqRaw {
    uint32_t a0, a1;  // Q5_K qs / Q3_K qs / Q2_K qs: the lane's 8 code bytes
    uint32_t b0, b1;  // Q5_K qh / Q3_K hmask: the lane's 8 high-bit bytes
    uint32_t s0, s1;  // scale words (see kq_lane_decode)
};

// A load through the read-only path (global memory) or a plain one (kSm:
// shared memory, where the superblocks sit after a TMA copy).
template <bool kSm, typename T>
__device__ __forceinline__ T kq_ld(const T *p) {
    if constexpr (kSm) return *p;
    else return __ldg(p);
}

// 8 bytes at a 2-byte aligned address, as two words (the aligned word below
// is formed from the pointer itself, which keeps its address space visible).
template <bool kSm = false>
__device__ __forceinline__ void kq_ld8_a2(const uint8_t *p, uint32_t &w0, uint32_t &w1) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    const uint32_t *w = reinterpret_cast<const uint32_t *>(p - (a & 3));
    const uint32_t x0 = kq_ld<kSm>(w), x1 = kq_ld<kSm>(w + 1);
    if ((a & 3) == 0) {
        w0 = x0;
        w1 = x1;
    } else {
        const uint32_t x2 = kq_ld<kSm>(w + 2);
        w0 = __funnelshift_r(x0, x1, 16);
        w1 = __funnelshift_r(x1, x2, 16);
    }
}

template <int kFmt, bool kSm = false>
__device__ __forceinline__ KqRaw kq_lane_load(const uint8_t *blk, int lane) {
    KqRaw r;
    const int h = lane >> 4, o = 8 * (lane & 3);
    if constexpr (kFmt == 5) {
        const int j = lane >> 2;
        const uint2 qs = kq_ld<kSm>(reinterpret_cast<const uint2 *>(blk + 48 + 32 * (j >> 1) + o));
        const uint2 qh = kq_ld<kSm>(reinterpret_cast<const uint2 *>(blk + 16 + o));
        const uint4 hd = kq_ld<kSm>(reinterpret_cast<const uint4 *>(blk));  // d, dmin, 12 scale bytes
        r.a0 = qs.x; r.a1 = qs.y; r.b0 = qh.x; r.b1 = qh.y;
        // Q4_K's scale packing: scale bytes 0-3 = hd.y, 4-7 = hd.z, 8-11 = hd.w
        const uint32_t k = 8u * (uint32_t)(j & 3);
        const uint32_t by = (hd.y >> k) & 0xFFu, bz = (hd.z >> k) & 0xFFu, bw = (hd.w >> k) & 0xFFu;
        const uint32_t sc = j < 4 ? (by & 63u) : ((bw & 15u) | ((by >> 6) << 4));
        const uint32_t mc = j < 4 ? (bz & 63u) : ((bw >> 4) | ((bz >> 6) << 4));
        r.s0 = hd.x;  // d | dmin << 16
        r.s1 = sc | (mc << 8);
    } else if constexpr (kFmt == 3) {
        kq_ld8_a2<kSm>(blk + 32 + 32 * h + o, r.a0, r.a1);
        kq_ld8_a2<kSm>(blk + o, r.b0, r.b1);
        const int j = lane >> 1;
        r.s0 = (uint32_t)kq_q3_field(blk + 96, j);
        r.s1 = (uint32_t)(*reinterpret_cast<const uint16_t *>(blk + 108));
    } else {
        const uint32_t *qs = reinterpret_cast<const uint32_t *>(blk + 16 + 32 * h + o);
        r.a0 = kq_ld<kSm>(qs);
        r.a1 = kq_ld<kSm>(qs + 1);
        r.b0 = r.b1 = 0;
        r.s0 = blk[lane >> 1];
        r.s1 = kq_ld<kSm>(reinterpret_cast<const uint32_t *>(blk + 80));  // d | dmin << 16
    }
    return r;
}

// byte e of a word, exactly as a float (2^23 + b - 2^23)
__device__ __forceinline__ float kq_byte_f(uint32_t w, int e) {
    return __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7440u + e)) - 8388608.0f;
}

// The 8 dequantized weights of lane l, each the plain definition's fp32
// value: Q5_K / Q2_K (d*sc) * q - dmin*mc, Q3_K (d*sc) * (q - 4).
template <int kFmt>
__device__ __forceinline__ void kq_lane_decode(const KqRaw &r, int lane, float (&v)[8]) {
    const int s = (lane >> 2) & 3, h = lane >> 4;
    if constexpr (kFmt == 5) {
        const int j = lane >> 2, nsh = 4 * (j & 1);
        const float S = __half2float(__ushort_as_half((unsigned short)(r.s0 & 0xFFFF))) * (float)(r.s1 & 0xFF);
        const float Mn = __half2float(__ushort_as_half((unsigned short)(r.s0 >> 16))) * (float)(r.s1 >> 8);
        const uint32_t q0 = ((r.a0 >> nsh) & 0x0F0F0F0Fu) | (((r.b0 >> j) & 0x01010101u) << 4);
        const uint32_t q1 = ((r.a1 >> nsh) & 0x0F0F0F0Fu) | (((r.b1 >> j) & 0x01010101u) << 4);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float p0 = S * kq_byte_f(q0, e), p1 = S * kq_byte_f(q1, e);
            v[e] = p0 - Mn;
            v[4 + e] = p1 - Mn;
        }
    } else if constexpr (kFmt == 3) {
        const float S = __half2float(__ushort_as_half((unsigned short)r.s1)) * (float)((int)r.s0 - 32);
        const int hb = 4 * h + s;
        const uint32_t q0 = ((r.a0 >> (2 * s)) & 0x03030303u) | (((r.b0 >> hb) & 0x01010101u) << 2);
        const uint32_t q1 = ((r.a1 >> (2 * s)) & 0x03030303u) | (((r.b1 >> hb) & 0x01010101u) << 2);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            v[e] = S * (kq_byte_f(q0, e) - 4.0f);
            v[4 + e] = S * (kq_byte_f(q1, e) - 4.0f);
        }
    } else {
        const float S = __half2float(__ushort_as_half((unsigned short)(r.s1 & 0xFFFF))) * (float)(r.s0 & 15);
        const float Mn = __half2float(__ushort_as_half((unsigned short)(r.s1 >> 16))) * (float)(r.s0 >> 4);
        const uint32_t q0 = (r.a0 >> (2 * s)) & 0x03030303u, q1 = (r.a1 >> (2 * s)) & 0x03030303u;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float p0 = S * kq_byte_f(q0, e), p1 = S * kq_byte_f(q1, e);
            v[e] = p0 - Mn;
            v[4 + e] = p1 - Mn;
        }
    }
}

template <int kFmt>
__device__ __forceinline__ void kq_lane_values(const uint8_t *blk, int lane, float (&v)[8]) {
    kq_lane_decode<kFmt>(kq_lane_load<kFmt>(blk, lane), lane, v);
}

// For the matmul: lane l's 8 codes as exact floats (Q3_K: q - 4) with the
// sub-block's S (and Mn), so that its share of a dot product is
// S * sum(c x) - Mn * sum(x) -- the scale and the min applied once per
// superblock instead of once per weight.
struct KqCodes {
    float S, Mn;
    float c[8];
};
template <int kFmt>
__device__ __forceinline__ KqCodes kq_lane_codes(const KqRaw &r, int lane) {
    KqCodes k;
    const int s = (lane >> 2) & 3, h = lane >> 4;
    uint32_t q0, q1;
    float bias = 8388608.0f;  // byte b under the float 2^23 exponent is 2^23 + b
    if constexpr (kFmt == 5) {
        const int j = lane >> 2, nsh = 4 * (j & 1);
        k.S = __half2float(__ushort_as_half((unsigned short)(r.s0 & 0xFFFF))) * (float)(r.s1 & 0xFF);
        k.Mn = __half2float(__ushort_as_half((unsigned short)(r.s0 >> 16))) * (float)(r.s1 >> 8);
        q0 = ((r.a0 >> nsh) & 0x0F0F0F0Fu) | (((r.b0 >> j) & 0x01010101u) << 4);
        q1 = ((r.a1 >> nsh) & 0x0F0F0F0Fu) | (((r.b1 >> j) & 0x01010101u) << 4);
    } else if constexpr (kFmt == 3) {
        k.S = __half2float(__ushort_as_half((unsigned short)r.s1)) * (float)((int)r.s0 - 32);
        k.Mn = 0.f;
        const int hb = 4 * h + s;
        q0 = ((r.a0 >> (2 * s)) & 0x03030303u) | (((r.b0 >> hb) & 0x01010101u) << 2);
        q1 = ((r.a1 >> (2 * s)) & 0x03030303u) | (((r.b1 >> hb) & 0x01010101u) << 2);
        bias = 8388612.0f;  // 2^23 + 4: the code minus 4, exactly
    } else {
        k.S = __half2float(__ushort_as_half((unsigned short)(r.s1 & 0xFFFF))) * (float)(r.s0 & 15);
        k.Mn = __half2float(__ushort_as_half((unsigned short)(r.s1 >> 16))) * (float)(r.s0 >> 4);
        q0 = (r.a0 >> (2 * s)) & 0x03030303u;
        q1 = (r.a1 >> (2 * s)) & 0x03030303u;
    }
    const uint64_t b2 = f2_pack(bias, bias);
#pragma unroll
    for (int e = 0; e < 4; e += 2) {  // code pairs, one packed subtraction each
        f2_unpack(f2_sub(f2_pack(__uint_as_float(__byte_perm(q0, 0x4B000000u, 0x7440u + e)),
                                 __uint_as_float(__byte_perm(q0, 0x4B000000u, 0x7441u + e))),
                         b2),
                  k.c[e], k.c[e + 1]);
        f2_unpack(f2_sub(f2_pack(__uint_as_float(__byte_perm(q1, 0x4B000000u, 0x7440u + e)),
                                 __uint_as_float(__byte_perm(q1, 0x4B000000u, 0x7441u + e))),
                         b2),
                  k.c[4 + e], k.c[5 + e]);
    }
    return k;
}
// acc + S * sum_k c_k x_k - Mn * sum_k x_k over the lane's 8 bf16 activations
// (xw: pairs, lower index in the low half).  Each sum runs as two packed
// fp32 lanes (even k, odd k, each in k order), added at the end.
template <int kFmt>
__device__ __forceinline__ float kq_codes_dot(const KqCodes &k, const uint32_t (&xw)[4], float acc) {
    uint64_t p2 = f2_pack(0.f, 0.f), s2 = f2_pack(0.f, 0.f);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const uint64_t x2 = f2_pack(__uint_as_float(xw[e] << 16), __uint_as_float(xw[e] & 0xFFFF0000u));
        p2 = f2_fma(f2_pack(k.c[2 * e], k.c[2 * e + 1]), x2, p2);
        if constexpr (kFmt != 3) s2 = f2_add(s2, x2);
    }
    float pe, po;
    f2_unpack(p2, pe, po);
    const float p = pe + po;
    if constexpr (kFmt == 3) {
        return fmaf(k.S, p, acc);
    } else {
        float se, so;
        f2_unpack(s2, se, so);
        return fmaf(k.S, p, fmaf(-k.Mn, se + so, acc));
    }
}

// ---------------------------------------------------------- dequantization
template <int kFmt>
__global__ void __launch_bounds__(kKqThreads) qmm_dequantize_kq_kernel(const uint8_t *__restrict__ src,
                                                                       float *__restrict__ dst, int64_t nblocks) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int64_t b = (int64_t)blockIdx.x * (kKqThreads / 32) + warp; b < nblocks;
         b += (int64_t)gridDim.x * (kKqThreads / 32)) {
        float v[8];
        kq_lane_values<kFmt>(src + b * kq_bytes(kFmt), lane, v);
        float4 *y = reinterpret_cast<float4 *>(dst + b * 256 + 8 * lane);
        y[0] = make_float4(v[0], v[1], v[2], v[3]);
        y[1] = make_float4(v[4], v[5], v[6], v[7]);
    }
}

// ------------------------------------------------------------------ matmul
// Y[M x N] = X[M x K] W^T.  A warp owns one weight row at a time; lane l takes
// weights 8l .. 8l + 7 of each superblock, decoded once per pass for up to
// kTok token rows: one token takes the exact codes and applies the sub-block
// scale and min once (kq_codes_dot); a pass of 8 dequantizes each weight once
// (one fp32 rounding) and multiplies it by the 8 tokens.  fp32 sums reduced
// across the warp.
template <int kFmt, int kTok>
__global__ void __launch_bounds__(kKqThreads, kTok == 1 ? 3 : 2) qmm_matmul_kq_kernel(const uint8_t *__restrict__ W,
                                                                   const uint16_t *__restrict__ X,
                                                                   float *__restrict__ Y, int M, int N, int K) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nsb = K / 256;
    const int64_t row_bytes = (int64_t)nsb * kq_bytes(kFmt);
    for (int64_t n = (int64_t)blockIdx.x * (kKqThreads / 32) + warp; n < N;
         n += (int64_t)gridDim.x * (kKqThreads / 32)) {
        const uint8_t *row = W + n * row_bytes;
        for (int m0 = 0; m0 < M; m0 += kTok) {
            const int mt = min(kTok, M - m0);
            float acc[kTok];
#pragma unroll
            for (int t = 0; t < kTok; ++t) acc[t] = 0.f;
            // superblocks whose loads are in flight together
            constexpr int kU = 4;
            for (int sb0 = 0; sb0 < nsb; sb0 += kU) {
                KqRaw raw[kU];
#pragma unroll
                for (int u = 0; u < kU; ++u)
                    if (sb0 + u < nsb) raw[u] = kq_lane_load<kFmt>(row + (int64_t)(sb0 + u) * kq_bytes(kFmt), lane);
#pragma unroll
                for (int u = 0; u < kU; ++u) {
                    if (sb0 + u >= nsb) break;
                    if constexpr (kTok == 1) {
                        const uint4 xv = __ldg(reinterpret_cast<const uint4 *>(X + (int64_t)m0 * K +
                                                                               (int64_t)(sb0 + u) * 256 + 8 * lane));
                        const uint32_t w[4] = {xv.x, xv.y, xv.z, xv.w};
                        acc[0] = kq_codes_dot<kFmt>(kq_lane_codes<kFmt>(raw[u], lane), w, acc[0]);
                    } else {
                        float v[8];
                        kq_lane_decode<kFmt>(raw[u], lane, v);
#pragma unroll
                        for (int t = 0; t < kTok; ++t) {
                            if (t < mt) {
                                const uint4 xv = __ldg(reinterpret_cast<const uint4 *>(
                                    X + (int64_t)(m0 + t) * K + (int64_t)(sb0 + u) * 256 + 8 * lane));
                                const uint32_t w[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
                                for (int e = 0; e < 4; ++e) {
                                    acc[t] = fmaf(v[2 * e], __uint_as_float(w[e] << 16), acc[t]);
                                    acc[t] = fmaf(v[2 * e + 1], __uint_as_float(w[e] & 0xFFFF0000u), acc[t]);
                                }
                            }
                        }
                    }
                }
            }
#pragma unroll
            for (int t = 0; t < kTok; ++t) {
                float s = acc[t];
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
                if (lane == 0 && t < mt) Y[(int64_t)(m0 + t) * N + n] = s;
            }
        }
    }
}

// ------------------------------------------------------------- Q5_K ISQ
// Q5_K quantizes like Q4_K with 5-bit codes, so it takes quantize.cu's Q4_K
// structure: one lane per 32-weight sub-block (8 lanes a superblock, 4
// superblocks a warp), codes four to a word from round2 with the same tie
// flagging, the Q4_K scale bytes, and the superblock assembled in shared
// memory and stored with 16-byte writes.  The fifth code bits (qh byte l,
// bit j: bit 4 of weight l of sub-block j) are gathered with shuffles: lane
// j moves its bits to bit j of each byte and the 8 lanes OR their words.
template <bool kSrcF32>
__global__ void __launch_bounds__(kQuantThreads, QMM_Q4_QUANT_MIN_BLOCKS)
qmm_quantize_q5_k_kernel(const void *__restrict__ src, uint8_t *__restrict__ dst, int64_t nsuper) {
    constexpr int kB = 176;
    __shared__ __align__(16) uint8_t stage[kQuantWarps][4 * kB];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int sj = lane & 7, sbl = lane >> 3;  // sub-block j, superblock in the warp tile
    uint8_t *st = stage[warp] + sbl * kB;
    const int64_t nwarps = (int64_t)gridDim.x * kQuantWarps;
    const int64_t step = nwarps * 4;
    int64_t s0 = ((int64_t)blockIdx.x * kQuantWarps + warp) * 4;
    Lane32<kSrcF32> Ln;
    if (!kSrcF32) Ln.load(src, (s0 + sbl) * 256 + sj * 32, s0 + sbl < nsuper);
    for (; s0 < nsuper; s0 += step) {
        const int64_t sb = s0 + sbl;
        const bool valid = sb < nsuper;  // uniform over each group of 8 lanes
        const int nvalid = (int)min((int64_t)4, nsuper - s0);
        Lane32<kSrcF32> L;
        if constexpr (kSrcF32) {
            L.load(src, sb * 256 + sj * 32, valid);
        } else {
            L = Ln;
            Ln.load(src, (sb + step) * 256 + sj * 32, sb + step < nsuper);
        }
        float mx, mn;  // max_i x_i and min(0, min_i x_i)
        L.extremes(mx, mn);
        mn = fminf(0.0f, mn);
        const float s = __fdiv_rn(__fsub_rn(mx, mn), 31.0f);
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
        const float tsc = df > 0.0f ? round_div(s, df) : 0.0f;
        const float tmc = dminf > 0.0f ? round_div(m, dminf) : 0.0f;
        const int sc = (int)clamp_f(tsc, 0.0f, 63.0f);
        const int mc = (int)clamp_f(tmc, 0.0f, 63.0f);
        const float S = __fmul_rn(df, (float)sc);
        const float Mn = __fmul_rn(dminf, (float)mc);
        uint32_t w[8];  // 5-bit codes, one per byte
#pragma unroll
        for (int i = 0; i < 8; ++i) w[i] = 0u;
        float r = 0.0f;
        bool tie = false;
        if (S > 0.0f) {
            r = rcp_approx(S);
            const uint64_t r2 = f2_pack(r, r), mn2 = f2_pack(Mn, Mn);
            float dev = 0.0f;
            // codes of u = x + Mn (its own rounding step) over S; monotone in x,
            // so when the extremes' codes lie well inside int16 the clamp to
            // [0, 31] runs on 16-bit pairs, otherwise on the floats
            const float khi = __fmul_rn(__fadd_rn(mx, Mn), r), klo = __fmul_rn(__fadd_rn(mn, Mn), r);
            if (khi < 30000.0f && klo > -30000.0f) {
                auto code2 = [&](int i) {
                    const uint64_t v = round2(f2_add(L.pair(i), mn2), r2, dev);
                    return __vimin_s16x2_relu(prmt((uint32_t)v, (uint32_t)(v >> 32), 0x5410u), 0x001F001Fu);
                };
#pragma unroll
                for (int i = 0; i < 8; ++i) w[i] = prmt(code2(4 * i), code2(4 * i + 2), 0x6420u);
            } else {
                auto code2 = [&](int i) { return clamp2(round2(f2_add(L.pair(i), mn2), r2, dev), 0.0f, 31.0f); };
#pragma unroll
                for (int i = 0; i < 8; ++i) w[i] = pack4_magic(code2(4 * i), code2(4 * i + 2));
            }
            // codes matter up to 31.5: 2^-23 * 31.75 + 2^-25 = 2^-18, Q4_K's guard
            tie = valid && dev >= kTieGuardQ4;
        }
        // low nibbles: sub-block 2c (low) and 2c + 1 (high) share qs chunk c
        uint32_t hw[8], hb[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            hw[i] = __shfl_xor_sync(0xffffffffu, w[i], 1);
            hb[i] = ((w[i] >> 4) & 0x01010101u) << sj;  // bit 4 of each code to bit sj of its byte
        }
#pragma unroll
        for (int o = 1; o <= 4; o <<= 1)
#pragma unroll
            for (int i = 0; i < 8; ++i) hb[i] |= __shfl_xor_sync(0xffffffffu, hb[i], o);
        const int sc4 = __shfl_down_sync(0xffffffffu, sc, 4);
        const int mc4 = __shfl_down_sync(0xffffffffu, mc, 4);
        if (valid) {
            if ((sj & 1) == 0) {
                uint4 *o = reinterpret_cast<uint4 *>(st + 48 + 32 * (sj >> 1));
                o[0] = make_uint4((w[0] & 0x0F0F0F0Fu) | ((hw[0] & 0x0F0F0F0Fu) << 4),
                                  (w[1] & 0x0F0F0F0Fu) | ((hw[1] & 0x0F0F0F0Fu) << 4),
                                  (w[2] & 0x0F0F0F0Fu) | ((hw[2] & 0x0F0F0F0Fu) << 4),
                                  (w[3] & 0x0F0F0F0Fu) | ((hw[3] & 0x0F0F0F0Fu) << 4));
                o[1] = make_uint4((w[4] & 0x0F0F0F0Fu) | ((hw[4] & 0x0F0F0F0Fu) << 4),
                                  (w[5] & 0x0F0F0F0Fu) | ((hw[5] & 0x0F0F0F0Fu) << 4),
                                  (w[6] & 0x0F0F0F0Fu) | ((hw[6] & 0x0F0F0F0Fu) << 4),
                                  (w[7] & 0x0F0F0F0Fu) | ((hw[7] & 0x0F0F0F0Fu) << 4));
            }
            if (sj == 1) {  // qh bytes 0-31
                uint4 *o = reinterpret_cast<uint4 *>(st + 16);
                o[0] = make_uint4(hb[0], hb[1], hb[2], hb[3]);
                o[1] = make_uint4(hb[4], hb[5], hb[6], hb[7]);
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
        // time, lane l taking weight l, and overwrites its nibble and qh bit
        for (uint32_t fl = __ballot_sync(0xffffffffu, tie); fl != 0; fl &= fl - 1) {
            const int l = __ffs(fl) - 1, jl = l & 7;
            const float Sl = __shfl_sync(0xffffffffu, S, l), rl = __shfl_sync(0xffffffffu, r, l);
            const float Ml = __shfl_sync(0xffffffffu, Mn, l);
            const float u = __fadd_rn(Lane32<kSrcF32>::reload(src, (s0 + (l >> 3)) * 256 + jl * 32, lane), Ml);
            const uint32_t c = int_byte(clamp_f(exact_code(u, Sl, rl, kTieGuardQ4), 0.0f, 31.0f));
            uint8_t *sbp = stage[warp] + (l >> 3) * kB;
            uint8_t *q = sbp + 48 + 32 * (jl >> 1) + lane;
            *q = (uint8_t)((jl & 1) ? ((*q & 0x0Fu) | ((c & 15u) << 4)) : ((*q & 0xF0u) | (c & 15u)));
            uint8_t *h = sbp + 16 + lane;
            *h = (uint8_t)((*h & ~(1u << jl)) | (((c >> 4) & 1u) << jl));
            __syncwarp();
        }
        const int nvec = nvalid * kB / 16;
        uint4 *out = reinterpret_cast<uint4 *>(dst + s0 * kB);
        for (int v = lane; v < nvec; v += 32) out[v] = reinterpret_cast<const uint4 *>(stage[warp])[v];
        __syncwarp();
    }
}

// ------------------------------------------------------ Q3_K / Q2_K ISQ
// The 16-weight sub-block formats on the same word-level structure: one lane
// per sub-block (16 lanes a superblock, 2 superblocks a warp), the lane's 16
// codes four to a word from round2 with the Q4_K tie flagging.  Lane j holds
// weights 16j .. 16j + 15 = bytes l = 16 (j mod 2) .. + 15 of half h = j div 8
// at shift s = (j div 2) mod 4; the low code bits of a byte come from the 4
// lanes that differ in s, Q3_K's hmask bits from the 8 that differ in s and h,
// gathered with shuffles (lane j moves its bits into place, the lanes OR).
// Q3_K superblocks are 2-byte aligned in a row, Q2_K 4-byte: halfword and
// word stores.
template <bool kSrcF32> struct Lane16;
template <> struct Lane16<true> {
    float x[16];
    __device__ __forceinline__ void load(const void *src, int64_t elem, bool valid) {
        const float4 *p = reinterpret_cast<const float4 *>(static_cast<const float *>(src) + elem);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float4 v = valid ? __ldg(p + i) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            x[4 * i] = v.x;
            x[4 * i + 1] = v.y;
            x[4 * i + 2] = v.z;
            x[4 * i + 3] = v.w;
        }
    }
    __device__ __forceinline__ uint64_t pair(int i) const { return f2_pack(x[i], x[i + 1]); }
    static __device__ __forceinline__ float reload(const void *src, int64_t elem, int j) {
        return __ldg(static_cast<const float *>(src) + elem + j);
    }
    __device__ __forceinline__ void extremes(float &mx, float &mn) const {
        mx = x[0];
        mn = x[0];
#pragma unroll
        for (int i = 1; i < 16; ++i) {
            mx = fmaxf(mx, x[i]);
            mn = fminf(mn, x[i]);
        }
    }
};
template <> struct Lane16<false> {
    uint32_t w[8];
    __device__ __forceinline__ void load(const void *src, int64_t elem, bool valid) {
        const uint4 *p = reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(src) + elem);
#pragma unroll
        for (int i = 0; i < 2; ++i) {
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
    __device__ __forceinline__ void extremes(float &mx, float &mn) const {
        __nv_bfloat162 vmax = *reinterpret_cast<const __nv_bfloat162 *>(&w[0]), vmin = vmax;
#pragma unroll
        for (int i = 1; i < 8; ++i) {
            const __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162 *>(&w[i]);
            vmax = __hmax2(vmax, v);
            vmin = __hmin2(vmin, v);
        }
        mx = fmaxf(__low2float(vmax), __high2float(vmax));
        mn = fminf(__low2float(vmin), __high2float(vmin));
    }
};

template <int kFmt, bool kSrcF32>
__global__ void __launch_bounds__(kQuantThreads, QMM_Q4_QUANT_MIN_BLOCKS)
qmm_quantize_k16_kernel(const void *__restrict__ src, uint8_t *__restrict__ dst, int64_t nsuper) {
    static_assert(kFmt == 3 || kFmt == 2, "16-weight sub-block formats");
    constexpr int kB = kq_bytes(kFmt);            // 110 / 84
    constexpr int kLo = kFmt == 3 ? 32 : 16;      // the low-bit (qs) bytes
    constexpr float kQLo = kFmt == 3 ? -4.0f : 0.0f, kQHi = 3.0f;
    __shared__ __align__(16) uint8_t stage[kQuantWarps][2 * kB];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int sj = lane & 15, sbl = lane >> 4;  // sub-block j, superblock in the warp tile
    const int hh = sj >> 3, ss = (sj >> 1) & 3, pp = sj & 1;
    uint8_t *st = stage[warp] + sbl * kB;
    const int64_t nwarps = (int64_t)gridDim.x * kQuantWarps;
    const int64_t step = nwarps * 2;
    int64_t s0 = ((int64_t)blockIdx.x * kQuantWarps + warp) * 2;
    Lane16<kSrcF32> Ln;
    if (!kSrcF32) Ln.load(src, (s0 + sbl) * 256 + sj * 16, s0 + sbl < nsuper);
    for (; s0 < nsuper; s0 += step) {
        const int64_t sb = s0 + sbl;
        const bool valid = sb < nsuper;  // uniform over each half-warp
        const int nvalid = (int)min((int64_t)2, nsuper - s0);
        Lane16<kSrcF32> L;
        if constexpr (kSrcF32) {
            L.load(src, sb * 256 + sj * 16, valid);
        } else {
            L = Ln;
            Ln.load(src, (sb + step) * 256 + sj * 16, sb + step < nsuper);
        }
        float mx, mn;
        L.extremes(mx, mn);
        float S = 0.0f, Mn = 0.0f, v0 = 0.0f, v1 = 0.0f;  // v0, v1: the lane's scale codes
        __half dh, dminh = __ushort_as_half((unsigned short)0);
        if constexpr (kFmt == 3) {
            // symmetric: s_j = max |x| / 3, d = fp16(max_j s_j / 31), sc in 0..31
            float amax = fmaxf(mx, -mn);
            amax = amax > 0.0f ? amax : 0.0f;
            const float s = __fdiv_rn(amax, 3.0f);
            float smax = s;
#pragma unroll
            for (int o = 1; o <= 8; o <<= 1) smax = fmaxf(smax, __shfl_xor_sync(0xffffffffu, smax, o));
            smax = smax > 0.0f ? smax : 0.0f;
            dh = __float2half_rn(__fdiv_rn(smax, 31.0f));
            const float df = __half2float(dh);
            v0 = df > 0.0f ? clamp_f(round_div(s, df), 0.0f, 31.0f) : 0.0f;
            S = __fmul_rn(df, v0);
        } else {
            // affine: s_j = (max - min(0, min)) / 3, m_j = 0 - min(0, min), d, dmin = fp16(max / 15)
            mn = fminf(0.0f, mn);
            const float s = __fdiv_rn(__fsub_rn(mx, mn), 3.0f);
            const float m = __fsub_rn(0.0f, mn);
            float smax = s, mmax = m;
#pragma unroll
            for (int o = 1; o <= 8; o <<= 1) {
                smax = fmaxf(smax, __shfl_xor_sync(0xffffffffu, smax, o));
                mmax = fmaxf(mmax, __shfl_xor_sync(0xffffffffu, mmax, o));
            }
            smax = smax > 0.0f ? smax : 0.0f;
            mmax = mmax > 0.0f ? mmax : 0.0f;
            dh = __float2half_rn(div_const<15>(smax));
            dminh = __float2half_rn(div_const<15>(mmax));
            const float df = __half2float(dh), dminf = __half2float(dminh);
            v0 = df > 0.0f ? clamp_f(round_div(s, df), 0.0f, 15.0f) : 0.0f;
            v1 = dminf > 0.0f ? clamp_f(round_div(m, dminf), 0.0f, 15.0f) : 0.0f;
            S = __fmul_rn(df, v0);
            Mn = __fmul_rn(dminf, v1);
        }
        // codes q (Q3_K: c + 4 with c in -4..3; Q2_K: 0..3), one per byte
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) w[i] = kFmt == 3 ? 0x04040404u : 0u;
        float r = 0.0f;
        bool tie = false;
        if (S > 0.0f) {
            r = rcp_approx(S);
            const uint64_t r2 = f2_pack(r, r), mn2 = f2_pack(Mn, Mn);
            float dev = 0.0f;
            auto u2 = [&](int i) { return kFmt == 3 ? L.pair(i) : f2_add(L.pair(i), mn2); };
            const float khi = __fmul_rn(kFmt == 3 ? mx : __fadd_rn(mx, Mn), r);
            const float klo = __fmul_rn(kFmt == 3 ? mn : __fadd_rn(mn, Mn), r);
            if (khi < 30000.0f && klo > -30000.0f) {
                // 16-bit pairs: (k - lo) clamped to [0, hi - lo]
                auto code2 = [&](int i) {
                    const uint64_t v = round2(u2(i), r2, dev);
                    uint32_t k2 = prmt((uint32_t)v, (uint32_t)(v >> 32), 0x5410u);
                    if constexpr (kFmt == 3) k2 = __vadd2(k2, 0x00040004u);
                    return __vimin_s16x2_relu(k2, kFmt == 3 ? 0x00070007u : 0x00030003u);
                };
#pragma unroll
                for (int i = 0; i < 4; ++i) w[i] = prmt(code2(4 * i), code2(4 * i + 2), 0x6420u);
            } else {
                auto code2 = [&](int i) { return clamp2(round2(u2(i), r2, dev), kQLo, kQHi); };
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    w[i] = pack4_magic(code2(4 * i), code2(4 * i + 2));
                    if constexpr (kFmt == 3) w[i] = __vadd4(w[i], 0x04040404u);
                }
            }
            // codes matter up to |Q| = 4.5: Q4_K's guard holds
            tie = valid && dev >= kTieGuardQ4;
        }
        // low 2 bits to bits 2s of their bytes, ORed over the 4 lanes that differ in s
        uint32_t lo[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) lo[i] = (w[i] & 0x03030303u) << (2 * ss);
#pragma unroll
        for (int o = 2; o <= 4; o <<= 1)
#pragma unroll
            for (int i = 0; i < 4; ++i) lo[i] |= __shfl_xor_sync(0xffffffffu, lo[i], o);
        uint32_t hb[4];  // Q3_K: bit 2 of q to bit 4h + s, ORed over the 8 lanes that differ in s, h
        if constexpr (kFmt == 3) {
#pragma unroll
            for (int i = 0; i < 4; ++i) hb[i] = ((w[i] >> 2) & 0x01010101u) << (4 * hh + ss);
#pragma unroll
            for (int o = 2; o <= 8; o <<= 1)
#pragma unroll
                for (int i = 0; i < 4; ++i) hb[i] |= __shfl_xor_sync(0xffffffffu, hb[i], o);
        }
        const int iv0 = (int)v0, iv1 = (int)v1;
        // Q3_K scale fields (sc + 32): byte j < 8 = field j | field j + 8 << 4; byte
        // 8 + j (j < 4) = bits 4-5 of fields j, j + 4, j + 8, j + 12 at bits 0, 2, 4, 6
        const int f0 = iv0 + 32;
        const int f4 = __shfl_down_sync(0xffffffffu, f0, 4), f8 = __shfl_down_sync(0xffffffffu, f0, 8);
        const int f12 = __shfl_down_sync(0xffffffffu, f0, 12);
        if (valid) {
            if ((sj & 6) == 0) {  // s == 0: 16 qs bytes at kLo + 32 h + 16 p
                uint16_t *o = reinterpret_cast<uint16_t *>(st + kLo + 32 * hh + 16 * pp);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    o[2 * i] = (uint16_t)(lo[i] & 0xFFFFu);
                    o[2 * i + 1] = (uint16_t)(lo[i] >> 16);
                }
            }
            if constexpr (kFmt == 3) {
                if ((sj & 14) == 0) {  // s == 0, h == 0: 16 hmask bytes at 16 p
                    uint16_t *o = reinterpret_cast<uint16_t *>(st + 16 * pp);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        o[2 * i] = (uint16_t)(hb[i] & 0xFFFFu);
                        o[2 * i + 1] = (uint16_t)(hb[i] >> 16);
                    }
                }
                if (sj < 8) st[96 + sj] = (uint8_t)((f0 & 15) | ((f8 & 15) << 4));
                if (sj < 4)
                    st[104 + sj] = (uint8_t)(((f0 >> 4) & 3) | (((f4 >> 4) & 3) << 2) | (((f8 >> 4) & 3) << 4) |
                                             (((f12 >> 4) & 3) << 6));
                if (sj == 0) *reinterpret_cast<uint16_t *>(st + 108) = __half_as_ushort(dh);
            } else {
                st[sj] = (uint8_t)(iv0 | (iv1 << 4));
                if (sj == 0) {
                    *reinterpret_cast<uint16_t *>(st + 80) = __half_as_ushort(dh);
                    *reinterpret_cast<uint16_t *>(st + 82) = __half_as_ushort(dminh);
                }
            }
        }
        __syncwarp();
        // sub-blocks with a possible tie: lanes 0-15 recompute weight `lane` of
        // the flagged sub-block and overwrite its code bits
        for (uint32_t fl = __ballot_sync(0xffffffffu, tie); fl != 0; fl &= fl - 1) {
            const int l = __ffs(fl) - 1, jl = l & 15;
            const float Sl = __shfl_sync(0xffffffffu, S, l), rl = __shfl_sync(0xffffffffu, r, l);
            const float Ml = __shfl_sync(0xffffffffu, Mn, l);
            if (lane < 16) {
                const float x = Lane16<kSrcF32>::reload(src, (s0 + (l >> 4)) * 256 + jl * 16, lane);
                const float u = kFmt == 3 ? x : __fadd_rn(x, Ml);
                const uint32_t q = (uint32_t)((int)clamp_f(exact_code(u, Sl, rl, kTieGuardQ4), kQLo, kQHi) -
                                              (int)kQLo);
                const int h = jl >> 3, s2 = 2 * ((jl >> 1) & 3), byte = 16 * (jl & 1) + lane;
                uint8_t *sbp = stage[warp] + (l >> 4) * kB;
                uint8_t *qb = sbp + kLo + 32 * h + byte;
                *qb = (uint8_t)((*qb & ~(3u << s2)) | ((q & 3u) << s2));
                if constexpr (kFmt == 3) {
                    const int hbit = 4 * h + (s2 >> 1);
                    uint8_t *hm = sbp + byte;
                    *hm = (uint8_t)((*hm & ~(1u << hbit)) | (((q >> 2) & 1u) << hbit));
                }
            }
            __syncwarp();
        }
        // the superblocks: halfwords (Q3_K, 2-byte aligned) or words (Q2_K)
        if constexpr (kFmt == 3) {
            const int n = nvalid * kB / 2;
            uint16_t *out = reinterpret_cast<uint16_t *>(dst + s0 * kB);
            for (int v = lane; v < n; v += 32) out[v] = reinterpret_cast<const uint16_t *>(stage[warp])[v];
        } else {
            const int n = nvalid * kB / 4;
            uint32_t *out = reinterpret_cast<uint32_t *>(dst + s0 * kB);
            for (int v = lane; v < n; v += 32) out[v] = reinterpret_cast<const uint32_t *>(stage[warp])[v];
        }
        __syncwarp();
    }
}

// ---------------------------------------------------------- embedding lookup
// out[t][0 .. D) = the dequantized row ids[t]: one warp per (token, superblock).
template <int kFmt, bool kBf16>
__global__ void __launch_bounds__(kKqThreads) qmm_embedding_kq_kernel(const uint8_t *__restrict__ table,
                                                                      const int64_t *__restrict__ ids,
                                                                      void *__restrict__ out, int64_t T, int64_t V,
                                                                      int64_t D) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t groups = D / 256;
    const int64_t row_bytes = groups * kq_bytes(kFmt);
    for (int64_t u = (int64_t)blockIdx.x * (kKqThreads / 32) + warp; u < T * groups;
         u += (int64_t)gridDim.x * (kKqThreads / 32)) {
        const int64_t t = u / groups, g = u - t * groups;
        const int64_t id = __ldg(ids + t);
        float v[8];
        if (id < 0 || id >= V) {
            if (lane == 0) record_error(kErrBadId);
#pragma unroll
            for (int e = 0; e < 8; ++e) v[e] = 0.f;
        } else {
            kq_lane_values<kFmt>(table + id * row_bytes + g * kq_bytes(kFmt), lane, v);
        }
        const int64_t base = t * D + g * 256 + 8 * lane;
        if constexpr (kBf16) {
            uint32_t p[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * e], v[2 * e + 1]);
                p[e] = *reinterpret_cast<const uint32_t *>(&h);
            }
            *reinterpret_cast<uint4 *>(static_cast<uint16_t *>(out) + base) = make_uint4(p[0], p[1], p[2], p[3]);
        } else {
            float4 *o = reinterpret_cast<float4 *>(static_cast<float *>(out) + base);
            o[0] = make_float4(v[0], v[1], v[2], v[3]);
            o[1] = make_float4(v[4], v[5], v[6], v[7]);
        }
    }
}

// ---------------------------------------------------------------- launchers
static int kq_grid(int64_t warps_of_work, int sms) {
    const int64_t ctas = (warps_of_work + kKqThreads / 32 - 1) / (kKqThreads / 32);
    const int64_t cap = (int64_t)sms * 8;
    return (int)(ctas < 1 ? 1 : ctas < cap ? ctas : cap);
}

cudaError_t launch_kq_quantize(int fmt, int src_f32, const void *src, void *dst, int64_t nweights, int sms,
                               cudaStream_t stream) {
    const int64_t nb = nweights / 256;
    if (fmt == 5) {
        if (nb == 0) return cudaSuccess;
        const int grid = grid_for(nb, 4 * kQuantWarps, sms);
        uint8_t *d = static_cast<uint8_t *>(dst);
        if (src_f32)
            qmm_quantize_q5_k_kernel<true><<<grid, kQuantThreads, 0, stream>>>(src, d, nb);
        else
            qmm_quantize_q5_k_kernel<false><<<grid, kQuantThreads, 0, stream>>>(src, d, nb);
        return cudaGetLastError();
    }
    if (nb == 0) return cudaSuccess;
    const int grid = grid_for(nb, 2 * kQuantWarps, sms);
    uint8_t *d = static_cast<uint8_t *>(dst);
    if (fmt == 3) {
        if (src_f32) qmm_quantize_k16_kernel<3, true><<<grid, kQuantThreads, 0, stream>>>(src, d, nb);
        else qmm_quantize_k16_kernel<3, false><<<grid, kQuantThreads, 0, stream>>>(src, d, nb);
    } else {
        if (src_f32) qmm_quantize_k16_kernel<2, true><<<grid, kQuantThreads, 0, stream>>>(src, d, nb);
        else qmm_quantize_k16_kernel<2, false><<<grid, kQuantThreads, 0, stream>>>(src, d, nb);
    }
    return cudaGetLastError();
}

cudaError_t launch_kq_dequantize(int fmt, const void *src, float *dst, int64_t nweights, int sms,
                                 cudaStream_t stream) {
    const int64_t nb = nweights / 256;
    const uint8_t *s = static_cast<const uint8_t *>(src);
    const int g = kq_grid(nb, sms);
    if (fmt == 5) qmm_dequantize_kq_kernel<5><<<g, kKqThreads, 0, stream>>>(s, dst, nb);
    else if (fmt == 3) qmm_dequantize_kq_kernel<3><<<g, kKqThreads, 0, stream>>>(s, dst, nb);
    else qmm_dequantize_kq_kernel<2><<<g, kKqThreads, 0, stream>>>(s, dst, nb);
    return cudaGetLastError();
}

template <int kFmt>
static cudaError_t kq_matmul_t(const uint8_t *w, const uint16_t *X, float *Y, int M, int N, int K, int sms,
                               cudaStream_t stream) {
    const int g = kq_grid(N, sms);
    // more tokens run in further passes of 8 over the row (its bytes then
    // come from L1 / L2): 16 token rows per pass cost registers and occupancy
    if (M == 1) qmm_matmul_kq_kernel<kFmt, 1><<<g, kKqThreads, 0, stream>>>(w, X, Y, M, N, K);
    else qmm_matmul_kq_kernel<kFmt, 8><<<g, kKqThreads, 0, stream>>>(w, X, Y, M, N, K);
    return cudaGetLastError();
}

cudaError_t launch_kq_matmul(int fmt, const void *W, const uint16_t *X, float *Y, int M, int N, int K, int sms,
                             cudaStream_t stream) {
    const uint8_t *w = static_cast<const uint8_t *>(W);
    if (fmt == 3) return kq_matmul_t<3>(w, X, Y, M, N, K, sms, stream);
    return kq_matmul_t<2>(w, X, Y, M, N, K, sms, stream);
}

template <int kFmt>
static cudaError_t kq_embedding_t(const void *table, const int64_t *ids, void *out, int bf16, int64_t T, int64_t V,
                                  int64_t D, int sms, cudaStream_t stream) {
    const int g = kq_grid(T * (D / 256), sms);
    const uint8_t *tb = static_cast<const uint8_t *>(table);
    if (bf16) qmm_embedding_kq_kernel<kFmt, true><<<g, kKqThreads, 0, stream>>>(tb, ids, out, T, V, D);
    else qmm_embedding_kq_kernel<kFmt, false><<<g, kKqThreads, 0, stream>>>(tb, ids, out, T, V, D);
    return cudaGetLastError();
}

cudaError_t launch_kq_embedding(int fmt, const void *table, const int64_t *ids, void *out, int bf16, int64_t T,
                                int64_t V, int64_t D, int sms, cudaStream_t stream) {
    if (fmt == 5) return kq_embedding_t<5>(table, ids, out, bf16, T, V, D, sms, stream);
    if (fmt == 3) return kq_embedding_t<3>(table, ids, out, bf16, T, V, D, sms, stream);
    return kq_embedding_t<2>(table, ids, out, bf16, T, V, D, sms, stream);
}

}  // namespace qmm
