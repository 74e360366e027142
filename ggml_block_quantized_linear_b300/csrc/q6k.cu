// q6k.cu -- the Q6_K format: ISQ, dequantization and the linear layer, plus
// the quantized embedding lookup of every format.
//
// mistral.rs, "Quantization types": the table "Q*K family" lists q6k at 6
// bits and section "Numeric shorthands" resolves `--isq 6` to Q6K on CUDA;
// section "Sensitive tensor precision" gives the token embeddings and the
// output head of a Q4K model the Q6K type (and of Q5K, Q6K, Q8_0 models the
// Q8_0 type, "the common high-precision Q target because quantized embedding
// kernels support it").  The byte layout (GGUF-shaped) and the quantizer are
// this library's reading, stated in include/qmm.h.
//
// A Q6_K superblock is 210 bytes, so superblocks are only 2-byte aligned in
// a packed row: the kernels here read them with 4-byte loads of the aligned
// words around them (no TMA boxes, which need 16-byte multiples).
#include "common.cuh"

namespace qmm {

constexpr int kQ6Bytes = 210;
constexpr int kQ6Threads = 256;  // 8 warps

// 8 bytes at a 2-byte aligned address, through the read-only path (global
// memory) or with plain loads (kSm: shared memory).  The aligned word below
// is formed from the pointer itself, which keeps its address space visible.
template <bool kSm = false>
__device__ __forceinline__ uint2 ld8_a2(const uint8_t *p) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    const uint32_t *w = reinterpret_cast<const uint32_t *>(p - (a & 3));
    const uint32_t sh = (uint32_t)(a & 3) * 8u;  // 0 or 16
    auto ld = [](const uint32_t *q) {
        if constexpr (kSm) return *q;
        else return __ldg(q);
    };
    const uint32_t w0 = ld(w), w1 = ld(w + 1);
    if (sh == 0) return make_uint2(w0, w1);
    const uint32_t w2 = ld(w + 2);
    return make_uint2(__funnelshift_r(w0, w1, sh), __funnelshift_r(w1, w2, sh));
}

// The 8 codes c = q - 32 of weights 8l .. 8l + 7 of a superblock (lane l):
// h = l / 16, s = (l / 4) % 4, first weight 32 s' + 8 (l % 4) of its 128-half.
// Low 4 bits: ql bytes 64 h + 32 (s & 1) + 8 (l % 4) + e (high nibble when
// s >= 2); high 2 bits: bits 2s, 2s + 1 of qh bytes 128 + 32 h + 8 (l % 4) + e.
template <bool kSm = false>
__device__ __forceinline__ void q6_lane_codes(const uint8_t *blk, int lane, float (&c)[8]) {
    const int h = lane >> 4, s = (lane >> 2) & 3, o = 8 * (lane & 3);
    const uint2 ql = ld8_a2<kSm>(blk + 64 * h + 32 * (s & 1) + o);
    const uint2 qh = ld8_a2<kSm>(blk + 128 + 32 * h + o);
    const uint32_t nsh = (uint32_t)(s >> 1) * 4u, hsh = 2u * (uint32_t)s;
    const uint32_t q0 = ((ql.x >> nsh) & 0x0F0F0F0Fu) | (((qh.x >> hsh) & 0x03030303u) << 4);
    const uint32_t q1 = ((ql.y >> nsh) & 0x0F0F0F0Fu) | (((qh.y >> hsh) & 0x03030303u) << 4);
    // byte b under the float 2^23 exponent is 2^23 + b; minus 2^23 + 32 gives
    // b - 32 exactly (code pairs, one packed subtraction each)
    const uint64_t b2 = f2_pack(8388640.0f, 8388640.0f);
#pragma unroll
    for (int e = 0; e < 4; e += 2) {
        f2_unpack(f2_sub(f2_pack(__uint_as_float(__byte_perm(q0, 0x4B000000u, 0x7440u + e)),
                                 __uint_as_float(__byte_perm(q0, 0x4B000000u, 0x7441u + e))),
                         b2),
                  c[e], c[e + 1]);
        f2_unpack(f2_sub(f2_pack(__uint_as_float(__byte_perm(q1, 0x4B000000u, 0x7440u + e)),
                                 __uint_as_float(__byte_perm(q1, 0x4B000000u, 0x7441u + e))),
                         b2),
                  c[4 + e], c[5 + e]);
    }
}

// sum_k c_k x_k over a lane's 8 codes and bf16 activations (xw: pairs, lower
// index in the low half), as two packed fp32 lanes (even k, odd k, each in k
// order) added at the end; the one-token kernels of q6k.cu and sbrows.cu
// share it, so their sums are the same bits.
__device__ __forceinline__ float q6_codes_dot(const float (&c)[8], const uint32_t (&xw)[4]) {
    uint64_t p2 = f2_pack(0.f, 0.f);
#pragma unroll
    for (int e = 0; e < 4; ++e)
        p2 = f2_fma(f2_pack(c[2 * e], c[2 * e + 1]),
                    f2_pack(__uint_as_float(xw[e] << 16), __uint_as_float(xw[e] & 0xFFFF0000u)), p2);
    float pe, po;
    f2_unpack(p2, pe, po);
    return pe + po;
}

// S = d * sc of lane l's sub-block (l / 2); exact in fp32.
__device__ __forceinline__ float q6_lane_scale(const uint8_t *blk, int lane) {
    const float d = __half2float(__ushort_as_half(*reinterpret_cast<const uint16_t *>(blk + 208)));
    const int sc = (int)(int8_t)blk[192 + (lane >> 1)];
    return d * (float)sc;
}

// ------------------------------------------------------------------- ISQ
// One warp per superblock; lane l holds weights 8l .. 8l + 7 (sub-block l / 2).
template <bool kSrcF32>
__global__ void __launch_bounds__(kQ6Threads) qmm_quantize_q6_k_kernel(const void *__restrict__ src,
                                                                       uint8_t *__restrict__ dst,
                                                                       int64_t nblocks) {
    __shared__ uint8_t qbuf[kQ6Threads / 32][256];
    __shared__ __align__(4) uint8_t obuf[kQ6Threads / 32][212];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint8_t *qw = qbuf[warp], *ow = obuf[warp];
    for (int64_t b = (int64_t)blockIdx.x * (kQ6Threads / 32) + warp; b < nblocks;
         b += (int64_t)gridDim.x * (kQ6Threads / 32)) {
        float x[8];
        if constexpr (kSrcF32) {
            const float4 *p = reinterpret_cast<const float4 *>(static_cast<const float *>(src) + b * 256 + 8 * lane);
            const float4 v0 = __ldg(p), v1 = __ldg(p + 1);
            x[0] = v0.x; x[1] = v0.y; x[2] = v0.z; x[3] = v0.w;
            x[4] = v1.x; x[5] = v1.y; x[6] = v1.z; x[7] = v1.w;
        } else {
            const uint4 v = __ldg(reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(src) + b * 256) + lane);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                x[2 * e] = __uint_as_float(w[e] << 16);
                x[2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
            }
        }
        float amax = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(x[e]));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));  // the sub-block's 16 weights
        const float sj = __fdiv_rn(amax, 31.0f);
        float smax = sj;
#pragma unroll
        for (int o = 2; o < 32; o <<= 1) smax = fmaxf(smax, __shfl_xor_sync(0xffffffffu, smax, o));
        const __half d16 = __float2half_rn(__fdiv_rn(smax, 127.0f));
        const float df = __half2float(d16);
        const int sc = df > 0.f ? (int)fminf(fmaxf(roundf(__fdiv_rn(sj, df)), 0.f), 127.f) : 0;
        const float S = df * (float)sc;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int c = S > 0.f ? (int)fminf(fmaxf(roundf(__fdiv_rn(x[e], S)), -32.f), 31.f) : 0;
            qw[8 * lane + e] = (uint8_t)(c + 32);
        }
        if ((lane & 1) == 0) ow[192 + (lane >> 1)] = (uint8_t)(int8_t)sc;
        if (lane == 0) *reinterpret_cast<uint16_t *>(ow + 208) = __half_as_ushort(d16);
        __syncwarp();
        // ql bytes 4 lane .. 4 lane + 3 and qh bytes 2 lane, 2 lane + 1
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int byte = 4 * lane + i;            // ql byte
            const int h = byte / 64, r = byte % 64;   // r = 32 (s & 1) + l'
            const int w = 128 * h + 32 * (r / 32) + r % 32;
            ow[byte] = (uint8_t)((qw[w] & 15) | ((qw[w + 64] & 15) << 4));
        }
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int byte = 2 * lane + i;            // qh byte
            const int h = byte / 32, l = byte % 32;
            const int w = 128 * h + l;
            ow[128 + byte] = (uint8_t)((qw[w] >> 4) | ((qw[w + 32] >> 4) << 2) | ((qw[w + 64] >> 4) << 4) |
                                       ((qw[w + 96] >> 4) << 6));
        }
        __syncwarp();
        // 210 bytes = 105 halfwords; the destination is 2-byte aligned
        uint16_t *out = reinterpret_cast<uint16_t *>(dst + b * kQ6Bytes);
        for (int i = lane; i < kQ6Bytes / 2; i += 32) out[i] = *reinterpret_cast<const uint16_t *>(ow + 2 * i);
        __syncwarp();
    }
}

// ---------------------------------------------------------- dequantization
__global__ void __launch_bounds__(kQ6Threads) qmm_dequantize_q6_k_kernel(const uint8_t *__restrict__ src,
                                                                         float *__restrict__ dst,
                                                                         int64_t nblocks) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int64_t b = (int64_t)blockIdx.x * (kQ6Threads / 32) + warp; b < nblocks;
         b += (int64_t)gridDim.x * (kQ6Threads / 32)) {
        const uint8_t *blk = src + b * kQ6Bytes;
        float c[8];
        q6_lane_codes(blk, lane, c);
        const float S = q6_lane_scale(blk, lane);
        // weights 8l .. 8l + 7 of the superblock = 128 h + 32 s + 8 (l % 4) + e
        const int h = lane >> 4, s = (lane >> 2) & 3, o = 8 * (lane & 3);
        float4 *y = reinterpret_cast<float4 *>(dst + b * 256 + 128 * h + 32 * s + o);
        y[0] = make_float4(S * c[0], S * c[1], S * c[2], S * c[3]);
        y[1] = make_float4(S * c[4], S * c[5], S * c[6], S * c[7]);
    }
}

// ------------------------------------------------------------------ matmul
// Y[M x N] = X[M x K] W^T, W Q6_K.  A warp owns one weight row at a time
// (grid-stride over rows) and up to kTok tokens; lane l takes weights
// 8l .. 8l + 7 of every superblock: exact integer codes times the fp32
// activations, the sub-block scale applied per superblock, fp32 sums reduced
// across the warp at the end of the row.  Four superblocks are loaded before
// any is used, so that their loads are in flight together.  Tokens beyond
// kTok run in further passes over the row.
template <int kTok>
__global__ void __launch_bounds__(kQ6Threads) qmm_matmul_q6_k_kernel(const uint8_t *__restrict__ W,
                                                                     const uint16_t *__restrict__ X,
                                                                     float *__restrict__ Y, int M, int N,
                                                                     int K) {
    constexpr int kU = 4;  // superblocks in flight per lane
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nsb = K / 256;
    const int64_t row_bytes = (int64_t)nsb * kQ6Bytes;
    const int h = lane >> 4, s = (lane >> 2) & 3, o = 8 * (lane & 3);
    const int koff = 128 * h + 32 * s + o;  // first k of this lane in a superblock
    for (int64_t n = (int64_t)blockIdx.x * (kQ6Threads / 32) + warp; n < N;
         n += (int64_t)gridDim.x * (kQ6Threads / 32)) {
        const uint8_t *row = W + n * row_bytes;
        for (int m0 = 0; m0 < M; m0 += kTok) {
            const int mt = min(kTok, M - m0);
            float acc[kTok];
#pragma unroll
            for (int t = 0; t < kTok; ++t) acc[t] = 0.f;
            for (int sb0 = 0; sb0 < nsb; sb0 += kU) {
                float c[kU][8], S[kU];
#pragma unroll
                for (int u = 0; u < kU; ++u) {
                    if (sb0 + u < nsb) {
                        const uint8_t *blk = row + (int64_t)(sb0 + u) * kQ6Bytes;
                        q6_lane_codes(blk, lane, c[u]);
                        S[u] = q6_lane_scale(blk, lane);
                    }
                }
#pragma unroll
                for (int t = 0; t < kTok; ++t) {
                    if (t < mt) {
#pragma unroll
                        for (int u = 0; u < kU; ++u) {
                            if (sb0 + u < nsb) {
                                const uint4 xv = __ldg(reinterpret_cast<const uint4 *>(
                                    X + (int64_t)(m0 + t) * K + (int64_t)(sb0 + u) * 256 + koff));
                                const uint32_t w[4] = {xv.x, xv.y, xv.z, xv.w};
                                acc[t] = fmaf(S[u], q6_codes_dot(c[u], w), acc[t]);
                            }
                        }
                    }
                }
            }
#pragma unroll
            for (int t = 0; t < kTok; ++t) {
                float v = acc[t];
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
                if (lane == 0 && t < mt) Y[(int64_t)(m0 + t) * N + n] = v;
            }
        }
    }
}

// ---------------------------------------------------------- embedding lookup
// out[t][0 .. D) = the dequantized row ids[t] of the packed table [V x D]: one
// warp per (token, 256-column group).  An id outside 0 .. V-1 writes zeros
// and records kErrBadId.
template <int kFmt, bool kBf16>
__global__ void __launch_bounds__(kQ6Threads) qmm_embedding_kernel(const uint8_t *__restrict__ table,
                                                                   const int64_t *__restrict__ ids,
                                                                   void *__restrict__ out, int64_t T,
                                                                   int64_t V, int64_t D) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t groups = D / 256;
    constexpr int kGB = kFmt == 8 ? kQ8GroupBytes : kFmt == 4 ? kQ4Bytes : kFmt == 6 ? kQ6Bytes : 256;
    const int64_t row_bytes = kFmt == kFp8 ? D + kFp8RowPad : groups * kGB;
    for (int64_t u = (int64_t)blockIdx.x * (kQ6Threads / 32) + warp; u < T * groups;
         u += (int64_t)gridDim.x * (kQ6Threads / 32)) {
        const int64_t t = u / groups, g = u - t * groups;
        const int64_t id = __ldg(ids + t);
        float v[8];
        int k0;  // first of the lane's 8 consecutive columns within the group
        if (id < 0 || id >= V) {
            if (lane == 0) record_error(kErrBadId);
#pragma unroll
            for (int e = 0; e < 8; ++e) v[e] = 0.f;
            k0 = 8 * lane;
        } else {
            const uint8_t *grp = table + id * row_bytes + g * kGB;
            if constexpr (kFmt == kFp8) {
                // codes 8 lane .. 8 lane + 7 of the group, times the row scale
                const float sc = __ldg(reinterpret_cast<const float *>(table + id * row_bytes + D));
                const uint2 q = __ldg(reinterpret_cast<const uint2 *>(grp + 8 * lane));
                const uint32_t w[2] = {q.x, q.y};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const uint32_t h2 = e4m3x2_to_h2(w[e >> 1] >> (16 * (e & 1)));
                    v[2 * e] = __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu))) * sc;
                    v[2 * e + 1] = __half2float(__ushort_as_half((unsigned short)(h2 >> 16))) * sc;
                }
                k0 = 8 * lane;
            } else if constexpr (kFmt == 8) {
                // block lane / 4, codes 8 (lane % 4) .. + 7
                const uint8_t *blk = grp + kQ8Bytes * (lane >> 2);
                const float d = __half2float(__ushort_as_half(__ldg(reinterpret_cast<const uint16_t *>(blk))));
                const uint2 q = ld8_a2(blk + 2 + 8 * (lane & 3));
                const uint32_t w[2] = {q.x, q.y};
#pragma unroll
                for (int e = 0; e < 8; ++e) v[e] = d * (float)(int8_t)((w[e >> 2] >> (8 * (e & 3))) & 0xFF);
                k0 = 8 * lane;
            } else if constexpr (kFmt == 4) {
                // sub-block j = lane / 4: bytes 32 (j / 2) + 8 (lane % 4) .. + 7, nibble j % 2
                const int j = lane >> 2;
                const uint4 hd = __ldg(reinterpret_cast<const uint4 *>(grp));
                const float d = __half2float(__ushort_as_half((unsigned short)(hd.x & 0xFFFF)));
                const float dmin = __half2float(__ushort_as_half((unsigned short)(hd.x >> 16)));
                auto sbyte = [&](int k) {
                    const uint32_t w = k < 4 ? hd.y : (k < 8 ? hd.z : hd.w);
                    return (w >> (8 * (k & 3))) & 0xFFu;
                };
                uint32_t sc, mc;
                if (j < 4) {
                    sc = sbyte(j) & 63u;
                    mc = sbyte(j + 4) & 63u;
                } else {
                    sc = (sbyte(j + 4) & 15u) | ((sbyte(j - 4) >> 6) << 4);
                    mc = (sbyte(j + 4) >> 4) | ((sbyte(j) >> 6) << 4);
                }
                const float S = d * (float)sc, Mn = dmin * (float)mc;
                const uint2 q = __ldg(reinterpret_cast<const uint2 *>(grp + 16 + 32 * (j >> 1) + 8 * (lane & 3)));
                const uint32_t w[2] = {q.x, q.y};
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const uint32_t code = (w[e >> 2] >> (8 * (e & 3) + 4 * (j & 1))) & 15u;
                    v[e] = S * (float)code - Mn;
                }
                k0 = 32 * j + 8 * (lane & 3);
            } else {
                float c[8];
                q6_lane_codes(grp, lane, c);
                const float S = q6_lane_scale(grp, lane);
#pragma unroll
                for (int e = 0; e < 8; ++e) v[e] = S * c[e];
                k0 = 128 * (lane >> 4) + 32 * ((lane >> 2) & 3) + 8 * (lane & 3);
            }
        }
        const int64_t base = t * D + g * 256 + k0;
        if constexpr (kBf16) {
            uint32_t pk[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const __nv_bfloat162 b2 = __floats2bfloat162_rn(v[2 * e], v[2 * e + 1]);
                pk[e] = *reinterpret_cast<const uint32_t *>(&b2);
            }
            *reinterpret_cast<uint4 *>(static_cast<uint16_t *>(out) + base) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        } else {
            float4 *y = reinterpret_cast<float4 *>(static_cast<float *>(out) + base);
            y[0] = make_float4(v[0], v[1], v[2], v[3]);
            y[1] = make_float4(v[4], v[5], v[6], v[7]);
        }
    }
}

// ----------------------------------------------------------------- launchers
static int q6_grid(int64_t warps_of_work, int sms) {
    int64_t g = (warps_of_work + (kQ6Threads / 32) - 1) / (kQ6Threads / 32);
    const int64_t cap = (int64_t)sms * 8;
    if (g > cap) g = cap;
    return g < 1 ? 1 : (int)g;
}

cudaError_t launch_q6k_quantize(int src_f32, const void *src, void *dst, int64_t nweights, int sms,
                                cudaStream_t stream) {
    const int64_t nb = nweights / 256;
    const int grid = q6_grid(nb, sms);
    if (src_f32)
        qmm_quantize_q6_k_kernel<true><<<grid, kQ6Threads, 0, stream>>>(src, static_cast<uint8_t *>(dst), nb);
    else
        qmm_quantize_q6_k_kernel<false><<<grid, kQ6Threads, 0, stream>>>(src, static_cast<uint8_t *>(dst), nb);
    return cudaGetLastError();
}

cudaError_t launch_q6k_dequantize(const void *src, float *dst, int64_t nweights, int sms, cudaStream_t stream) {
    const int64_t nb = nweights / 256;
    qmm_dequantize_q6_k_kernel<<<q6_grid(nb, sms), kQ6Threads, 0, stream>>>(static_cast<const uint8_t *>(src),
                                                                            dst, nb);
    return cudaGetLastError();
}

cudaError_t launch_q6k_matmul(const void *W, const uint16_t *X, float *Y, int M, int N, int K, int sms,
                              cudaStream_t stream) {
    const uint8_t *w = static_cast<const uint8_t *>(W);
    const int grid = q6_grid(N, sms);
    if (M == 1)
        qmm_matmul_q6_k_kernel<1><<<grid, kQ6Threads, 0, stream>>>(w, X, Y, M, N, K);
    else if (M <= 8)
        qmm_matmul_q6_k_kernel<8><<<grid, kQ6Threads, 0, stream>>>(w, X, Y, M, N, K);
    else
        qmm_matmul_q6_k_kernel<16><<<grid, kQ6Threads, 0, stream>>>(w, X, Y, M, N, K);
    return cudaGetLastError();
}

template <int kFmt>
static cudaError_t launch_embedding_t(const void *table, const int64_t *ids, void *out, int bf16, int64_t T,
                                      int64_t V, int64_t D, int sms, cudaStream_t stream) {
    const int grid = q6_grid(T * (D / 256), sms);
    const uint8_t *tb = static_cast<const uint8_t *>(table);
    if (bf16)
        qmm_embedding_kernel<kFmt, true><<<grid, kQ6Threads, 0, stream>>>(tb, ids, out, T, V, D);
    else
        qmm_embedding_kernel<kFmt, false><<<grid, kQ6Threads, 0, stream>>>(tb, ids, out, T, V, D);
    return cudaGetLastError();
}

cudaError_t launch_embedding(int fmt, const void *table, const int64_t *ids, void *out, int bf16, int64_t T,
                             int64_t V, int64_t D, int sms, cudaStream_t stream) {
    if (fmt == 8) return launch_embedding_t<8>(table, ids, out, bf16, T, V, D, sms, stream);
    if (fmt == 4) return launch_embedding_t<4>(table, ids, out, bf16, T, V, D, sms, stream);
    if (fmt == kFp8) return launch_embedding_t<kFp8>(table, ids, out, bf16, T, V, D, sms, stream);
    return launch_embedding_t<6>(table, ids, out, bf16, T, V, D, sms, stream);
}

}  // namespace qmm
