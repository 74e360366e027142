// gemv_rows.cu -- decode matmul for M <= 16 tokens without thread-block
// clusters: persistent CTAs, each owning whole 16-row tiles over all of K.
//
// CTA b takes the row tiles b, b + G, b + 2G, ... (G = grid size, at most
// the number of CTAs resident on the GPU at once), so the weight stream of a
// CTA runs on from one tile into the next without a CTA launch, a ring
// refill or an activation restage in between.
//  * Producer warp (one thread): first the activations (bf16, one 1-D bulk
//    copy per token row), then one 2-D tensor-map TMA copy per stage of
//    16 rows x 2 chunks of 256 weights (8.5 KB Q8_0, 4.5 KB Q4_K, 5.5 KB
//    Q5_K).  In shared
//    memory a stage row is 544 / 288 bytes long, which puts the 8 rows read by
//    one 64-bit load of a warp on distinct banks.
//  * Eight consumer warps: chunk i of a tile goes to warp i mod 8, so the two
//    chunks of a stage go to the warp pair (2p, 2p + 1), p = stage mod 4.
//    Every pair has its own sub-ring of stages, so a stage is only ever
//    reused by the warps that consumed it (an mbarrier parity wait cannot
//    tell phase k from k + 2).  The activations are converted in place to
//    binary16 once per CTA (when all of K fits; otherwise once per tile and
//    window of K).  Per chunk: exact integer codes on m16n8k16 tensor-core
//    MMAs, scales in fp32 per 32-weight block (see gemv.cu).
//  * Reducer warp: at the end of a tile each consumer warp leaves its
//    partial sums in a double-buffered shared array and moves on; the reducer
//    adds the eight partials in warp order (deterministic) and stores the
//    tile's outputs.  There is no cluster and no workspace.
// Q8_0 / Q4_K use it when the row tiles alone fill the GPU's SMs, for up to
// 8 tokens (one 8-token MMA column tile) or, while up to 128 KB of
// activations stay resident, up to 16 (two tiles); Q5_K and FP8 (which have
// no cluster kernel) for every M <= 16.  The ring depth, the consumer warps
// and the activation window are planned per (M, K) from the resident CTAs
// per SM.
#include <atomic>
#include <mutex>

#include "common.cuh"

namespace qmm {

constexpr int kRowsR = 16;
// Consumer warps per CTA: 8, or 16 when only one CTA fits on an SM (many
// tokens or a long K keep a large activation window resident); warp pairs
// are half that, then the producer warp and the reducer warp.
template <int kW> struct RowsWarps {
    static constexpr int kPairs = kW / 2, kProd = kW, kRed = kW + 1, kThreads = (kW + 2) * 32;
};
constexpr int kYBufsR = 2;
constexpr int kCoefStrideR = 20;  // floats per row of a warp's Q4_K coefficient table (padded)
// Activations held in shared memory at once: M * window chunks <= 256
// (128 KB of binary16; one CTA per SM then, but no per-tile restaging).
#ifndef QMM_ROWS_X_BUDGET
#define QMM_ROWS_X_BUDGET 256
#endif
constexpr int kRowsXChunkBudget = QMM_ROWS_X_BUDGET;

struct RowsLayout {
    int ring, xh, xs, coef, ypart, bars, total;
};

// Bytes a chunk advances in a packed row, and half the shared-memory pitch of
// a stage row (FP8: two 256-byte chunks plus 32 bytes of the next, a 544-byte
// pitch that keeps a warp's code loads on distinct banks, as Q8_0's does).
// Q5_K: a 176-byte superblock per chunk, pitch 352 (88 words: the 8 rows of a
// half-warp's 64-bit code loads land on distinct banks, as for Q4_K).
constexpr int kQ5Bytes = 176;
__host__ __device__ constexpr int rows_chunk_bytes(int fmt) {
    return fmt == 8 ? kQ8GroupBytes : fmt == 4 ? kQ4Bytes : fmt == 5 ? kQ5Bytes : 256;
}
__host__ __device__ constexpr int rows_half_pitch(int fmt) {
    return fmt == 4 ? kQ4Bytes : fmt == 5 ? kQ5Bytes : kQ8GroupBytes;
}
// the affine formats (codes times a sub-block scale minus a sub-block min)
__host__ __device__ constexpr bool rows_affine(int fmt) { return fmt == 4 || fmt == 5; }

// mt = 8 * (token tiles): the stride of the Q4_K block sums per 32-block.
__host__ __device__ inline RowsLayout rows_layout(int fmt, int M, int dpp, int win, int mt, int nw) {
    const int cb = rows_half_pitch(fmt);
    RowsLayout L;
    int off = 0;
    L.ring = off;
    off += (nw / 2) * dpp * kRowsR * 2 * cb;  // a stage: 16 rows x 2 chunks (multiple of 128 bytes)
    L.xh = off;
    off += M * (win * kGroup + 32) * 2;       // token rows, 32 halves of padding between them
    L.xs = off;
    off += rows_affine(fmt) ? win * 8 * mt * 4 : 0;   // Q4_K / Q5_K: sum of x per 32-block and token
    L.coef = off;
    off += rows_affine(fmt) ? nw * kRowsR * kCoefStrideR * 4 : 0;
    L.ypart = off;
    off += kYBufsR * nw * kRowsR * M * 4;
    off = (off + 15) & ~15;
    L.bars = off;
    off += (2 * (nw / 2) * dpp + 2 + 2 * kYBufsR) * 8;
    L.total = off;
    return L;
}

struct RowsParams {
    float *Y;
    const uint16_t *X;
    const uint8_t *W;   // FP8: the packed rows, for the row scales
    int64_t row_bytes;  // packed bytes per row
    int M, N, K;
    int nchunks;  // K / 256
    int ntiles;   // ceil(N / 16)
    int dpp;      // ring stages per warp pair
    int win;      // activation window in chunks: nchunks, or a multiple of 8
};

// Convert the raw bf16 activations of a window, landed by TMA at xh (token m
// at xh + m * xstride), in place to binary16 (round to nearest), each group
// of 4 stored in the order (0, 2, 1, 3) so that one 16-byte load yields both
// B fragments of an MMA; Q4_K and Q5_K also sum each 32-weight block per token.
template <int kFmt, int kMT, int kW>
__device__ __forceinline__ void rows_convert_x(int M, __half *xh, float *xs, int xstride, int wn,
                                               int tid) {
    const int ngr = (wn * kGroup) / 8;  // 8-element groups per token
    int m = 0, kg = tid;
    while (kg >= ngr && m < M) { kg -= ngr; ++m; }
    for (; m < M;) {
        uint4 *p = reinterpret_cast<uint4 *>(xh + m * xstride + 8 * kg);
        const uint4 v = *p;
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        float f[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            f[2 * e] = __uint_as_float(w[e] << 16);
            f[2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
        }
        const __half2 h02 = __floats2half2_rn(f[0], f[2]);
        const __half2 h13 = __floats2half2_rn(f[1], f[3]);
        const __half2 h46 = __floats2half2_rn(f[4], f[6]);
        const __half2 h57 = __floats2half2_rn(f[5], f[7]);
        uint4 o;
        o.x = *reinterpret_cast<const uint32_t *>(&h02);
        o.y = *reinterpret_cast<const uint32_t *>(&h13);
        o.z = *reinterpret_cast<const uint32_t *>(&h46);
        o.w = *reinterpret_cast<const uint32_t *>(&h57);
        *p = o;
        if constexpr (rows_affine(kFmt)) {
            // lanes 4j .. 4j + 3 hold one 32-weight block (ngr is a multiple of 32)
            const float2 s02 = __half22float2(h02), s13 = __half22float2(h13);
            const float2 s46 = __half22float2(h46), s57 = __half22float2(h57);
            float sum = ((s02.x + s13.x) + (s02.y + s13.y)) + ((s46.x + s57.x) + (s46.y + s57.y));
            sum += __shfl_xor_sync(0xffffffffu, sum, 1);
            sum += __shfl_xor_sync(0xffffffffu, sum, 2);
            if ((kg & 3) == 0) xs[(kg >> 2) * kMT + m] = sum;
        }
        kg += kW * 32;
        while (kg >= ngr && m < M) { kg -= ngr; ++m; }
    }
}

// 8 code bytes at shared address p with p mod 8 == kMod8, as two words,
// using 8-byte loads where the alignment allows.
template <int kMod8>
__device__ __forceinline__ void rq8_codes(const uint8_t *p, uint32_t &w0, uint32_t &w1) {
    if constexpr (kMod8 == 0) {
        const uint2 v = *reinterpret_cast<const uint2 *>(p);
        w0 = v.x;
        w1 = v.y;
    } else if constexpr (kMod8 == 4) {
        w0 = *reinterpret_cast<const uint32_t *>(p);
        w1 = *reinterpret_cast<const uint32_t *>(p + 4);
    } else if constexpr (kMod8 == 2) {  // bytes 2..9 of [p - 2, p + 14)
        const uint2 a = *reinterpret_cast<const uint2 *>(p - 2);
        const uint2 b = *reinterpret_cast<const uint2 *>(p + 6);
        w0 = __byte_perm(a.x, a.y, 0x5432);
        w1 = __byte_perm(a.y, b.x, 0x5432);
    } else {  // 6: bytes 2..9 of [p - 2, p + 10)
        const uint32_t a = *reinterpret_cast<const uint32_t *>(p - 2);
        const uint2 b = *reinterpret_cast<const uint2 *>(p + 2);
        w0 = __byte_perm(a, b.x, 0x5432);
        w1 = __byte_perm(b.x, b.y, 0x5432);
    }
}

// One Q8_0 block (32 weights) of rows g and g + 8 (row bases r0, r1, 16-byte
// aligned) against tokens g + 8 nt (nt < kNT) at xb + nt * 8 * xstride,
// present when v0 (nt = 0) / v1 (nt = 1).
template <int kB, int kNT>
__device__ __forceinline__ void rq8_block(const uint8_t *r0, const uint8_t *r1, const __half *xb, int xstride,
                                          int t, bool v0, bool v1, float (&acc)[kNT][4]) {
    constexpr int kOff = kQ8Bytes * kB + 2;
    constexpr int kMod8 = kOff % 8;
    const float d0 = h2f_bits(*reinterpret_cast<const uint16_t *>(r0 + kQ8Bytes * kB));
    const float d1 = h2f_bits(*reinterpret_cast<const uint16_t *>(r1 + kQ8Bytes * kB));
    uint32_t a0, a1, b0, b1;
    rq8_codes<kMod8>(r0 + kOff + 8 * t, a0, a1);
    rq8_codes<kMod8>(r1 + kOff + 8 * t, b0, b1);
    a0 ^= 0x80808080u; a1 ^= 0x80808080u; b0 ^= 0x80808080u; b1 ^= 0x80808080u;
    const uint32_t A0[4] = {q8_exact(q8_pair02(a0)), q8_exact(q8_pair02(b0)),
                            q8_exact(q8_pair13(a0)), q8_exact(q8_pair13(b0))};
    const uint32_t A1[4] = {q8_exact(q8_pair02(a1)), q8_exact(q8_pair02(b1)),
                            q8_exact(q8_pair13(a1)), q8_exact(q8_pair13(b1))};
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt) {
        const uint4 xv = x_frag(xb + nt * 8 * xstride + kQ8Weights * kB + 8 * t, nt == 0 ? v0 : v1);
        float c[4] = {0.f, 0.f, 0.f, 0.f};
        mma_f16_16816(c, A0, xv.x, xv.y);
        mma_f16_16816(c, A1, xv.z, xv.w);
        acc[nt][0] = fmaf(d0, c[0], acc[nt][0]);
        acc[nt][1] = fmaf(d0, c[1], acc[nt][1]);
        acc[nt][2] = fmaf(d1, c[2], acc[nt][2]);
        acc[nt][3] = fmaf(d1, c[3], acc[nt][3]);
    }
}

// FP8 E4M3: one 32-weight block of rows g and g + 8, the lane's codes 8t ..
// 8t + 7 paired (0, 2), (1, 3) like the staged activations; the codes convert
// exactly to binary16 and there is no block scale (the row scale is applied
// to the finished sums).  Each block's two MMAs start from zero and are then
// added to acc, which keeps the MMA dependency chains two long.
template <int kB, int kNT>
__device__ __forceinline__ void r8_block(const uint8_t *r0, const uint8_t *r1, const __half *xb, int xstride,
                                         int t, bool v0, bool v1, float (&acc)[kNT][4]) {
    const uint2 a = *reinterpret_cast<const uint2 *>(r0 + 32 * kB + 8 * t);
    const uint2 b = *reinterpret_cast<const uint2 *>(r1 + 32 * kB + 8 * t);
    // bytes (0, 2) and (1, 3) of a word as one E4M3 pair each
    auto p02 = [](uint32_t w) { return e4m3x2_to_h2(prmt(w, 0u, 0x4420u)); };
    auto p13 = [](uint32_t w) { return e4m3x2_to_h2(prmt(w, 0u, 0x4431u)); };
    const uint32_t A0[4] = {p02(a.x), p02(b.x), p13(a.x), p13(b.x)};
    const uint32_t A1[4] = {p02(a.y), p02(b.y), p13(a.y), p13(b.y)};
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt) {
        const uint4 xv = x_frag(xb + nt * 8 * xstride + kQ8Weights * kB + 8 * t, nt == 0 ? v0 : v1);
        float c[4] = {0.f, 0.f, 0.f, 0.f};
        mma_f16_16816(c, A0, xv.x, xv.y);
        mma_f16_16816(c, A1, xv.z, xv.w);
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[nt][e] += c[e];
    }
}

// Q4_K scale/min decode of one chunk (16 rows x 8 sub-blocks): lane r + 16 h
// decodes row r, sub-blocks 4h .. 4h + 3, with word-parallel unpacking of the
// 6-bit fields; writes (S_j * 2^24 or S_j * 2^20, -Mn_j) pairs to cw.
__device__ __forceinline__ void rq4_coefs(const uint8_t *row0, int pitch, float *cw, int lane) {
    const int r = lane & 15, h = lane >> 4;
    const uint4 hd = *reinterpret_cast<const uint4 *>(row0 + r * pitch);
    const float d = h2f_bits(hd.x), dmin = h2f_bits(hd.x >> 16);
    const uint32_t sc = h ? ((hd.w & 0x0F0F0F0Fu) | ((hd.y >> 2) & 0x30303030u)) : (hd.y & 0x3F3F3F3Fu);
    const uint32_t mc = h ? (((hd.w >> 4) & 0x0F0F0F0Fu) | ((hd.z >> 2) & 0x30303030u)) : (hd.z & 0x3F3F3F3Fu);
    // byte b -> 2^23 + b as a float, then one fma: (2^23 + b) * s - 2^23 * s = b * s, exact
    const float dlo = d * 16777216.0f, dhi = d * 1048576.0f;  // even / odd sub-block (low / high nibble)
    float o[8];
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
        const float fs = __uint_as_float(__byte_perm(sc, 0x4B000000u, 0x7540 + jj));
        const float fm = __uint_as_float(__byte_perm(mc, 0x4B000000u, 0x7540 + jj));
        const float ds = (jj & 1) ? dhi : dlo;
        o[2 * jj] = fmaf(fs, ds, -8388608.0f * ds);
        o[2 * jj + 1] = fmaf(fm, -dmin, 8388608.0f * dmin);
    }
    float4 *dst = reinterpret_cast<float4 *>(cw + r * kCoefStrideR + 8 * h);
    dst[0] = make_float4(o[0], o[1], o[2], o[3]);
    dst[1] = make_float4(o[4], o[5], o[6], o[7]);
}

// 64 weights (sub-blocks 2c, 2c + 1) of rows g and g + 8 of a Q4_K chunk;
// xsb: the chunk's block sums, stride 8 kNT per 32-block.
template <int kC, int kNT>
__device__ __forceinline__ void rq4_group(const uint8_t *r0, const uint8_t *r1, const __half *xb, int xstride,
                                          const float *xsb, const float *cw, int g, int t, bool v0, bool v1,
                                          float (&acc)[kNT][4]) {
    constexpr int kMT = 8 * kNT;
    const uint2 qa = *reinterpret_cast<const uint2 *>(r0 + 16 + 32 * kC + 8 * t);
    const uint2 qb = *reinterpret_cast<const uint2 *>(r1 + 16 + 32 * kC + 8 * t);
    const float4 ca = *reinterpret_cast<const float4 *>(cw + g * kCoefStrideR + 4 * kC);
    const float4 cb = *reinterpret_cast<const float4 *>(cw + (g + 8) * kCoefStrideR + 4 * kC);
    const uint32_t qa0s = qa.x >> 8, qa1s = qa.y >> 8, qb0s = qb.x >> 8, qb1s = qb.y >> 8;
    // masked nibble pairs are binary16 subnormals: q * 2^-24 (low), q * 2^-20 (high)
    const uint32_t L0[4] = {qa.x & 0x000F000Fu, qb.x & 0x000F000Fu, qa0s & 0x000F000Fu, qb0s & 0x000F000Fu};
    const uint32_t L1[4] = {qa.y & 0x000F000Fu, qb.y & 0x000F000Fu, qa1s & 0x000F000Fu, qb1s & 0x000F000Fu};
    const uint32_t H0[4] = {qa.x & 0x00F000F0u, qb.x & 0x00F000F0u, qa0s & 0x00F000F0u, qb0s & 0x00F000F0u};
    const uint32_t H1[4] = {qa.y & 0x00F000F0u, qb.y & 0x00F000F0u, qa1s & 0x00F000F0u, qb1s & 0x00F000F0u};
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt) {
        const __half *xq = xb + nt * 8 * xstride + 64 * kC + 8 * t;
        const uint4 xl = x_frag(xq, nt == 0 ? v0 : v1);
        const uint4 xhv = x_frag(xq + 32, nt == 0 ? v0 : v1);
        float cl[4] = {0.f, 0.f, 0.f, 0.f}, chh[4] = {0.f, 0.f, 0.f, 0.f};
        mma_f16_16816(cl, L0, xl.x, xl.y);
        mma_f16_16816(cl, L1, xl.z, xl.w);
        mma_f16_16816(chh, H0, xhv.x, xhv.y);
        mma_f16_16816(chh, H1, xhv.z, xhv.w);
        const float2 sl = *reinterpret_cast<const float2 *>(xsb + (2 * kC) * kMT + nt * 8 + 2 * t);
        const float2 sh = *reinterpret_cast<const float2 *>(xsb + (2 * kC + 1) * kMT + nt * 8 + 2 * t);
        acc[nt][0] = fmaf(ca.w, sh.x, fmaf(ca.y, sl.x, fmaf(ca.z, chh[0], fmaf(ca.x, cl[0], acc[nt][0]))));
        acc[nt][1] = fmaf(ca.w, sh.y, fmaf(ca.y, sl.y, fmaf(ca.z, chh[1], fmaf(ca.x, cl[1], acc[nt][1]))));
        acc[nt][2] = fmaf(cb.w, sh.x, fmaf(cb.y, sl.x, fmaf(cb.z, chh[2], fmaf(cb.x, cl[2], acc[nt][2]))));
        acc[nt][3] = fmaf(cb.w, sh.y, fmaf(cb.y, sl.y, fmaf(cb.z, chh[3], fmaf(cb.x, cl[3], acc[nt][3]))));
    }
}

// Q5_K: rq4_group's 64 weights with 5-bit codes.  The chunk's codes sit at
// byte 48 (16 of header, 32 of qh before them); bit j of qh byte l is bit 4
// of weight l of sub-block j.  qh* hold the lane's qh bytes 8t .. 8t + 7 of
// rows g and g + 8, qh*8 the same shifted down a byte (the odd bytes).  The
// fifth bit joins the subnormal binary16 codes: bit 4 under the low nibble
// (q * 2^-24), bit 8 under the high one (q * 2^-20), so rq4_coefs' scales
// apply unchanged.
template <int kSh>
__device__ __forceinline__ uint32_t shl_c(uint32_t v) {
    if constexpr (kSh >= 0) return v << kSh;
    else return v >> -kSh;
}
template <int kC, int kNT>
__device__ __forceinline__ void rq5_group(const uint8_t *r0, const uint8_t *r1, uint2 qha, uint2 qhb, uint2 qha8,
                                          uint2 qhb8, const __half *xb, int xstride, const float *xsb,
                                          const float *cw, int g, int t, bool v0, bool v1,
                                          float (&acc)[kNT][4]) {
    constexpr int kMT = 8 * kNT;
    const uint2 qa = *reinterpret_cast<const uint2 *>(r0 + 48 + 32 * kC + 8 * t);
    const uint2 qb = *reinterpret_cast<const uint2 *>(r1 + 48 + 32 * kC + 8 * t);
    const float4 ca = *reinterpret_cast<const float4 *>(cw + g * kCoefStrideR + 4 * kC);
    const float4 cb = *reinterpret_cast<const float4 *>(cw + (g + 8) * kCoefStrideR + 4 * kC);
    const uint32_t qa0s = qa.x >> 8, qa1s = qa.y >> 8, qb0s = qb.x >> 8, qb1s = qb.y >> 8;
    // sub-block 2c: low nibble | qh bit 2c at bit 4; sub-block 2c + 1: high nibble | qh bit 2c + 1 at bit 8
    auto lo = [](uint32_t q, uint32_t h) { return (q & 0x000F000Fu) | (shl_c<4 - 2 * kC>(h) & 0x00100010u); };
    auto hi = [](uint32_t q, uint32_t h) { return (q & 0x00F000F0u) | (shl_c<7 - 2 * kC>(h) & 0x01000100u); };
    const uint32_t L0[4] = {lo(qa.x, qha.x), lo(qb.x, qhb.x), lo(qa0s, qha8.x), lo(qb0s, qhb8.x)};
    const uint32_t L1[4] = {lo(qa.y, qha.y), lo(qb.y, qhb.y), lo(qa1s, qha8.y), lo(qb1s, qhb8.y)};
    const uint32_t H0[4] = {hi(qa.x, qha.x), hi(qb.x, qhb.x), hi(qa0s, qha8.x), hi(qb0s, qhb8.x)};
    const uint32_t H1[4] = {hi(qa.y, qha.y), hi(qb.y, qhb.y), hi(qa1s, qha8.y), hi(qb1s, qhb8.y)};
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt) {
        const __half *xq = xb + nt * 8 * xstride + 64 * kC + 8 * t;
        const uint4 xl = x_frag(xq, nt == 0 ? v0 : v1);
        const uint4 xhv = x_frag(xq + 32, nt == 0 ? v0 : v1);
        float cl[4] = {0.f, 0.f, 0.f, 0.f}, chh[4] = {0.f, 0.f, 0.f, 0.f};
        mma_f16_16816(cl, L0, xl.x, xl.y);
        mma_f16_16816(cl, L1, xl.z, xl.w);
        mma_f16_16816(chh, H0, xhv.x, xhv.y);
        mma_f16_16816(chh, H1, xhv.z, xhv.w);
        const float2 sl = *reinterpret_cast<const float2 *>(xsb + (2 * kC) * kMT + nt * 8 + 2 * t);
        const float2 sh = *reinterpret_cast<const float2 *>(xsb + (2 * kC + 1) * kMT + nt * 8 + 2 * t);
        acc[nt][0] = fmaf(ca.w, sh.x, fmaf(ca.y, sl.x, fmaf(ca.z, chh[0], fmaf(ca.x, cl[0], acc[nt][0]))));
        acc[nt][1] = fmaf(ca.w, sh.y, fmaf(ca.y, sl.y, fmaf(ca.z, chh[1], fmaf(ca.x, cl[1], acc[nt][1]))));
        acc[nt][2] = fmaf(cb.w, sh.x, fmaf(cb.y, sl.x, fmaf(cb.z, chh[2], fmaf(cb.x, cl[2], acc[nt][2]))));
        acc[nt][3] = fmaf(cb.w, sh.y, fmaf(cb.y, sl.y, fmaf(cb.z, chh[3], fmaf(cb.x, cl[3], acc[nt][3]))));
    }
}

// kNT token tiles of 8 (M <= 8 kNT); two tiles double the accumulators, so
// their register budget allows two CTAs per SM instead of three.
template <int kFmt, int kNT, int kW>
__global__ void __launch_bounds__(RowsWarps<kW>::kThreads, kW == 8 ? (kNT == 1 ? 3 : 2) : 1)
qmm_gemv_rows_kernel(const __grid_constant__ CUtensorMap wmap, const RowsParams p) {
    constexpr int kWarpsR = kW, kPairsR = RowsWarps<kW>::kPairs;
    constexpr int kProdWarpR = RowsWarps<kW>::kProd, kRedWarpR = RowsWarps<kW>::kRed;
    constexpr int kThreadsR = RowsWarps<kW>::kThreads;
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int kCB = rows_chunk_bytes(kFmt);            // a chunk's advance in a packed row
    constexpr int kPitch = 2 * rows_half_pitch(kFmt);      // stage row: two chunks (FP8: + 32 bytes)
    constexpr int kStage = kRowsR * kPitch;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nch = p.nchunks, dpp = p.dpp, win = p.win, M = p.M;
    const bool resident = win >= nch;  // activations staged once per CTA
    const int xstride = win * kGroup + 32;
    const RowsLayout L = rows_layout(kFmt, M, dpp, win, 8 * kNT, kW);
    uint8_t *ring = smem + L.ring;
    __half *xh = reinterpret_cast<__half *>(smem + L.xh);
    float *xs = reinterpret_cast<float *>(smem + L.xs);
    float *ypart = reinterpret_cast<float *>(smem + L.ypart);
    const int nst = kPairsR * dpp;
    const uint32_t bar0 = smem_addr(smem + L.bars);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (nst + s); };
    const uint32_t xfull = bar0 + 16u * nst, xempty = xfull + 8u;
    const uint32_t yfull0 = xempty + 8u, yempty0 = yfull0 + 8u * kYBufsR;

    if (tid == 0) {
        for (int s = 0; s < nst; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 2);
        }
        mbar_init(xfull, 1);
        mbar_init(xempty, kWarpsR);
        for (int b = 0; b < kYBufsR; ++b) {
            mbar_init(yfull0 + 8u * b, kWarpsR);
            mbar_init(yempty0 + 8u * b, 1);
        }
        fence_mbar_init();
    }
    // block sums of padding tokens (m >= M) stay zero for the whole kernel
    constexpr int kMT = 8 * kNT;
    if constexpr (rows_affine(kFmt))
        for (int idx = tid; idx < win * 8 * kMT; idx += kThreadsR) xs[idx] = 0.f;
    if (warp == kProdWarpR && lane == 0) {
        // descriptor fetch and L2 prefetch of the first tile's leading stages
        // (safe before the dependency wait: nothing lands in shared memory)
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&wmap)) : "memory");
        for (int j = 0; 2 * j < nch && j < nst; ++j)
            tma_prefetch_l2_2d(&wmap, 2 * j * (kCB / 8), (int)blockIdx.x * kRowsR);
        // and of the first activation window, which gates every consumer
        for (int m = 0; m < M; ++m)
            bulk_prefetch_l2(p.X + (int64_t)m * p.K, (uint32_t)(min(win, nch) * kGroup * 2));
    }
    __syncthreads();
    // programmatic dependent launch: see gemv.cu
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (warp == kProdWarpR) {
        // ---------------- producer (one thread)
        if (lane == 0) {
            bool ok = true;
            int xseq = 0;
            int dpos[kPairsR], ph[kPairsR];
            bool lap[kPairsR];  // slot used before
#pragma unroll
            for (int i = 0; i < kPairsR; ++i) {
                dpos[i] = ph[i] = 0;
                lap[i] = false;
            }
            for (int tile = blockIdx.x; ok && tile < p.ntiles; tile += gridDim.x) {
                const int row0 = tile * kRowsR;
                for (int w0 = 0; ok && w0 < nch; w0 += win) {
                    const int wn = min(win, nch - w0);
                    if (!resident || xseq == 0) {
                        // the previous window must be fully read before it is overwritten
                        if (xseq > 0 && !mbar_wait(xempty, (xseq - 1) & 1, kErrGemvEmptyWait)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(xfull, (uint32_t)(M * wn * kGroup * 2));
                        for (int m = 0; m < M; ++m)
                            bulk_g2s(smem_addr(xh + m * xstride), p.X + (int64_t)m * p.K + w0 * kGroup,
                                     (uint32_t)(wn * kGroup * 2), xfull);
                        ++xseq;
                    }
                    const int j_end = (w0 + wn + 1) / 2;  // stages of the tile up to this window's end
                    for (int j0 = w0 / 2; ok && j0 < j_end; j0 += kPairsR) {
#pragma unroll
                        for (int pp = 0; pp < kPairsR; ++pp) {
                            if (ok && j0 + pp < j_end) {
                                const int s = pp + kPairsR * dpos[pp];
                                if (lap[pp] && !mbar_wait(empty_bar(s), ph[pp] ^ 1, kErrGemvEmptyWait)) {
                                    ok = false;  // bug path: consumers then time out on their full barriers
                                } else {
                                    // a box may run past K (zero filled); its bytes all count
                                    mbar_arrive_expect_tx(full_bar(s), (uint32_t)kStage);
                                    tma_load_2d(smem_addr(ring + s * kStage), &wmap, 2 * (j0 + pp) * (kCB / 8),
                                                row0, full_bar(s));
                                    if (++dpos[pp] == dpp) {
                                        dpos[pp] = 0;
                                        ph[pp] ^= 1;
                                        lap[pp] = true;
                                    }
                                }
                            }
                        }
                    }
                }
            }
        }
    } else if (warp == kRedWarpR) {
        // ---------------- reducer: fixed-order sum of the eight partials of a tile
        bool ok = true;
        int u = 0;
        for (int tile = blockIdx.x; tile < p.ntiles; tile += gridDim.x, ++u) {
            const int b = u & (kYBufsR - 1);
            const uint32_t yf = yfull0 + 8u * b, ye = yempty0 + 8u * b;
            if (ok) ok = mbar_wait_warp(yf, (u / kYBufsR) & 1, kErrGemvFullWait);
            if (!ok) continue;
            const float *yb = ypart + b * (kWarpsR * kRowsR * M);
            const int row0 = tile * kRowsR;
            for (int idx = lane; idx < kRowsR * M; idx += 32) {
                const int r = idx / M, m = idx - r * M;
                if (row0 + r < p.N) {
                    float sum = 0.f;
#pragma unroll
                    for (int w = 0; w < kWarpsR; ++w) sum += yb[(w * kRowsR + r) * M + m];
                    if constexpr (kFmt == kFp8)  // the row scale follows the row's codes
                        sum *= __ldg(reinterpret_cast<const float *>(p.W + (int64_t)(row0 + r) * p.row_bytes + p.K));
                    p.Y[(int64_t)m * p.N + row0 + r] = sum;
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(ye);
        }
    } else {
        // ---------------- consumers: warp w takes chunks w, w + 8, ... of every tile
        const int g = lane >> 2, t = lane & 3;
        const int pr = warp >> 1, hb = warp & 1;
        const __half *xrow = xh + g * xstride;
        const bool v0 = g < M, v1 = g + 8 < M;  // tokens g and g + 8 are real
        float *cw = reinterpret_cast<float *>(smem + L.coef) + warp * kRowsR * kCoefStrideR;
        bool ok = true;  // warp-uniform, see gemv.cu
        int dpos = 0, ph = 0, xseq = 0, u = 0;
        for (int tile = blockIdx.x; tile < p.ntiles; tile += gridDim.x, ++u) {
            float acc[kNT][4] = {};
            for (int w0 = 0; w0 < nch; w0 += win) {
                const int wn = min(win, nch - w0);
                if (!resident || xseq == 0) {
                    if (ok) ok = mbar_wait_warp(xfull, xseq & 1, kErrGemvFullWait);
                    if (ok) rows_convert_x<kFmt, kMT, kW>(M, xh, xs, xstride, wn, tid);
                    named_bar_sync(1, kWarpsR * 32);
                }
                const int j_end = (w0 + wn + 1) / 2;
                for (int j = w0 / 2 + pr; j < j_end; j += kPairsR) {
                    const int s = pr + kPairsR * dpos;
                    // both warps of the pair wait for the data before releasing
                    // the stage, also when this warp's chunk is past K
                    if (ok) ok = mbar_wait_warp(full_bar(s), ph, kErrGemvFullWait);
                    const int i = 2 * j + hb;
                    if (ok && i < w0 + wn) {
                        const int li = i - w0;
                        const uint8_t *cbase = ring + s * kStage + hb * kCB;  // row r at cbase + r * kPitch
                        const uint8_t *r0 = cbase + g * kPitch;
                        const uint8_t *r1 = cbase + (g + 8) * kPitch;
                        const __half *xb = xrow + li * kGroup;
                        if constexpr (kFmt == kFp8) {
                            r8_block<0, kNT>(r0, r1, xb, xstride, t, v0, v1, acc);
                            r8_block<1, kNT>(r0, r1, xb, xstride, t, v0, v1, acc);
                            r8_block<2, kNT>(r0, r1, xb, xstride, t, v0, v1, acc);
                            r8_block<3, kNT>(r0, r1, xb, xstride, t, v0, v1, acc);
                            r8_block<4, kNT>(r0, r1, xb, xstride, t, v0, v1, acc);
                            r8_block<5, kNT>(r0, r1, xb, xstride, t, v0, v1, acc);
                            r8_block<6, kNT>(r0, r1, xb, xstride, t, v0, v1, acc);
                            r8_block<7, kNT>(r0, r1, xb, xstride, t, v0, v1, acc);
                        } else if constexpr (kFmt == 8) {
                            rq8_block<0, kNT>(r0, r1, xb, xstride, t, v0, v1, acc);
                            rq8_block<1, kNT>(r0, r1, xb, xstride, t, v0, v1, acc);
                            rq8_block<2, kNT>(r0, r1, xb, xstride, t, v0, v1, acc);
                            rq8_block<3, kNT>(r0, r1, xb, xstride, t, v0, v1, acc);
                            rq8_block<4, kNT>(r0, r1, xb, xstride, t, v0, v1, acc);
                            rq8_block<5, kNT>(r0, r1, xb, xstride, t, v0, v1, acc);
                            rq8_block<6, kNT>(r0, r1, xb, xstride, t, v0, v1, acc);
                            rq8_block<7, kNT>(r0, r1, xb, xstride, t, v0, v1, acc);
                        } else if constexpr (kFmt == 5) {
                            rq4_coefs(cbase, kPitch, cw, lane);  // Q5_K's header is Q4_K's
                            __syncwarp();
                            const float *xsb = xs + li * 8 * kMT;
                            const uint2 qha = *reinterpret_cast<const uint2 *>(r0 + 16 + 8 * t);
                            const uint2 qhb = *reinterpret_cast<const uint2 *>(r1 + 16 + 8 * t);
                            const uint2 qha8 = make_uint2(qha.x >> 8, qha.y >> 8);
                            const uint2 qhb8 = make_uint2(qhb.x >> 8, qhb.y >> 8);
                            rq5_group<0, kNT>(r0, r1, qha, qhb, qha8, qhb8, xb, xstride, xsb, cw, g, t, v0, v1, acc);
                            rq5_group<1, kNT>(r0, r1, qha, qhb, qha8, qhb8, xb, xstride, xsb, cw, g, t, v0, v1, acc);
                            rq5_group<2, kNT>(r0, r1, qha, qhb, qha8, qhb8, xb, xstride, xsb, cw, g, t, v0, v1, acc);
                            rq5_group<3, kNT>(r0, r1, qha, qhb, qha8, qhb8, xb, xstride, xsb, cw, g, t, v0, v1, acc);
                        } else {
                            rq4_coefs(cbase, kPitch, cw, lane);
                            __syncwarp();
                            const float *xsb = xs + li * 8 * kMT;
                            rq4_group<0, kNT>(r0, r1, xb, xstride, xsb, cw, g, t, v0, v1, acc);
                            rq4_group<1, kNT>(r0, r1, xb, xstride, xsb, cw, g, t, v0, v1, acc);
                            rq4_group<2, kNT>(r0, r1, xb, xstride, xsb, cw, g, t, v0, v1, acc);
                            rq4_group<3, kNT>(r0, r1, xb, xstride, xsb, cw, g, t, v0, v1, acc);
                        }
                    }
                    __syncwarp();
                    if (ok && lane == 0) mbar_arrive(empty_bar(s));
                    if (++dpos == dpp) {
                        dpos = 0;
                        ph ^= 1;
                    }
                }
                if (!resident) {
                    // this warp is done with the window's activations
                    __syncwarp();
                    if (lane == 0) mbar_arrive(xempty);
                }
                ++xseq;
            }
            // hand the tile's partial sums to the reducer
            const int b = u & (kYBufsR - 1);
            if (ok && u >= kYBufsR)
                ok = mbar_wait_warp(yempty0 + 8u * b, ((u / kYBufsR) - 1) & 1, kErrGemvEmptyWait);
            float *yp = ypart + (b * kWarpsR + warp) * kRowsR * M;
#pragma unroll
            for (int nt = 0; nt < kNT; ++nt) {
                const int m0 = 8 * nt + 2 * t;
                if (m0 < M) {
                    yp[g * M + m0] = acc[nt][0];
                    yp[(g + 8) * M + m0] = acc[nt][2];
                }
                if (m0 + 1 < M) {
                    yp[g * M + m0 + 1] = acc[nt][1];
                    yp[(g + 8) * M + m0 + 1] = acc[nt][3];
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(yfull0 + 8u * b);
        }
    }
}

template <int kFmt, int kNT, int kW>
static cudaError_t rows_set_attrs() {
    static std::atomic<uint64_t> done{0};
    return set_smem_limit_once(reinterpret_cast<const void *>(qmm_gemv_rows_kernel<kFmt, kNT, kW>), 227 * 1024,
                               done);
}

// Resident CTAs per SM for a given dynamic shared-memory size (registers,
// threads and shared memory all counted by the runtime).
template <int kFmt, int kNT, int kW>
static int rows_occupancy(int smem) {
    int n = 0;
    if (rows_set_attrs<kFmt, kNT, kW>() != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, qmm_gemv_rows_kernel<kFmt, kNT, kW>,
                                                      RowsWarps<kW>::kThreads, (size_t)smem) != cudaSuccess)
        return 1;
    return n < 1 ? 1 : n;
}

#ifndef QMM_ROWS_FORCE_DPP  // 0: chosen by the plan
#define QMM_ROWS_FORCE_DPP 0
#endif
#ifndef QMM_ROWS_MAX_DPP
#define QMM_ROWS_MAX_DPP 4
#endif

struct RowsPlan {
    int dev, M, K, dpp, win, smem, occ, warps;
};

// Plan for (M, K) with kW consumer warps: activation window (all of K when
// M * chunks fits the budget), then the sub-ring depth per warp pair with
// the most weight bytes in flight per SM (resident CTAs x ring bytes),
// preferring more resident CTAs on ties.
template <int kFmt, int kNT, int kW>
static RowsPlan rows_plan_warps(int dev, int M, int K) {
    constexpr int kCB = rows_half_pitch(kFmt);
    const int nch = K / kGroup;
    int win = nch;
    if (M * nch > kRowsXChunkBudget) {
        win = (kRowsXChunkBudget / M) / 8 * 8;
        if (win < 8) win = 8;
    }
    RowsPlan best{dev, M, K, 0, win, 0, 0, kW};
    long best_bytes = -1;
    for (int d = 1; d <= QMM_ROWS_MAX_DPP; ++d) {
        if (QMM_ROWS_FORCE_DPP > 0 && d != QMM_ROWS_FORCE_DPP) continue;
        const int sm = rows_layout(kFmt, M, d, win, 8 * kNT, kW).total;
        if (sm > 227 * 1024) break;
        const int occ = rows_occupancy<kFmt, kNT, kW>(sm);
        const long bytes = (long)occ * (kW / 2) * d * kRowsR * 2 * kCB;
        if (bytes > best_bytes || (bytes == best_bytes && occ > best.occ)) {
            best_bytes = bytes;
            best = RowsPlan{dev, M, K, d, win, sm, occ, kW};
        }
    }
    return best;
}

#ifndef QMM_ROWS_WARPS  // 0: chosen by the plan; 8 or 16 forces that many consumer warps
#define QMM_ROWS_WARPS 0
#endif

// Eight consumer warps per CTA while two or more CTAs fit on an SM;
// sixteen when a single CTA does (the activations of many tokens or of a
// long K fill shared memory), which doubles the warps that hide latency.
// Q4_K, whose consumers do the most arithmetic per byte, always gains from
// them; Q8_0 and FP8 only while the ring keeps as many stages in flight
// (eight pairs' rings of one stage can hold fewer than four pairs' deeper
// ones), measured on the decode shapes.
template <int kFmt, int kNT>
static RowsPlan rows_plan_compute(int dev, int M, int K) {
    const RowsPlan p8 = rows_plan_warps<kFmt, kNT, 8>(dev, M, K);
    if (QMM_ROWS_WARPS == 8) return p8;
    if (QMM_ROWS_WARPS != 16 && p8.dpp > 0 && p8.occ > 1) return p8;
    const RowsPlan p16 = rows_plan_warps<kFmt, kNT, 16>(dev, M, K);
    if (p16.dpp == 0) return p8;
    if (QMM_ROWS_WARPS == 16 || p8.dpp == 0 || rows_affine(kFmt)) return p16;
    const long b8 = (long)p8.occ * 4 * p8.dpp, b16 = (long)p16.occ * 8 * p16.dpp;  // stages in flight per SM
    return b16 >= b8 ? p16 : p8;
}

// The plan depends on (device, M, K) only; it is computed once (the
// occupancy queries cost host time) and kept in a small table.
template <int kFmt, int kNT>
static RowsPlan rows_plan(int dev, int M, int K) {
    static std::mutex mu;
    static RowsPlan table[64];
    static int count = 0;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < count; ++i)
        if (table[i].dev == dev && table[i].M == M && table[i].K == K) return table[i];
    const RowsPlan pl = rows_plan_compute<kFmt, kNT>(dev, M, K);
    table[count < 64 ? count++ : (int)(((unsigned)M * 31u + (unsigned)K) % 64u)] = pl;
    return pl;
}

template <int kFmt, int kNT, int kW>
static cudaError_t launch_rows_w(const void *W, RowsParams &p, const RowsPlan &pl, int sms,
                                 cudaStream_t stream) {
    constexpr int kCB = rows_chunk_bytes(kFmt);
    constexpr int kHalfPitch = rows_half_pitch(kFmt);
    cudaError_t e = rows_set_attrs<kFmt, kNT, kW>();
    if (e != cudaSuccess) return e;
    p.nchunks = p.K / kGroup;
    p.ntiles = (p.N + kRowsR - 1) / kRowsR;
    p.dpp = pl.dpp;
    p.win = pl.win;
    const long cap = (long)sms * pl.occ;
    const int grid = (int)(p.ntiles < cap ? p.ntiles : cap);
    // the matrix as 8-byte elements; a box is 16 rows x 2 chunks (FP8: + 32
    // bytes; past a row's end the box is zero-filled)
    const int64_t row_bytes = kFmt == kFp8 ? (int64_t)p.K + kFp8RowPad : (int64_t)p.nchunks * kCB;
    p.W = static_cast<const uint8_t *>(W);
    p.row_bytes = row_bytes;
    CUtensorMap wmap;
    e = encode_tmap_2d(&wmap, W, CU_TENSOR_MAP_DATA_TYPE_UINT64, (uint64_t)(row_bytes / 8),
                       (uint64_t)p.N, (uint64_t)row_bytes, (uint32_t)(2 * kHalfPitch / 8), kRowsR);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(RowsWarps<kW>::kThreads, 1, 1);
    cfg.dynamicSmemBytes = (size_t)pl.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, qmm_gemv_rows_kernel<kFmt, kNT, kW>, wmap, p);
}

template <int kFmt, int kNT>
static cudaError_t launch_rows_t(const void *W, RowsParams &p, int sms, cudaStream_t stream) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const RowsPlan pl = rows_plan<kFmt, kNT>(dev, p.M, p.K);
    if (pl.dpp == 0) return cudaErrorInvalidConfiguration;  // no plan fits shared memory
    return pl.warps == 16 ? launch_rows_w<kFmt, kNT, 16>(W, p, pl, sms, stream)
                          : launch_rows_w<kFmt, kNT, 8>(W, p, pl, sms, stream);
}

cudaError_t launch_gemv_rows(int fmt, const void *W, const uint16_t *X, float *Y, int M, int N, int K,
                             int sms, cudaStream_t stream) {
    RowsParams p;
    p.Y = Y;
    p.X = X;
    p.M = M;
    p.N = N;
    p.K = K;
    if (fmt == kFp8)
        return M > 8 ? launch_rows_t<kFp8, 2>(W, p, sms, stream) : launch_rows_t<kFp8, 1>(W, p, sms, stream);
    if (fmt == 5)
        return M > 8 ? launch_rows_t<5, 2>(W, p, sms, stream) : launch_rows_t<5, 1>(W, p, sms, stream);
    if (M > 8)
        return fmt == 8 ? launch_rows_t<8, 2>(W, p, sms, stream) : launch_rows_t<4, 2>(W, p, sms, stream);
    return fmt == 8 ? launch_rows_t<8, 1>(W, p, sms, stream) : launch_rows_t<4, 1>(W, p, sms, stream);
}

}  // namespace qmm
