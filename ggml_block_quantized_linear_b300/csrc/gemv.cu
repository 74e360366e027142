// gemv.cu -- decode-shaped quantized matmul, Y[M x N] = X[M x K] * W^T,
// for M <= 16 tokens over packed Q8_0 / Q4_K weights W[N x K].
//
// The mistral.rs documentation ("Quantization types", section NVFP4) splits
// CUDA linears into a dedicated matrix-vector kernel for small decode
// batches and tiled matrix multiplication for larger ones; this is the
// small-batch kernel of that split, written for the Q8_0 / Q4_K formats.
//
// Design (HBM-bound: the packed weights are read exactly once):
//  * A CTA owns 64 weight rows and a contiguous range of K; the CTAs that
//    share a row tile form one thread-block cluster (split-K).  Their partial
//    sums are reduced through distributed shared memory in rank order, so
//    the result is deterministic and needs no workspace.
//  * One producer thread streams the CTA's 64 rows, 256 weights (272 / 144
//    bytes) per row per stage, as ONE 2-D tensor-map TMA copy per stage
//    (cp.async.bulk.tensor) into a ring of shared-memory stages guarded by
//    mbarriers.  Rows past N are zero-filled by the TMA unit.
//  * Eight consumer warps run warp-level tensor-core MMAs: warp w takes the
//    16 rows 16 * (w % 4) .. + 15 and one half of every 256-weight chunk
//    (blocks 0-3 or 4-7; Q4_K sub-blocks 0-3 or 4-7), so that twice as many
//    warps hide latency; the two halves are added in shared memory.  The
//    MMAs are m16n8k16 (f16 inputs, fp32 accumulation) with the weight rows
//    as the M side and the (padded) tokens as N.  The MMA operands are the
//    integer codes, which binary16 holds exactly: an int8 code goes through
//    one PRMT under a binary16 exponent (1152 + q) and one HSUB2 back to q;
//    a masked pair of 4-bit codes already is a pair of binary16 subnormals
//    (q * 2^-24, or q * 2^-20 for a high nibble).  The scales are applied in
//    fp32 after each 32-weight block, R being the MMA result of the block:
//    Q8_0  d * R;  Q4_K  S_j * R - Mn_j * sum_k x  (the power of two of the
//    subnormal folded into S_j), sum_k x per sub-block and token coming from
//    the staged activations.
//  * The activations of the CTA's K range are converted once to binary16
//    (round to nearest) in shared memory, each group of 4 stored in the
//    order (0, 2, 1, 3) so that one 16-byte load yields both B fragments.
#include "common.cuh"

namespace qmm {

constexpr int kGemvRowGroups = 4;                   // 16-row groups per CTA
constexpr int kGemvKHalves = 2;                     // consumer warps per row group
constexpr int kGemvWarps = kGemvRowGroups * kGemvKHalves;  // consumer warps
constexpr int kGemvRows = 16 * kGemvRowGroups;      // weight rows per CTA
constexpr int kGemvThreads = (kGemvWarps + 1) * 32; // + one producer warp
constexpr int kGemvMaxStages = 4;

struct GemvParams {
    const uint8_t *W;
    const uint16_t *X;
    float *Y;
    int M, N, K;
    int64_t row_bytes;  // packed bytes per weight row
    int nchunks;        // K / 256
    int stages;         // shared-memory ring depth
    int kr_max;         // activation window: K staged at once (multiple of 256)
};

struct GemvLayout {
    int ring, xh, xs, coef, ypart, bars, total;
};

// Byte offsets of the shared-memory regions; identical on host and device.
__host__ __device__ inline GemvLayout gemv_layout(int fmt, int nt, int M, int stages, int kr_max) {
    const int slot = fmt == 8 ? kQ8GroupBytes : kQ4Bytes;  // dense rows, as the TMA box lands
    const int mt = 8 * nt;
    GemvLayout L;
    int off = 0;
    L.ring = off;
    off += stages * kGemvRows * slot;
    L.xh = off;
    off += M * (kr_max + 32) * 2;  // only the real tokens are staged
    L.xs = off;
    off += (kr_max / 32) * mt * 4;
    L.coef = off;
    off += (fmt == 4 ? kGemvWarps * 16 * 8 * 4 : 0);
    L.ypart = off;
    off += kGemvKHalves * kGemvRows * mt * 4;
    off = (off + 15) & ~15;
    L.bars = off;
    off += 2 * stages * 8;
    L.total = off;
    return L;
}

__device__ __forceinline__ float h2f_bits(uint32_t b) {
    return __half2float(__ushort_as_half((unsigned short)(b & 0xFFFF)));
}

// 8 code bytes of a Q8_0 block at smem address p (p mod 8 == kMod8).
template <int kMod8>
__device__ __forceinline__ void load_q8_codes(const uint8_t *p, uint32_t &w0, uint32_t &w1) {
    if constexpr (kMod8 == 0) {
        const uint2 v = *reinterpret_cast<const uint2 *>(p);
        w0 = v.x;
        w1 = v.y;
    } else if constexpr (kMod8 == 4) {
        w0 = *reinterpret_cast<const uint32_t *>(p);
        w1 = *reinterpret_cast<const uint32_t *>(p + 4);
    } else {  // 2 mod 4
        const uint32_t a = *reinterpret_cast<const uint32_t *>(p - 2);
        const uint32_t b = *reinterpret_cast<const uint32_t *>(p + 2);
        const uint32_t c = *reinterpret_cast<const uint32_t *>(p + 6);
        w0 = __byte_perm(a, b, 0x5432);
        w1 = __byte_perm(b, c, 0x5432);
    }
}

// int8 codes -> binary16 (1152 + q): flip the sign bit (u = q + 128) and put
// u under a binary16 exponent of 1024.  Lanes take positions (0,2) or (1,3).
__device__ __forceinline__ uint32_t q8_pair02(uint32_t u) { return prmt(u, 0x64646464u, 0x4240u); }
__device__ __forceinline__ uint32_t q8_pair13(uint32_t u) { return prmt(u, 0x64646464u, 0x4341u); }
// (1152 + q) - 1152 = q, exact in binary16.  The MMA then multiplies the
// exact codes: no large offset enters the fp32 sums (an offset left in would
// cost ~2^-24 * 1152 * d * |sum x| of accuracy).
__device__ __forceinline__ uint32_t hsub_bits(uint32_t v, uint32_t c) {
    __half2 r = __hsub2(*reinterpret_cast<const __half2 *>(&v), *reinterpret_cast<const __half2 *>(&c));
    return *reinterpret_cast<uint32_t *>(&r);
}
__device__ __forceinline__ uint32_t q8_exact(uint32_t v) { return hsub_bits(v, 0x64806480u); }

// 16-byte B-fragment load of token row (g + 8 nt); tokens >= M are zero.
__device__ __forceinline__ uint4 x_frag(const __half *p, bool valid) {
    return valid ? *reinterpret_cast<const uint4 *>(p) : make_uint4(0u, 0u, 0u, 0u);
}

template <int kB, int kNT>
__device__ __forceinline__ void q8_block(const uint8_t *r0, const uint8_t *r1, const __half *xrow,
                                         int xstride, const float *xs, int blk, int t, int gvalid,
                                         float (&acc)[kNT][4]) {
    // code offset of this block inside the row slot: 34b + 2 + 8t
    constexpr int kOff = kQ8Bytes * kB + 2;
    constexpr int kMod8 = kOff % 8;
    const float d0 = h2f_bits(*reinterpret_cast<const uint16_t *>(r0 + kQ8Bytes * kB));
    const float d1 = h2f_bits(*reinterpret_cast<const uint16_t *>(r1 + kQ8Bytes * kB));
    uint32_t a0, a1, b0, b1;  // rows g (a*) and g+8 (b*), words 0/1
    load_q8_codes<kMod8>(r0 + kOff + 8 * t, a0, a1);
    load_q8_codes<kMod8>(r1 + kOff + 8 * t, b0, b1);
    a0 ^= 0x80808080u; a1 ^= 0x80808080u; b0 ^= 0x80808080u; b1 ^= 0x80808080u;
    const uint32_t A0[4] = {q8_exact(q8_pair02(a0)), q8_exact(q8_pair02(b0)),
                            q8_exact(q8_pair13(a0)), q8_exact(q8_pair13(b0))};
    const uint32_t A1[4] = {q8_exact(q8_pair02(a1)), q8_exact(q8_pair02(b1)),
                            q8_exact(q8_pair13(a1)), q8_exact(q8_pair13(b1))};
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt) {
        const uint4 xv = x_frag(xrow + nt * 8 * xstride + kQ8Weights * kB + 8 * t, nt * 8 < gvalid);
        float c[4] = {0.f, 0.f, 0.f, 0.f};
        mma_f16_16816(c, A0, xv.x, xv.y);
        mma_f16_16816(c, A1, xv.z, xv.w);
        acc[nt][0] = fmaf(d0, c[0], acc[nt][0]);
        acc[nt][1] = fmaf(d0, c[1], acc[nt][1]);
        acc[nt][2] = fmaf(d1, c[2], acc[nt][2]);
        acc[nt][3] = fmaf(d1, c[3], acc[nt][3]);
    }
}

template <int kNT>
__device__ __forceinline__ void q4k_half(const uint8_t *base, int rstride, const uint8_t *r0, const uint8_t *r1,
                                         const __half *xr, int xstride, const float *xs, int li,
                                         float *cw, int lane, int g, int t, int gvalid, int kh,
                                         float (&acc)[kNT][4]) {
    constexpr int kMT = 8 * kNT;
    // per-row coefficients (a_j, b_j) of this half's 4 sub-blocks; lane
    // (row = lane / 2) decodes sub-blocks 4 kh + 2 (lane & 1) + {0, 1}
    {
        const int rr = lane >> 1;
        const uint4 h = *reinterpret_cast<const uint4 *>(base + rr * rstride);
        const float dsc = h2f_bits(h.x), dmn = h2f_bits(h.x >> 16);
        auto sbyte = [&](int k) {  // scale byte k (selects, no local-memory array)
            const uint32_t w = k < 4 ? h.y : (k < 8 ? h.z : h.w);
            return (w >> (8 * (k & 3))) & 0xFFu;
        };
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) {
            const int jl = 2 * (lane & 1) + jj;  // 0..3 inside the half
            const int j = 4 * kh + jl;
            uint32_t sc, mc;
            if (j < 4) {
                sc = sbyte(j) & 63u;
                mc = sbyte(j + 4) & 63u;
            } else {
                sc = (sbyte(j + 4) & 15u) | ((sbyte(j - 4) >> 6) << 4);
                mc = (sbyte(j + 4) >> 4) | ((sbyte(j) >> 6) << 4);
            }
            // S_j * 2^24 (low nibble: sub-block even) or S_j * 2^20 (high), -Mn_j
            cw[rr * 8 + 2 * jl] = dsc * (float)sc * ((j & 1) ? 1048576.0f : 16777216.0f);
            cw[rr * 8 + 2 * jl + 1] = -(dmn * (float)mc);
        }
    }
    __syncwarp();
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
        const int c = 2 * kh + cc;  // 64-weight chunk: sub-blocks 2c (low) and 2c+1 (high)
        const uint2 qa = *reinterpret_cast<const uint2 *>(r0 + 16 + 32 * c + 8 * t);
        const uint2 qb = *reinterpret_cast<const uint2 *>(r1 + 16 + 32 * c + 8 * t);
        const float4 ca = *reinterpret_cast<const float4 *>(cw + g * 8 + 4 * cc);
        const float4 cb = *reinterpret_cast<const float4 *>(cw + (g + 8) * 8 + 4 * cc);
        const uint32_t qa0s = qa.x >> 8, qa1s = qa.y >> 8, qb0s = qb.x >> 8, qb1s = qb.y >> 8;
        // a masked nibble pair IS a pair of binary16 subnormals: q * 2^-24 (low
        // nibble) and q * 2^-20 (high nibble), exact; the MMA sums q x exactly
        // scaled, and 2^24 / 2^20 are folded into S_j
        auto lo = [&](uint32_t w) { return w & 0x000F000Fu; };
        auto hi = [&](uint32_t w) { return w & 0x00F000F0u; };
        const uint32_t L0[4] = {lo(qa.x), lo(qb.x), lo(qa0s), lo(qb0s)};
        const uint32_t L1[4] = {lo(qa.y), lo(qb.y), lo(qa1s), lo(qb1s)};
        const uint32_t H0[4] = {hi(qa.x), hi(qb.x), hi(qa0s), hi(qb0s)};
        const uint32_t H1[4] = {hi(qa.y), hi(qb.y), hi(qa1s), hi(qb1s)};
        const int blo = li * 8 + 2 * c;
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt) {
            const __half *xq = xr + nt * 8 * xstride + 64 * c + 8 * t;
            const uint4 xl = x_frag(xq, nt * 8 < gvalid);
            const uint4 xhv = x_frag(xq + 32, nt * 8 < gvalid);
            float cl[4] = {0.f, 0.f, 0.f, 0.f}, chh[4] = {0.f, 0.f, 0.f, 0.f};
            mma_f16_16816(cl, L0, xl.x, xl.y);
            mma_f16_16816(cl, L1, xl.z, xl.w);
            mma_f16_16816(chh, H0, xhv.x, xhv.y);
            mma_f16_16816(chh, H1, xhv.z, xhv.w);
            const float2 sl = *reinterpret_cast<const float2 *>(xs + blo * kMT + nt * 8 + 2 * t);
            const float2 sh = *reinterpret_cast<const float2 *>(xs + (blo + 1) * kMT + nt * 8 + 2 * t);
            // S_lo R_lo + S_hi R_hi - Mn_lo Xs_lo - Mn_hi Xs_hi (coefficients hold -Mn)
            acc[nt][0] = fmaf(ca.w, sh.x, fmaf(ca.y, sl.x, fmaf(ca.z, chh[0], fmaf(ca.x, cl[0], acc[nt][0]))));
            acc[nt][1] = fmaf(ca.w, sh.y, fmaf(ca.y, sl.y, fmaf(ca.z, chh[1], fmaf(ca.x, cl[1], acc[nt][1]))));
            acc[nt][2] = fmaf(cb.w, sh.x, fmaf(cb.y, sl.x, fmaf(cb.z, chh[2], fmaf(cb.x, cl[2], acc[nt][2]))));
            acc[nt][3] = fmaf(cb.w, sh.y, fmaf(cb.y, sl.y, fmaf(cb.z, chh[3], fmaf(cb.x, cl[3], acc[nt][3]))));
        }
    }
    __syncwarp();
}

template <int kFmt, int kNT>
__global__ void __launch_bounds__(kGemvThreads)
qmm_gemv_cluster_kernel(const __grid_constant__ CUtensorMap wmap, const GemvParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int kCB = kFmt == 8 ? kQ8GroupBytes : kQ4Bytes;  // bytes per row per chunk
    constexpr int kSlot = kCB;
    constexpr int kMT = 8 * kNT;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t nsplit = cluster_nctarank(), rank = cluster_ctarank();
    const int row0 = blockIdx.x * kGemvRows;
    const int c_begin = (int)((int64_t)p.nchunks * rank / nsplit);
    const int c_end = (int)((int64_t)p.nchunks * (rank + 1) / nsplit);
    const int nloc = c_end - c_begin;
    const int kbase = c_begin * kGroup;
    const int xstride = p.kr_max + 32;
    const GemvLayout L = gemv_layout(kFmt, kNT, p.M, p.stages, p.kr_max);
    uint8_t *ring = smem + L.ring;
    __half *xh = reinterpret_cast<__half *>(smem + L.xh);
    float *xs = reinterpret_cast<float *>(smem + L.xs);
    float *coef = reinterpret_cast<float *>(smem + L.coef);
    float *ypart = reinterpret_cast<float *>(smem + L.ypart);
    const uint32_t bar0 = smem_addr(smem + L.bars);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (p.stages + s); };

    if (tid == 0) {
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), kGemvWarps);
        }
        fence_mbar_init();
    }
    // block sums of padding tokens (m >= M) stay zero for the whole kernel
    for (int idx = tid; idx < (p.kr_max / 32) * kMT; idx += kGemvThreads) xs[idx] = 0.f;
    if (warp == kGemvWarps && lane == 0) {
        // descriptor fetch and an L2 prefetch of the first weight stages:
        // safe before the dependency wait below (L2 stays coherent with the
        // previous kernel's writes; nothing lands in shared memory yet)
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&wmap)) : "memory");
        for (int i = 0; i < nloc && i < 2 * p.stages; ++i)
            tma_prefetch_l2_2d(&wmap, (c_begin + i) * (kCB / 2), row0);
        // and of this CTA's first activation window
        const int wk = min(p.kr_max, nloc * kGroup);
        for (int m = 0; m < p.M; ++m) bulk_prefetch_l2(p.X + (int64_t)m * p.K + kbase, (uint32_t)(wk * 2));
    }
    __syncthreads();
    // Programmatic dependent launch: everything above overlaps the tail of
    // the previous kernel in the stream; no shared-memory copy, activation
    // read or output write happens before that kernel has completed and
    // flushed.  The next kernel may start its own prologue now.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (warp == kGemvWarps) {
        // ---------------- producer: one 2-D TMA copy of the row tile per chunk
        for (int i = 0; i < nloc; ++i) {
            const int s = i % p.stages;
            if (i >= p.stages &&
                !mbar_wait_warp(empty_bar(s), ((i / p.stages) - 1) & 1, kErrGemvEmptyWait))
                break;  // bug path: consumers then time out on their full barriers
            if (lane == 0) {
                mbar_arrive_expect_tx(full_bar(s), (uint32_t)(kGemvRows * kCB));
                tma_load_2d(smem_addr(ring + s * kGemvRows * kSlot), &wmap,
                            (c_begin + i) * (kCB / 2), row0, full_bar(s));
            }
            __syncwarp();
        }
    } else {
        // ---------------- consumers
        const int g = lane >> 2, t = lane & 3;
        float acc[kNT][4];
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt)
            acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
        const __half *xrow = xh + g * xstride;  // token g (+ 8 nt); read only if < M
        const int gvalid = p.M - g;             // token g + 8 nt is real iff 8 nt < gvalid
        const int rgrp = warp % kGemvRowGroups, kh = warp / kGemvRowGroups;
        float *cw = coef + warp * 16 * 8;
        const int win = p.kr_max / kGroup;  // chunks per activation window
        // `ok` is warp-uniform; after a timed-out wait the warp skips its
        // remaining waits and MMAs but still takes every named barrier.
        bool ok = true;
        for (int w0 = 0; w0 < nloc; w0 += win) {
            const int wn = min(win, nloc - w0);
            if (w0 > 0) named_bar_sync(1, kGemvWarps * 32);  // previous window fully read
            // stage the window's activations as binary16 (+ 32-weight block sums)
            const int ngr = (wn * kGroup) / 8;  // 8-element groups per token
            const int kw = kbase + w0 * kGroup;
            for (int idx = tid; idx < p.M * ngr; idx += kGemvWarps * 32) {
                const int m = idx / ngr, kg = idx - m * ngr;
                const uint4 v =
                    __ldg(reinterpret_cast<const uint4 *>(p.X + (int64_t)m * p.K + kw + 8 * kg));
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
                *reinterpret_cast<uint4 *>(xh + m * xstride + 8 * kg) = o;
                const float2 s02 = __half22float2(h02), s13 = __half22float2(h13);
                const float2 s46 = __half22float2(h46), s57 = __half22float2(h57);
                float sum = ((s02.x + s13.x) + (s02.y + s13.y)) + ((s46.x + s57.x) + (s46.y + s57.y));
                sum += __shfl_xor_sync(0xffffffffu, sum, 1);
                sum += __shfl_xor_sync(0xffffffffu, sum, 2);
                if ((kg & 3) == 0) xs[(kg >> 2) * kMT + m] = sum;
            }
            named_bar_sync(1, kGemvWarps * 32);

            // main loop over the window's K chunks
            for (int li = 0; li < wn; ++li) {
                const int i = w0 + li;
                const int s = i % p.stages;
                if (ok) ok = mbar_wait_warp(full_bar(s), (i / p.stages) & 1, kErrGemvFullWait);
                if (!ok) continue;
                const uint8_t *base = ring + (s * kGemvRows + 16 * rgrp) * kSlot;
                const uint8_t *r0 = base + g * kSlot;
                const uint8_t *r1 = base + (g + 8) * kSlot;
                const __half *xr = xrow + li * kGroup;
                if constexpr (kFmt == 8) {
                    if (kh == 0) {
                        q8_block<0, kNT>(r0, r1, xr, xstride, xs, li * 8 + 0, t, gvalid, acc);
                        q8_block<1, kNT>(r0, r1, xr, xstride, xs, li * 8 + 1, t, gvalid, acc);
                        q8_block<2, kNT>(r0, r1, xr, xstride, xs, li * 8 + 2, t, gvalid, acc);
                        q8_block<3, kNT>(r0, r1, xr, xstride, xs, li * 8 + 3, t, gvalid, acc);
                    } else {
                        q8_block<4, kNT>(r0, r1, xr, xstride, xs, li * 8 + 4, t, gvalid, acc);
                        q8_block<5, kNT>(r0, r1, xr, xstride, xs, li * 8 + 5, t, gvalid, acc);
                        q8_block<6, kNT>(r0, r1, xr, xstride, xs, li * 8 + 6, t, gvalid, acc);
                        q8_block<7, kNT>(r0, r1, xr, xstride, xs, li * 8 + 7, t, gvalid, acc);
                    }
                } else {
                    q4k_half<kNT>(base, kSlot, r0, r1, xr, xstride, xs, li, cw, lane, g, t, gvalid, kh, acc);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(empty_bar(s));
            }
        }
        // partial sums of this CTA and K half: ypart[kh][row][token]
        const int rg = 16 * rgrp + g;
        float *yp = ypart + kh * kGemvRows * kMT;
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt) {
            *reinterpret_cast<float2 *>(yp + rg * kMT + nt * 8 + 2 * t) = make_float2(acc[nt][0], acc[nt][1]);
            *reinterpret_cast<float2 *>(yp + (rg + 8) * kMT + nt * 8 + 2 * t) =
                make_float2(acc[nt][2], acc[nt][3]);
        }
    }

    // ---------------- split-K reduction across the cluster, in rank order
    cluster_sync_all();
    const int rpr = kGemvRows / (int)nsplit;
    for (int idx = tid; idx < rpr * kMT; idx += kGemvThreads) {
        const int r = (int)rank * rpr + idx / kMT, m = idx % kMT;
        if (m < p.M && row0 + r < p.N) {
            const uint32_t a0 = smem_addr(ypart + r * kMT + m);
            const uint32_t a1 = smem_addr(ypart + (kGemvRows + r) * kMT + m);
            float sum = 0.f;
            for (uint32_t q = 0; q < nsplit; ++q)
                sum += ld_dsmem_f32(map_to_rank(a0, q)) + ld_dsmem_f32(map_to_rank(a1, q));
            p.Y[(int64_t)m * p.N + row0 + r] = sum;
        }
    }
    cluster_sync_all();
}

// ------------------------------------------------------------- launcher
// Activation window (in 256-weight chunks) staged in shared memory at once,
// and ring depth, per format / token tile.
#ifndef QMM_GEMV_STAGES_Q8
#define QMM_GEMV_STAGES_Q8 3
#endif
#ifndef QMM_GEMV_STAGES_Q4
#define QMM_GEMV_STAGES_Q4 4
#endif
#ifndef QMM_GEMV_WAVE_PCT  // grid size allowed, in % of one wave of resident CTAs
#define QMM_GEMV_WAVE_PCT 100
#endif
#ifndef QMM_GEMV_PDL
#define QMM_GEMV_PDL 1
#endif
#ifndef QMM_GEMV_WINDOW_NT2  // activation window in chunks with 9..16 tokens
#define QMM_GEMV_WINDOW_NT2 4
#endif
static int gemv_window(int nt) { return nt == 1 ? 8 : QMM_GEMV_WINDOW_NT2; }
static int gemv_stages(int fmt) { return fmt == 8 ? QMM_GEMV_STAGES_Q8 : QMM_GEMV_STAGES_Q4; }

struct GemvPlan {
    int nsplit, stages, kr_max, smem;
};

// Split-K factor (cluster size along K) and shared-memory plan: the largest
// power of two <= 8 that keeps every CTA on at least two chunks and the grid
// within one wave of resident CTAs.
static GemvPlan gemv_plan(int fmt, int M, int N, int K, int sms) {
    const int nt = M <= 8 ? 1 : 2;
    const int tiles = (N + kGemvRows - 1) / kGemvRows;
    const int nchunks = K / kGroup;
    GemvPlan best = {0, 0, 0, 0};
    for (int s = 1; s <= 8; s *= 2) {
        if (s > 1 && nchunks < 2 * s) break;
        const int per = (nchunks + s - 1) / s;
        GemvPlan pl;
        pl.nsplit = s;
        pl.stages = per < gemv_stages(fmt) ? per : gemv_stages(fmt);
        pl.kr_max = (per < gemv_window(nt) ? per : gemv_window(nt)) * kGroup;
        pl.smem = gemv_layout(fmt, nt, M, pl.stages, pl.kr_max).total;
        const int by_smem = (228 * 1024) / (pl.smem + 1024);
        const int by_warps = 64 / (kGemvThreads / 32);
        const int per_sm = by_smem < by_warps ? by_smem : by_warps;
        if (s == 1 || tiles * s * 100 <= sms * per_sm * QMM_GEMV_WAVE_PCT) best = pl;
        else break;
    }
    return best;
}

template <int kFmt, int kNT>
static cudaError_t launch_gemv_t(const GemvParams &p, const GemvPlan &pl, cudaStream_t stream) {
    // packed weights viewed as uint16 [N][row_bytes / 2]; box = 64 rows x one
    // 256-weight group
    constexpr int kCB = kFmt == 8 ? kQ8GroupBytes : kQ4Bytes;
    CUtensorMap wmap;
    cudaError_t te = encode_tmap_2d(&wmap, p.W, CU_TENSOR_MAP_DATA_TYPE_UINT16,
                                    (uint64_t)(p.row_bytes / 2), (uint64_t)p.N,
                                    (uint64_t)p.row_bytes, kCB / 2, kGemvRows);
    if (te != cudaSuccess) return te;
    static std::atomic<uint64_t> attr_done{0};
    cudaError_t e = set_smem_limit_once(reinterpret_cast<const void *>(qmm_gemv_cluster_kernel<kFmt, kNT>), 227 * 1024,
                                        attr_done);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((p.N + kGemvRows - 1) / kGemvRows), (unsigned)pl.nsplit, 1);
    cfg.blockDim = dim3(kGemvThreads, 1, 1);
    cfg.dynamicSmemBytes = (size_t)pl.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = (unsigned)pl.nsplit;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = QMM_GEMV_PDL;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, qmm_gemv_cluster_kernel<kFmt, kNT>, wmap, p);
}

cudaError_t launch_gemv(int fmt, const void *W, const uint16_t *X, float *Y, int M, int N, int K,
                        int sms, cudaStream_t stream) {
    GemvParams p;
    p.W = static_cast<const uint8_t *>(W);
    p.X = X;
    p.Y = Y;
    p.M = M;
    p.N = N;
    p.K = K;
    p.nchunks = K / kGroup;
    p.row_bytes = (int64_t)p.nchunks * (fmt == 8 ? kQ8GroupBytes : kQ4Bytes);
    const GemvPlan pl = gemv_plan(fmt, M, N, K, sms);
    p.stages = pl.stages;
    p.kr_max = pl.kr_max;
    if (fmt == 8)
        return M <= 8 ? launch_gemv_t<8, 1>(p, pl, stream) : launch_gemv_t<8, 2>(p, pl, stream);
    return M <= 8 ? launch_gemv_t<4, 1>(p, pl, stream) : launch_gemv_t<4, 2>(p, pl, stream);
}

}  // namespace qmm
