// gemm.cu -- prefill-shaped quantized matmul (M > 16 tokens) on the 5th-
// generation tensor cores: Y[M x N] = X[M x K] * W^T, W packed Q8_0, Q4_K,
// Q5_K or FP8 E4M3 with row scales.
//
// The mistral.rs documentation ("Quantization types") sends larger dense
// batches to tiled matrix multiplication (section NVFP4) and describes FP8
// W8A16 GEMMs that convert each weight tile to BF16 / F16 inside the GEMM
// (section FP8).  This kernel does the same for the GGML block formats: the
// packed weight tile is dequantized in registers into tensor memory and fed
// to tcgen05.mma.
//
// Operand precision.  The dequantized weights are rounded to binary16 (not
// bf16): the relative error 2^-11 per weight keeps every output inside
// 1e-3 * sum|w x| even for a one-hot activation row, which bf16's 2^-9 does
// not.  tcgen05 kind::f16 needs both operands in one type, so the bf16
// activations are converted to binary16 once per call (first kernel below)
// into the caller's workspace.  The GEMM follows that launch by programmatic
// dependent launch: its prologue and weight stages overlap the conversion,
// and the roles that read X or write Y, tickets or partial tiles wait for it.
//
// Tile: 128 weight rows (the MMA's M side, "swap AB") x BN tokens (MMA N:
// 32, 64, 128 or 256, the smallest that holds M up to 128; above that 256)
// x 128 K per stage (two 64-wide 128B-swizzled activation boxes); persistent
// CTAs (one per SM) walk the work units.  The dequantized weights go to
// tensor memory, not shared memory: each dequantizing thread owns one weight
// row (one TMEM lane) and a 32-wide slice of the stage's K, converts its 32
// weights in registers and writes them with tcgen05.st; the MMA reads A from
// TMEM and only the activations from shared memory (tcgen05.mma with A in
// TMEM).  That keeps the A stores, their bank conflicts and the MMA's A
// reads off the shared-memory port.  One full barrier per stage counts the
// activation bytes and the 16 dequantizing warps; one MMA commit frees it.
// TMEM holds the A stages (64 columns each) and the fp32 accumulators: two
// of BN columns alternating between units for BN up to 128 (three stages),
// one of 256 columns for 256-token tiles (two stages), which the
// dequantizing warps drain themselves where they would otherwise wait for
// the unit's last MMA.
// 256-token tiles, four waves or more (stream-K): the (tile,
// packed group) pairs, token tile fastest, are cut into one contiguous run
// per CTA, so every CTA has the same K work and the last wave is not left
// part-empty.  A run is at least one tile long, so a tile falls to at most
// two CTAs; both add their parts onto a Y tile that the conversion launch
// zeroed.  With fewer output tiles than SMs, K is split into parts (a unit is
// one part of one tile).  256-token tiles: at most two parts, both added onto
// a Y zeroed by the conversion launch.  (Two additions onto zero commute, so
// neither result depends on the order of the parts.)  Smaller tiles: up to
// 8 parts, one unit per CTA; each part stores its partial tile in the
// workspace and takes a ticket, and in the CTA whose part arrives last every
// warp, once its role has ended, helps add all parts in part order into Y.
// All are deterministic and nothing ever waits for another CTA.
//   warp 0       TMA producer of the binary16 activation tiles (128B-swizzled
//                boxes)
//   warp 1       TMEM allocator and single-thread MMA issuer
//   warps 2-17   dequantize packed weights into the TMEM A stages (warp w
//                writes TMEM lanes 32 (w mod 4) .. + 31, K slice (w - 2) / 4);
//                with one 256-column accumulator they also drain it
//   warps 18-21  epilogue: read an accumulator back (tcgen05.ld) and store Y
//                (two accumulators)
//   warp 22      TMA producer of the packed weights (separate from warp 0 so
//                that the dequantizing warps never wait behind activation
//                stages)
// Every wait is bounded (common.cuh); TMEM is always released.
#include <type_traits>

#include "common.cuh"

namespace qmm {

#ifndef QMM_GEMM_MAX_PARTS  // K parts per tile for token tiles below 256
#define QMM_GEMM_MAX_PARTS 8
#endif
constexpr int kGemmBM = 128;        // weight rows per CTA (MMA M)
constexpr int kGemmBK = 128;        // K per stage: two 128-byte swizzle atoms of f16
constexpr int kGemmAtomK = 64;      // K of one 128B-swizzled atom (one TMA box, one descriptor base)
#ifndef QMM_GEMM_DEQ_WARPS
#define QMM_GEMM_DEQ_WARPS 16
#endif
constexpr int kGemmDeqWarps = QMM_GEMM_DEQ_WARPS;  // 8 or 16 (128 rows / (4 rows x warps) passes)
constexpr int kGemmEpiWarps = 4;
// warps: 0 activation producer, 1 MMA, then the dequantizing warps, the
// epilogue warps and the packed-weight producer
constexpr int kGemmWarpPackedTma = 2 + kGemmDeqWarps + kGemmEpiWarps;
constexpr int kGemmThreads = (kGemmWarpPackedTma + 1) * 32;
constexpr int kGemmStagesP = 2;     // packed weight groups
constexpr int kGemmACols = kGemmBK / 2;  // TMEM columns of one A stage (two binary16 per column)
constexpr int kGemmStepsPerGroup = kGroup / kGemmBK;  // K steps per packed 256-weight group
static_assert(kGemmDeqWarps == 16, "four warps per TMEM lane quarter, one per 32-wide K slice of a stage");
// accumulators: two of BN columns (BN <= 128) or one of 256
__host__ __device__ constexpr int gemm_nbuf(int bn) { return bn == 256 ? 1 : 2; }
// K-step stages: an activation stage (BN x 256 bytes of shared memory) and
// a TMEM A stage (64 columns) each, filled and released together; two for
// 256-token tiles (shared memory and TMEM bound it), three below
__host__ __device__ constexpr int gemm_stages(int bn) { return bn == 256 ? 2 : 3; }
// TMEM columns allocated: accumulators then A stages, rounded up to a power of two
__host__ __device__ constexpr int gemm_tmem_cols(int fmt, int bn) {
    return gemm_nbuf(bn) * bn + gemm_stages(bn) * kGemmACols <= 32    ? 32
           : gemm_nbuf(bn) * bn + gemm_stages(bn) * kGemmACols <= 64  ? 64
           : gemm_nbuf(bn) * bn + gemm_stages(bn) * kGemmACols <= 128 ? 128
           : gemm_nbuf(bn) * bn + gemm_stages(bn) * kGemmACols <= 256 ? 256
                                                                          : 512;
}
static_assert(2 * 128 + 3 * 64 <= 512 && 256 + 2 * 64 <= 512, "accumulators and A stages fit TMEM");
// Shared-memory pitch of a packed weight row in a stage (FP8: a 256-byte group
// plus 16 bytes of the next, which keeps the dequantizing warps' loads on
// distinct banks as Q8_0's 272 bytes do), and a group's advance in a row.
// (Q5_K: 176 bytes, 44 words: the 8 rows of a quarter-warp's 16-byte loads
// land on distinct banks.)
constexpr int kGemmQ5Bytes = 176;
__host__ __device__ constexpr int gemm_group_bytes(int fmt) {
    return fmt == 4 ? kQ4Bytes : fmt == 5 ? kGemmQ5Bytes : kQ8GroupBytes;
}
__host__ __device__ constexpr int gemm_group_advance(int fmt) {
    return fmt == 8 ? kQ8GroupBytes : fmt == 4 ? kQ4Bytes : fmt == 5 ? kGemmQ5Bytes : 256;
}

struct GemmLayout {
    int b, p, bars, total;  // offsets from the 1024-aligned base
};

__host__ __device__ inline GemmLayout gemm_layout(int fmt, int bn) {
    GemmLayout L;
    int off = 0;
    L.b = off;
    off += gemm_stages(bn) * bn * kGemmBK * 2;
    L.p = off;
    off += kGemmStagesP * kGemmBM * gemm_group_bytes(fmt);
    off = (off + 15) & ~15;
    L.bars = off;
    off += 64 * 8;  // barriers, TMEM address slot, last-part flag
    L.total = off + 1024;  // + alignment slack of the dynamic base
    return L;
}

// ------------------------------------------------------------ tcgen05 / UMMA
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[smem] * B[smem]^T, both K-major, kind::f16.
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem]^T, kind::f16: A's 128 rows are the TMEM
// lanes, two binary16 K values per 32-bit column (16 K = 8 columns).
__device__ __forceinline__ void umma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// 8 consecutive 32-bit columns of this thread's TMEM lane, and the wait
// for this thread's TMEM stores.
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&v)[8]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(v[0]),
                 "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
                 : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
            taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
        "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
        : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
// Arrive (once) on an mbarrier when all previously issued tcgen05 ops of
// this thread have completed.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}
// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle,
// 8-row core groups 1024 bytes apart (SBO), sm_100 descriptor version 1.
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t smem_addr) {
    uint64_t d = 0;
    d |= (uint64_t)((smem_addr >> 4) & 0x3FFFu);  // start address
    d |= (uint64_t)1u << 16;                      // leading byte offset (unused with SW128)
    d |= (uint64_t)(1024u >> 4) << 32;            // stride byte offset
    d |= (uint64_t)1u << 46;                      // descriptor version
    d |= (uint64_t)2u << 61;                      // SWIZZLE_128B
    return d;
}
// Instruction descriptor of kind::f16: A = B = f16, D = f32, both K-major.
__host__ __device__ constexpr uint32_t umma_idesc_f16(int m, int n) {
    return (1u << 4)                       // D format f32
           | (0u << 7) | (0u << 10)        // A, B format f16
           | ((uint32_t)(n >> 3) << 17)    // N / 8
           | ((uint32_t)(m >> 4) << 24);   // M / 16
}
// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
          "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
          "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]),
          "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]),
          "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
// Wait for the conversion launch (programmatic dependent launch): its
// activations, zeroed Y tiles and cleared tickets are visible afterwards.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ----------------------------------------------------- activation conversion
// Stream-K tiles shared by two CTAs: the tile holding pair c G / ctas for
// each CTA boundary c = 1 .. ctas - 1 that falls inside a tile (tile t =
// weight tile * tiles_m + token tile, BN tokens x 128 weight rows).
struct SplitTiles {
    int ctas;        // 0: none
    int gtot, tiles_m, bn, M, N;
    int64_t gall;    // (tile, group) pairs
};

// X bf16 -> binary16 (round to nearest), 8 elements per thread.  With a K
// split, the same launch also clears the tiles' tickets (nt words) or zeroes
// Y (ny floats) for the parts to add onto; with stream-K it zeroes the Y
// tiles that two CTAs share.
__global__ void __launch_bounds__(256) qmm_x_to_f16_kernel(const uint16_t *__restrict__ X,
                                                           __half *__restrict__ Xh, int64_t n8,
                                                           int *__restrict__ tickets, int nt,
                                                           float *__restrict__ Yz, int64_t ny,
                                                           const SplitTiles st) {
    // the GEMM behind this launch may start its prologue and weight stages now
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    for (int i = blockIdx.x * 256 + threadIdx.x; i < nt; i += gridDim.x * 256) tickets[i] = 0;
    const int64_t y4 = ny / 4;  // Y is 16-byte aligned
    for (int64_t i = (int64_t)blockIdx.x * 256 + threadIdx.x; i < y4; i += (int64_t)gridDim.x * 256)
        reinterpret_cast<float4 *>(Yz)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (blockIdx.x == 0 && threadIdx.x < ny - 4 * y4) Yz[4 * y4 + threadIdx.x] = 0.f;
    // one boundary per block: its tile, then 128 consecutive n per token row
    for (int c = 1 + (int)blockIdx.x; c < st.ctas; c += (int)gridDim.x) {
        const int64_t b = st.gall * c / st.ctas;
        if (b % st.gtot == 0) continue;  // the boundary falls between tiles
        const int t = (int)(b / st.gtot);
        const int m0 = (t % st.tiles_m) * st.bn, n0 = (t / st.tiles_m) * 128;
        const int rows = min(st.bn, st.M - m0);
        if ((st.N & 3) == 0) {  // whole float4s (n0 is a multiple of 128)
            const int c4 = min(32, (st.N - n0) / 4);
            for (int e = threadIdx.x; e < rows * 32; e += 256)
                if ((e & 31) < c4)
                    reinterpret_cast<float4 *>(Yz + (int64_t)(m0 + (e >> 5)) * st.N + n0)[e & 31] =
                        make_float4(0.f, 0.f, 0.f, 0.f);
        } else {
            const int cn = min(128, st.N - n0);
            for (int e = threadIdx.x; e < rows * 128; e += 256)
                if ((e & 127) < cn) Yz[(int64_t)(m0 + (e >> 7)) * st.N + n0 + (e & 127)] = 0.f;
        }
    }
    for (int64_t i = (int64_t)blockIdx.x * 256 + threadIdx.x; i < n8; i += (int64_t)gridDim.x * 256) {
        const uint4 v = __ldg(reinterpret_cast<const uint4 *>(X) + i);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t o[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const __half2 h = __floats2half2_rn(__uint_as_float(w[e] << 16),
                                                __uint_as_float(w[e] & 0xFFFF0000u));
            o[e] = *reinterpret_cast<const uint32_t *>(&h);
        }
        reinterpret_cast<uint4 *>(Xh)[i] = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

// --------------------------------------------------------- dequantization
// Each function turns 16 weights of one packed row (the row's K slice
// 16 kq .. 16 kq + 15 of 64-wide K step kJ of a 256-weight group) into 8
// binary16 pairs, lower K in the low half.

// Q8_0: the slice is half of block 2 kJ + kq / 2; its 16 code bytes start 2
// bytes into the block (+16 for the second half), read as two aligned
// 16-byte words and shifted into place; d * q is rounded once.
template <int kJ, int kHi>
__device__ __forceinline__ void deq16_q8_0(const uint8_t *prow, int h, uint32_t (&r)[8]) {
    constexpr int kB = 2 * kJ + kHi;            // block inside the group
    constexpr int kOff = kQ8Bytes * kB + 2;     // first code byte of the block
    constexpr int kS = kOff & 15, kBase = kOff & ~15;
    // (the last block's codes end the 272-byte row: one aligned word, kS = 0)
    const uint4 *w = reinterpret_cast<const uint4 *>(prow + kBase + 16 * h);
    const uint4 a = w[0], b = kS != 0 ? w[1] : make_uint4(0u, 0u, 0u, 0u);
    const uint32_t v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    uint32_t c[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        c[i] = (kS & 3) ? __funnelshift_r(v[kS / 4 + i], v[kS / 4 + i + 1], 16) : v[kS / 4 + i];
    const __half d = __ushort_as_half(*reinterpret_cast<const uint16_t *>(prow + kQ8Bytes * kB));
    const __half2 d2 = __halves2half2(d, d);
    const __half2 bias = __floats2half2_rn(1152.0f, 1152.0f);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t u = c[i] ^ 0x80808080u;
        uint32_t lo = prmt(u, 0x64646464u, 0x4140u), hi = prmt(u, 0x64646464u, 0x4342u);
        __half2 hl = __hmul2(__hsub2(*reinterpret_cast<__half2 *>(&lo), bias), d2);  // q exact, then d * q
        __half2 hh = __hmul2(__hsub2(*reinterpret_cast<__half2 *>(&hi), bias), d2);
        r[2 * i] = *reinterpret_cast<uint32_t *>(&hl);
        r[2 * i + 1] = *reinterpret_cast<uint32_t *>(&hh);
    }
}

// Q4_K: the slice is weights 16 (kq % 2) .. + 15 of sub-block 2 kJ + kq / 2,
// i.e. one nibble of 16 consecutive code bytes; S q - Mn with one rounding
// in fp32 (two weights per packed instruction), then binary16.
__device__ __forceinline__ void deq16_q4_k(const uint8_t *prow, int j, int kq, float S, float Mn,
                                           uint32_t (&r)[8]) {
    const uint4 q = *reinterpret_cast<const uint4 *>(prow + 16 + 32 * j + 16 * (kq & 1));
    const int sh = (kq >> 1) * 4;
    const uint32_t n[4] = {(q.x >> sh) & 0x0F0F0F0Fu, (q.y >> sh) & 0x0F0F0F0Fu, (q.z >> sh) & 0x0F0F0F0Fu,
                           (q.w >> sh) & 0x0F0F0F0Fu};
    const uint64_t s2 = f2_pack(S, S), nm2 = f2_pack(-Mn, -Mn);
    const uint64_t k2 = f2_pack(-8388608.0f, -8388608.0f);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const uint32_t nw = n[e >> 1];
        const int b0 = (2 * e) & 3;
        const uint64_t qq = f2_add(f2_pack(__uint_as_float(prmt(nw, 0x4B000000u, 0x7440u + b0)),
                                           __uint_as_float(prmt(nw, 0x4B000000u, 0x7440u + b0 + 1))),
                                   k2);
        float v0, v1;
        f2_unpack(f2_fma(s2, qq, nm2), v0, v1);
        const __half2 hv = __floats2half2_rn(v0, v1);
        r[e] = *reinterpret_cast<const uint32_t *>(&hv);
    }
}

// Q5_K: Q4_K's slice with the fifth code bits: the codes sit at byte 48 of
// the superblock, and bit sb (the sub-block) of qh byte l (16 + l) is bit 4
// of weight l.
__device__ __forceinline__ void deq16_q5_k(const uint8_t *prow, int j, int kq, float S, float Mn,
                                           uint32_t (&r)[8]) {
    const uint4 q = *reinterpret_cast<const uint4 *>(prow + 48 + 32 * j + 16 * (kq & 1));
    const uint4 h = *reinterpret_cast<const uint4 *>(prow + 16 + 16 * (kq & 1));
    const int sh = (kq >> 1) * 4, sb = 2 * j + (kq >> 1);
    const uint32_t n[4] = {((q.x >> sh) & 0x0F0F0F0Fu) | (((h.x >> sb) & 0x01010101u) << 4),
                           ((q.y >> sh) & 0x0F0F0F0Fu) | (((h.y >> sb) & 0x01010101u) << 4),
                           ((q.z >> sh) & 0x0F0F0F0Fu) | (((h.z >> sb) & 0x01010101u) << 4),
                           ((q.w >> sh) & 0x0F0F0F0Fu) | (((h.w >> sb) & 0x01010101u) << 4)};
    const uint64_t s2 = f2_pack(S, S), nm2 = f2_pack(-Mn, -Mn);
    const uint64_t k2 = f2_pack(-8388608.0f, -8388608.0f);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const uint32_t nw = n[e >> 1];
        const int b0 = (2 * e) & 3;
        const uint64_t qq = f2_add(f2_pack(__uint_as_float(prmt(nw, 0x4B000000u, 0x7440u + b0)),
                                           __uint_as_float(prmt(nw, 0x4B000000u, 0x7440u + b0 + 1))),
                                   k2);
        float v0, v1;
        f2_unpack(f2_fma(s2, qq, nm2), v0, v1);
        const __half2 hv = __floats2half2_rn(v0, v1);
        r[e] = *reinterpret_cast<const uint32_t *>(&hv);
    }
}

// FP8: 16 codes converted exactly to binary16; the row scale is applied to
// the finished sums.
__device__ __forceinline__ void deq16_fp8(const uint8_t *prow, int j, int kq, uint32_t (&r)[8]) {
    const uint4 q = *reinterpret_cast<const uint4 *>(prow + 64 * j + 16 * kq);
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        r[2 * i] = e4m3x2_to_h2(w[i]);
        r[2 * i + 1] = e4m3x2_to_h2(w[i] >> 16);
    }
}

// Q4_K (S_j, Mn_j) of sub-block sj from the row's superblock header (d,
// dmin, 12 scale bytes as the words h.y, h.z, h.w): exact fp32 products.
__device__ __forceinline__ void q4k_coef(const uint4 &h, int sj, float &S, float &Mn) {
    const float dsc = __half2float(__ushort_as_half((unsigned short)(h.x & 0xFFFF)));
    const float dmn = __half2float(__ushort_as_half((unsigned short)(h.x >> 16)));
    const uint32_t sw[3] = {h.y, h.z, h.w};
    auto sb = [&](int k) { return (sw[k >> 2] >> (8 * (k & 3))) & 0xFFu; };
    uint32_t sc, mc;
    if (sj < 4) {
        sc = sb(sj) & 63u;
        mc = sb(sj + 4) & 63u;
    } else {
        sc = (sb(sj + 4) & 15u) | ((sb(sj - 4) >> 6) << 4);
        mc = (sb(sj + 4) >> 4) | ((sb(sj) >> 6) << 4);
    }
    S = dsc * (float)sc;
    Mn = dmn * (float)mc;
}

// ------------------------------------------------------------------ kernel
struct GemmParams {
    float *Y;
    const uint8_t *W;   // FP8: the packed rows, for the row scales
    int64_t row_bytes;  // packed bytes per row
    float *partials;  // ticket mode: [tile][part][128 rows][BN columns] fp32
    int *tickets;     // ticket mode: parts of each tile done so far (cleared by the conversion launch)
    int M, N, K;
    int ksplit;       // K parts per output tile
    int tickets_mode; // 1: partial tiles + tickets; 0: (ksplit 2) add onto a zeroed Y
};

// Persistent: CTA b computes the output tiles b, b + gridDim.x, ... (weight
// tile index fastest).  Every ring index (packed groups, activation stages,
// A stages) runs on across tiles, and the two TMEM accumulators alternate
// between tiles, so the epilogue of one tile overlaps the main loop of the
// next.
template <int kFmt, int kBN, bool kSK>
__global__ void __launch_bounds__(kGemmThreads, 1)
qmm_gemm_kernel(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap wmap,
                const GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    constexpr int kSA = gemm_stages(kBN);
    constexpr int kCB = gemm_group_bytes(kFmt);
    constexpr int kNbuf = gemm_nbuf(kBN);                    // TMEM accumulators
    constexpr uint32_t kBBytes = kBN * kGemmBK * 2;          // one activation stage
    constexpr int kTmemCols = gemm_tmem_cols(kFmt, kBN);
    constexpr uint32_t kBAtom = kBN * 128;                   // one 64-K atom of an activation stage
    constexpr int kACol0 = kNbuf * kBN;                      // first TMEM column of the A stages
    constexpr uint32_t kPBytes = kGemmBM * kCB;
    const GemmLayout L = gemm_layout(kFmt, kBN);
    // 1024-byte aligned base for the 128B-swizzled stages, kept as an offset
    // into the shared array so that every access compiles to LDS / STS
    // (an address rounded through an integer would be a generic pointer)
    uint8_t *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // work unit u = ((token tile * tiles_n + weight tile) * ksplit + K part);
    // CTA b takes units b, b + gridDim.x, ...  Consecutive CTAs run
    // neighbouring weight tiles against the same token tile, so an
    // activation tile is read from DRAM about once and then from L2.
    // Stream-K: tile t = weight tile * tiles_m + token tile, and CTA b takes
    // the pairs [b G / gridDim.x, (b + 1) G / gridDim.x) of the G = tiles x
    // groups (tile, group) pairs, i.e. a few consecutive tiles, mostly one
    // weight tile against consecutive token tiles (the weight tile is then
    // often still in L2; X, a few MB to tens of MB, mostly stays there).
    const int cid = (int)blockIdx.x, nctas = (int)gridDim.x;
    const int tiles_n = (p.N + kGemmBM - 1) / kGemmBM, tiles_m = (p.M + kBN - 1) / kBN;
    const int ksplit = p.ksplit;
    const int gtot = p.K / kGroup;
    const int units = tiles_n * tiles_m * ksplit;
    static_assert(!kSK || kBN == 256, "stream-K runs 256-token tiles");
    constexpr bool sk = kSK;
    // stream-K run [s0, s1): tiles t_first .. t_first + my_tiles - 1, from
    // group g_first of the first to group g_end of the last (exclusive)
    int t_first = 0, g_first = 0, g_end = gtot, my_tiles;
    if (sk) {
        const int64_t gall = (int64_t)tiles_n * tiles_m * gtot;
        const int64_t s0 = gall * cid / nctas, s1 = gall * (cid + 1) / nctas;
        t_first = (int)(s0 / gtot);
        const int t_last = (int)((s1 - 1) / gtot);
        my_tiles = s1 > s0 ? t_last - t_first + 1 : 0;
        g_first = (int)(s0 - (int64_t)t_first * gtot);
        g_end = (int)(s1 - (int64_t)t_last * gtot);
    } else {
        my_tiles = units > cid ? (units - 1 - cid) / nctas + 1 : 0;
    }
    auto tile_base = [&](int lt) { return sk ? t_first + lt : (cid + lt * nctas) / ksplit; };
    auto tile_n0 = [&](int lt) {
        return (sk ? tile_base(lt) / tiles_m : tile_base(lt) % tiles_n) * kGemmBM;
    };
    auto tile_m0 = [&](int lt) { return (sk ? tile_base(lt) % tiles_m : tile_base(lt) / tiles_n) * kBN; };
    auto kpart = [&](int lt) { return (cid + lt * nctas) % ksplit; };
    // packed groups [kg0, kg1) of the unit's K part (parts differ by at most
    // one group), or of the tile's share of the stream-K run
    auto kg0 = [&](int lt) {
        if (sk) return lt == 0 ? g_first : 0;
        return (int)((int64_t)gtot * kpart(lt) / ksplit);
    };
    auto kg1 = [&](int lt) {
        if (sk) return lt == my_tiles - 1 ? g_end : gtot;
        return (int)((int64_t)gtot * (kpart(lt) + 1) / ksplit);
    };
    // the unit covers all of K: store Y; otherwise add onto the zeroed Y (or, with tickets, a partial tile)
    auto whole = [&](int lt) { return kg0(lt) == 0 && kg1(lt) == gtot; };

    const uint32_t bar = smem_addr(smem + L.bars);
    // stage s is full when its activation copy has landed and all dequantizing
    // warps have stored their A slices; one MMA commit empties it
    auto full = [&](int s) { return bar + 8u * s; };
    auto empty = [&](int s) { return bar + 8u * (4 + s); };
    auto p_full = [&](int s) { return bar + 8u * (16 + s); };
    auto p_empty = [&](int s) { return bar + 8u * (18 + s); };
    auto acc_full = [&](int b) { return bar + 8u * (20 + b); };
    auto acc_empty = [&](int b) { return bar + 8u * (22 + b); };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L.bars + 8 * 24);
    volatile int *last_slot = reinterpret_cast<volatile int *>(smem + L.bars + 8 * 25);

    if (tid == 0) {
        *last_slot = 0;
        for (int s = 0; s < kSA; ++s) {
            mbar_init(full(s), kGemmDeqWarps + 1);
            mbar_init(empty(s), 1);
        }
        for (int s = 0; s < kGemmStagesP; ++s) {
            mbar_init(p_full(s), 1);
            mbar_init(p_empty(s), kGemmDeqWarps);
        }
        for (int b = 0; b < kNbuf; ++b) {
            mbar_init(acc_full(b), 1);
            mbar_init(acc_empty(b), kNbuf == 1 ? kGemmDeqWarps : kGemmEpiWarps);
        }
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_addr(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------ activation TMA producer
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&xmap)) : "memory");
            griddep_wait();  // the binary16 activations of the conversion launch
            bool ok = true;
            int bi = 0;  // running activation stage counter
            for (int lt = 0; lt < my_tiles && ok; ++lt) {
                const int m0 = tile_m0(lt), kbase = kGemmStepsPerGroup * kg0(lt);
                const int ksteps = kGemmStepsPerGroup * (kg1(lt) - kg0(lt));
                for (int ks = 0; ks < ksteps && ok; ++ks, ++bi) {
                    const int sb = bi % kSA;
                    if (bi >= kSA) ok = mbar_wait(empty(sb), ((bi / kSA) - 1) & 1, kErrGemmWait);
                    if (!ok) break;
                    mbar_arrive_expect_tx(full(sb), kBBytes);
#pragma unroll
                    for (int a = 0; a < kGemmBK / kGemmAtomK; ++a)  // one box per 64-K atom
                        tma_load_2d(smem_addr(smem + L.b + sb * kBBytes + a * kBAtom), &xmap,
                                    (kbase + ks) * kGemmBK + a * kGemmAtomK, m0, full(sb));
                }
            }
        }
    } else if (warp == kGemmWarpPackedTma) {
        // ------------------------------------------------ packed-weight TMA producer
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&wmap)) : "memory");
            bool ok = true;
            int gi = 0;  // running packed-group counter
            for (int lt = 0; lt < my_tiles && ok; ++lt) {
                const int n0 = tile_n0(lt), gbase = kg0(lt), groups = kg1(lt) - kg0(lt);
                for (int g = 0; g < groups && ok; ++g, ++gi) {
                    const int sp = gi % kGemmStagesP;
                    if (gi >= kGemmStagesP)
                        ok = mbar_wait(p_empty(sp), ((gi / kGemmStagesP) - 1) & 1, kErrGemmWait);
                    if (!ok) break;
                    mbar_arrive_expect_tx(p_full(sp), kPBytes);
                    tma_load_2d(smem_addr(smem + L.p + sp * kPBytes), &wmap,
                                (gbase + g) * (gemm_group_advance(kFmt) / 2), n0, p_full(sp));
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = umma_idesc_f16(kGemmBM, kBN);
            bool ok = true;
            int ki = 0;  // running k-step counter (A and activation rings)
            for (int lt = 0; lt < my_tiles; ++lt) {
                const int buf = lt % kNbuf, use = lt / kNbuf;
                const int ksteps = kGemmStepsPerGroup * (kg1(lt) - kg0(lt));
                const uint32_t dacc = tmem + (uint32_t)(buf * kBN);
                if (ok && use > 0) ok = mbar_wait(acc_empty(buf), (use - 1) & 1, kErrGemmWait);
                for (int ks = 0; ks < ksteps && ok; ++ks, ++ki) {
                    const int s = ki % kSA;
                    ok = mbar_wait(full(s), (ki / kSA) & 1, kErrGemmWait);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t at = tmem + (uint32_t)(kACol0 + s * kGemmACols);
                    const uint32_t bs = smem_addr(smem + L.b + s * kBBytes);
#pragma unroll
                    for (int kk = 0; kk < kGemmBK / 16; ++kk) {
                        // 16 K per MMA: 8 TMEM columns of A; B: atom kk / 4, +32 bytes per step inside it
                        const uint64_t bd = umma_desc_sw128(bs + (uint32_t)((kk >> 2) * kBAtom)) + 2 * (kk & 3);
                        umma_f16_ts(dacc, at + (uint32_t)(8 * kk), bd, idesc, (ks | kk) != 0);
                    }
                    umma_commit(empty(s));
                }
                umma_commit(acc_full(buf));  // also after an error: releases the epilogue
            }
        }
    } else if (warp < 2 + kGemmDeqWarps) {
        // ------------------------------------------------ dequantize packed tiles into TMEM
        // K step j of a group (128 K) splits into four 32-wide slices, one per
        // warp of a lane quarter; a slice is two of the 16-wide pieces the
        // deq16_* functions convert (64-wide index J = 2 j + kq / 2, piece
        // 2 (kq % 2) + h), and 16 TMEM columns
        const int q = warp & 3;          // TMEM lane quarter this warp may access
        const int kq = (warp - 2) >> 2;  // 32-wide K slice of each 128-wide K step
        const int r = 32 * q + lane;     // this thread's weight row (TMEM lane)
        const uint32_t alane = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(kACol0 + 16 * kq);
        bool ok = true;
        int gi = 0, ki = 0;
        // With one accumulator (256-token tiles) these warps also drain it:
        // unit u's epilogue runs where they would otherwise wait for the MMA
        // to finish u (the K step kSA - 1 steps into unit u + 1, whose stage
        // slot the last K step of u frees), sixteen warps instead of four,
        // each storing 64 of the 256 columns of its 32 rows.
        int epi_unit = -1, epi_at = 0;
        auto drain = [&](int lt) {
            griddep_wait();  // Y (zeroed by the conversion launch for K parts)
            if (ok) ok = mbar_wait_warp(acc_full(0), lt & 1, kErrGemmWait);
            tc_fence_after();
            const int n = tile_n0(lt) + r, m0 = tile_m0(lt);
            const bool wh = sk ? whole(lt) : ksplit == 1;
            float rs = 1.f;
            if constexpr (kFmt == kFp8)
                if (n < p.N) rs = __ldg(reinterpret_cast<const float *>(p.W + (int64_t)n * p.row_bytes + p.K));
            if (ok) {
#pragma unroll 1
                for (int c = 0; c < 2; ++c) {
                    const int col = 64 * kq + 32 * c;
                    uint32_t v[32];
                    tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)col, v);
                    if (n < p.N) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            const int m = m0 + col + i;
                            if (m >= p.M) continue;
                            const float y = __uint_as_float(v[i]) * rs;
                            if (wh) p.Y[(int64_t)m * p.N + n] = y;
                            else atomicAdd(p.Y + (int64_t)m * p.N + n, y);
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty(0));
        };
        for (int lt = 0; lt < my_tiles; ++lt) {
            for (int g = kg0(lt); g < kg1(lt); ++g, ++gi) {
                const int sp = gi % kGemmStagesP;
                if (ok) ok = mbar_wait_warp(p_full(sp), (gi / kGemmStagesP) & 1, kErrGemmWait);
                const uint8_t *prow = smem + L.p + sp * kPBytes + r * kCB;
                float S[2], Mn[2];  // Q4_K / Q5_K: (S_j, Mn_j) of this thread's sub-block 4 j + kq in each K step
                if constexpr (kFmt == 4 || kFmt == 5) {
                    if (ok) {
                        const uint4 h = *reinterpret_cast<const uint4 *>(prow);
#pragma unroll
                        for (int j = 0; j < 2; ++j) q4k_coef(h, 4 * j + kq, S[j], Mn[j]);
                    }
                }
                // the two 128-wide K steps of the group (j a compile-time constant)
                auto step = [&](auto jc) {
                    constexpr int j = decltype(jc)::value;
                    const int sa = ki % kSA;
                    if (kNbuf == 1 && epi_unit >= 0 && ki == epi_at) {
                        drain(epi_unit);
                        epi_unit = -1;
                    }
                    if (ok && ki >= kSA) ok = mbar_wait_warp(empty(sa), ((ki / kSA) - 1) & 1, kErrGemmWait);
                    if (ok) {
                        tc_fence_after();
                        uint32_t v[16];
                        uint32_t(&v0)[8] = *reinterpret_cast<uint32_t(*)[8]>(&v[0]);
                        uint32_t(&v1)[8] = *reinterpret_cast<uint32_t(*)[8]>(&v[8]);
                        [[maybe_unused]] const int J = 2 * j + (kq >> 1), pc = 2 * (kq & 1);
                        if constexpr (kFmt == kFp8) {
                            deq16_fp8(prow, J, pc, v0);
                            deq16_fp8(prow, J, pc + 1, v1);
                        } else if constexpr (kFmt == 8) {
                            // piece pc + h of 64-wide step J: block 2 J + (pc + h) / 2 = 2 J + (kq % 2), half h
                            if (kq >> 1) {
                                if (kq & 1) { deq16_q8_0<2 * j + 1, 1>(prow, 0, v0); deq16_q8_0<2 * j + 1, 1>(prow, 1, v1); }
                                else        { deq16_q8_0<2 * j + 1, 0>(prow, 0, v0); deq16_q8_0<2 * j + 1, 0>(prow, 1, v1); }
                            } else {
                                if (kq & 1) { deq16_q8_0<2 * j, 1>(prow, 0, v0); deq16_q8_0<2 * j, 1>(prow, 1, v1); }
                                else        { deq16_q8_0<2 * j, 0>(prow, 0, v0); deq16_q8_0<2 * j, 0>(prow, 1, v1); }
                            }
                        } else if constexpr (kFmt == 5) {
                            deq16_q5_k(prow, J, pc, S[j], Mn[j], v0);
                            deq16_q5_k(prow, J, pc + 1, S[j], Mn[j], v1);
                        } else {
                            deq16_q4_k(prow, J, pc, S[j], Mn[j], v0);
                            deq16_q4_k(prow, J, pc + 1, S[j], Mn[j], v1);
                        }
                        tmem_st16(alane + (uint32_t)(sa * kGemmACols), v);
                        tmem_wait_st();
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(full(sa));
                    ++ki;
                };
                step(std::integral_constant<int, 0>{});
                step(std::integral_constant<int, 1>{});
                __syncwarp();
                if (lane == 0) mbar_arrive(p_empty(sp));
            }
            if (kNbuf == 1) {
                if (epi_unit >= 0) drain(epi_unit);  // a unit shorter than kSA steps (none today)
                epi_unit = lt;
                epi_at = ki + kSA - 1;
            }
        }
        if (kNbuf == 1 && epi_unit >= 0) drain(epi_unit);
    } else {
        // ------------------------------------------------ epilogue: TMEM -> Y (two accumulators;
        // with one, the dequantizing warps drain it)
        const int quarter = warp & 3;  // this warp may read TMEM lanes 32*quarter .. +31
        const int r = 32 * quarter + lane;  // weight row within the tile
        const int etid = tid - 32 * (2 + kGemmDeqWarps);  // 0 .. 127
        griddep_wait();  // Y and the tickets (cleared by the conversion launch)
        bool ok = true;
        for (int lt = 0; lt < (kNbuf == 1 ? 0 : my_tiles); ++lt) {
            const int buf = lt % kNbuf, use = lt / kNbuf;
            const int n0 = tile_n0(lt), m0 = tile_m0(lt);
            if (ok) ok = mbar_wait_warp(acc_full(buf), use & 1, kErrGemmWait);
            tc_fence_after();
            const int n = n0 + r;
            const int tile = tile_base(lt);
            // FP8: this row's scale (rows past N read nothing)
            float rs = 1.f;
            if constexpr (kFmt == kFp8)
                if (n < p.N) rs = __ldg(reinterpret_cast<const float *>(p.W + (int64_t)n * p.row_bytes + p.K));
            float *pw = p.partials + ((int64_t)tile * ksplit + kpart(lt)) * (kBN * kGemmBM);
            if (ok) {
#pragma unroll 1
                for (int col = 0; col < kBN; col += 32) {
                    uint32_t v[32];
                    tmem_ld32(tmem + ((uint32_t)(32 * quarter) << 16) + (uint32_t)(buf * kBN + col), v);
                    if constexpr (kFmt == kFp8) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * rs);
                    }
                    if (!p.tickets_mode) {
                        if (n < p.N) {
#pragma unroll
                            for (int i = 0; i < 32; ++i) {
                                const int m = m0 + col + i;
                                if (m >= p.M) continue;
                                if (ksplit == 1) p.Y[(int64_t)m * p.N + n] = __uint_as_float(v[i]);
                                else atomicAdd(p.Y + (int64_t)m * p.N + n, __uint_as_float(v[i]));
                            }
                        }
                    } else {
                        // this part's sums, column-major (a token's 128 rows contiguous)
#pragma unroll
                        for (int i = 0; i < 32; ++i) pw[(col + i) * kGemmBM + r] = __uint_as_float(v[i]);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty(buf));
            if (p.tickets_mode) {
                // ticket: the last part of the tile to finish adds all parts
                // in order, with every warp of the CTA (after the roles end)
                __threadfence();
                named_bar_sync(2, kGemmEpiWarps * 32);
                if (etid == 0) *last_slot = atomicAdd(p.tickets + tile, 1) == ksplit - 1;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    if constexpr (kNbuf == 2) {
        if (p.tickets_mode && *last_slot) {
            griddep_wait();
            // this CTA's unit (with tickets, every CTA has one) finished its
            // tile last: Y = part 0 + part 1 + ... in part order, four rows
            // (one float4 of each column-major partial tile) per thread and
            // step, with every warp of the CTA
            __threadfence();
            const int lt = my_tiles - 1, n0 = tile_n0(lt), m0 = tile_m0(lt);
            constexpr int kQ = kBN * kGemmBM / 4;  // float4s per partial tile
            const float4 *pt = reinterpret_cast<const float4 *>(p.partials) + (int64_t)tile_base(lt) * ksplit * kQ;
#pragma unroll 1
            for (int e = tid; e < kQ; e += kGemmThreads) {
                float4 a[QMM_GEMM_MAX_PARTS];
#pragma unroll
                for (int q = 0; q < QMM_GEMM_MAX_PARTS; ++q)
                    if (q < ksplit) a[q] = __ldcg(pt + (int64_t)q * kQ + e);
#pragma unroll
                for (int q = 1; q < QMM_GEMM_MAX_PARTS; ++q) {
                    if (q < ksplit) {
                        a[0].x += a[q].x; a[0].y += a[q].y; a[0].z += a[q].z; a[0].w += a[q].w;
                    }
                }
                const int m = m0 + e / (kGemmBM / 4), n = n0 + 4 * (e % (kGemmBM / 4));
                if (m >= p.M || n >= p.N) continue;
                float *y = p.Y + (int64_t)m * p.N + n;
                if ((p.N & 3) == 0) {
                    *reinterpret_cast<float4 *>(y) = a[0];
                } else {
                    const float o[4] = {a[0].x, a[0].y, a[0].z, a[0].w};
                    for (int i = 0; i < 4 && n + i < p.N; ++i) y[i] = o[i];
                }
            }
        }
    }
}

// ---------------------------------------------------------------- launcher
// Token tile and K split of a problem.  BN: the smallest of 32 / 64 / 128
// that holds M, else 256.  256-token tiles at least as many as the SMs:
// stream-K.  Otherwise K parts: as many as fill the SMs with one unit each
// when the output tiles alone do not (at most one part per packed group of
// K; two for 256-token tiles).
constexpr int kGemmStreamKWaves = 4;  // 256-token tiles per SM from which stream-K runs
struct GemmPlan {
    int bn, ksplit, tiles, tickets, stream_k;
};
static GemmPlan gemm_plan(int M, int N, int K, int sms) {
    GemmPlan pl;
    const int groups = K / kGroup;
    const int tiles_n = (N + kGemmBM - 1) / kGemmBM;
    // two K halves when the tiles fill under about half of the SMs
    auto occupancy = [&](int u) {
        const int waves = (u + sms - 1) / sms;
        return (double)u / ((double)waves * sms);
    };
    auto halves = [&](int tiles) {
        return (groups % 2 == 0 && occupancy(2 * tiles) > occupancy(tiles) + 0.2) ? 2 : 1;
    };
    pl.bn = M <= 32 ? 32 : M <= 64 ? 64 : M <= 128 ? 128 : 256;
    pl.tiles = tiles_n * ((M + pl.bn - 1) / pl.bn);
    pl.stream_k = 0;
    if (pl.bn == 256) {
        // four or more waves of tiles: stream-K (it recovers the idle part of
        // the last wave, up to one unit; its cut tiles cost a few microseconds)
        pl.stream_k = pl.tiles >= kGemmStreamKWaves * sms;
        pl.ksplit = pl.stream_k ? 1 : halves(pl.tiles);
        pl.tickets = 0;
    } else {
        // (tiles x parts <= SMs: each CTA runs one unit, which the final
        // reduction of the kernel relies on)
        int ks = sms / pl.tiles;
        if (ks > groups) ks = groups;
        if (ks > QMM_GEMM_MAX_PARTS) ks = QMM_GEMM_MAX_PARTS;
        pl.ksplit = ks < 1 ? 1 : ks;
        pl.tickets = pl.ksplit > 1;
    }
    return pl;
}

// Workspace: the binary16 copy of X, then (with a K split) the partial tiles
// and one ticket word per tile, each region 256-byte aligned.
struct GemmWorkspace {
    size_t xh, partials, tickets, total;
};
static GemmWorkspace gemm_workspace(int M, int N, int K, int sms) {
    const GemmPlan pl = gemm_plan(M, N, K, sms);
    auto up = [](size_t v) { return (v + 255) & ~(size_t)255; };
    GemmWorkspace w;
    w.xh = 0;
    w.partials = up((size_t)M * (size_t)K * 2);
    const size_t pbytes = pl.tickets ? (size_t)pl.tiles * pl.ksplit * pl.bn * kGemmBM * 4 : 0;
    w.tickets = up(w.partials + pbytes);
    w.total = w.tickets + (pl.tickets ? up((size_t)pl.tiles * 4) : 0);
    return w;
}

size_t gemm_workspace_bytes(int fmt, int M, int N, int K, int sms) {
    (void)fmt;
    return gemm_workspace(M, N, K, sms).total;
}

template <int kFmt, int kBN>
static cudaError_t launch_gemm_t(const void *W, const uint16_t *X, float *Y, int M, int N, int K,
                                 void *workspace, int sms, cudaStream_t stream) {
    const GemmPlan pl = gemm_plan(M, N, K, sms);
    const GemmWorkspace ws = gemm_workspace(M, N, K, sms);
    uint8_t *wb = static_cast<uint8_t *>(workspace);
    __half *Xh = reinterpret_cast<__half *>(wb + ws.xh);
    const int nt = pl.tickets ? pl.tiles : 0;
    const int64_t ny = (!pl.tickets && pl.ksplit > 1) ? (int64_t)M * N : 0;  // Y to add the halves onto
    const int64_t n8 = (int64_t)M * K / 8;
    const int grid = pl.stream_k ? sms : (pl.tiles * pl.ksplit < sms ? pl.tiles * pl.ksplit : sms);
    if (pl.tickets && pl.tiles * pl.ksplit > grid) return cudaErrorInvalidConfiguration;  // one unit per CTA
    SplitTiles st;
    st.ctas = pl.stream_k ? grid : 0;
    st.gtot = K / kGroup;
    st.tiles_m = (M + kBN - 1) / kBN;
    st.bn = kBN;
    st.M = M;
    st.N = N;
    st.gall = (int64_t)pl.tiles * st.gtot;
    const int64_t work = n8 > ny / 4 ? n8 : ny / 4;
    int cgrid = (int)((work + 255) / 256);
    if (cgrid > 148 * 16) cgrid = 148 * 16;
    if (cgrid < st.ctas - 1) cgrid = st.ctas - 1;  // a block per stream-K boundary
    if (cgrid < 1) cgrid = 1;
    qmm_x_to_f16_kernel<<<cgrid, 256, 0, stream>>>(X, Xh, n8, reinterpret_cast<int *>(wb + ws.tickets), nt,
                                                   Y, ny, st);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;

    CUtensorMap xmap, wmap;
    e = encode_tmap_2d(&xmap, Xh, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, (uint64_t)K, (uint64_t)M,
                       (uint64_t)K * 2, kGemmAtomK, kBN, CU_TENSOR_MAP_SWIZZLE_128B);
    if (e != cudaSuccess) return e;
    // a box is 128 rows x one stage pitch (FP8: past a row's end, zero-filled)
    constexpr int kCB = gemm_group_bytes(kFmt);
    const int64_t row_bytes =
        kFmt == kFp8 ? (int64_t)K + kFp8RowPad : (int64_t)(K / kGroup) * gemm_group_advance(kFmt);
    e = encode_tmap_2d(&wmap, W, CU_TENSOR_MAP_DATA_TYPE_UINT16, (uint64_t)(row_bytes / 2),
                       (uint64_t)N, (uint64_t)row_bytes, kCB / 2, kGemmBM);
    if (e != cudaSuccess) return e;

    const GemmLayout L = gemm_layout(kFmt, kBN);
    static std::atomic<uint64_t> attr_done{0}, attr_done_sk{0};
    e = set_smem_limit_once(reinterpret_cast<const void *>(qmm_gemm_kernel<kFmt, kBN, false>), L.total, attr_done);
    if (e != cudaSuccess) return e;
    if constexpr (kBN == 256) {
        if (pl.stream_k) {
            e = set_smem_limit_once(reinterpret_cast<const void *>(qmm_gemm_kernel<kFmt, 256, true>), L.total,
                                    attr_done_sk);
            if (e != cudaSuccess) return e;
        }
    }
    GemmParams p;
    p.Y = Y;
    p.W = static_cast<const uint8_t *>(W);
    p.row_bytes = row_bytes;
    p.partials = reinterpret_cast<float *>(wb + ws.partials);
    p.tickets = reinterpret_cast<int *>(wb + ws.tickets);
    p.M = M;
    p.N = N;
    p.K = K;
    p.ksplit = pl.ksplit;
    p.tickets_mode = pl.tickets;
    // one persistent CTA per SM (stream-K: exactly one per SM, the runs'
    // divisor), by programmatic dependent launch: the CTAs' prologue and
    // weight stages overlap the conversion launch, and the roles that read X
    // or write Y, the tickets or the partial tiles wait for it (griddep_wait)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(kGemmThreads, 1, 1);
    cfg.dynamicSmemBytes = (size_t)L.total;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if constexpr (kBN == 256) {
        if (pl.stream_k) return cudaLaunchKernelEx(&cfg, qmm_gemm_kernel<kFmt, 256, true>, xmap, wmap, p);
    }
    return cudaLaunchKernelEx(&cfg, qmm_gemm_kernel<kFmt, kBN, false>, xmap, wmap, p);
}

template <int kFmt>
static cudaError_t launch_gemm_f(const void *W, const uint16_t *X, float *Y, int M, int N, int K,
                                 void *workspace, int sms, cudaStream_t stream) {
    switch (gemm_plan(M, N, K, sms).bn) {
    case 32: return launch_gemm_t<kFmt, 32>(W, X, Y, M, N, K, workspace, sms, stream);
    case 64: return launch_gemm_t<kFmt, 64>(W, X, Y, M, N, K, workspace, sms, stream);
    case 128: return launch_gemm_t<kFmt, 128>(W, X, Y, M, N, K, workspace, sms, stream);
    default: return launch_gemm_t<kFmt, 256>(W, X, Y, M, N, K, workspace, sms, stream);
    }
}

cudaError_t launch_gemm(int fmt, const void *W, const uint16_t *X, float *Y, int M, int N, int K,
                        void *workspace, size_t workspace_bytes, int sms, cudaStream_t stream) {
    if (workspace_bytes < gemm_workspace_bytes(fmt, M, N, K, sms)) return cudaErrorInvalidValue;
    if (fmt == 8) return launch_gemm_f<8>(W, X, Y, M, N, K, workspace, sms, stream);
    if (fmt == kFp8) return launch_gemm_f<kFp8>(W, X, Y, M, N, K, workspace, sms, stream);
    if (fmt == 5) return launch_gemm_f<5>(W, X, Y, M, N, K, workspace, sms, stream);
    return launch_gemm_f<4>(W, X, Y, M, N, K, workspace, sms, stream);
}

}  // namespace qmm
