// gemv_rows.cu -- decode matmul for M <= 8 tokens without thread-block
// clusters: one CTA owns 16 weight rows over the whole K.
//
// Each CTA streams its tile with one 2-D tensor-map TMA copy (16 rows x 256
// weights) per chunk into a deep ring (up to 16 / 32 stages), and eight
// consumer warps take the chunks round-robin (chunk i -> warp i % 8).  The per-chunk arithmetic is the
// one of gemv.cu (exact integer codes on m16n8k16 tensor-core MMAs, scales in
// fp32 per 32-weight block).  The eight warps' partial sums are added in
// shared memory in warp order, so the result is deterministic; there is no
// cluster barrier, no distributed shared memory and no workspace.  Used when
// the row count alone fills the GPU's SMs and the activations are few enough
// (M <= 8) to restage cheaply per CTA.
#include "common.cuh"

namespace qmm {

constexpr int kRowsR = 16;
constexpr int kWarpsR = 8;
constexpr int kThreadsR = (kWarpsR + 1) * 32;

struct RowsLayout {
    int ring, xh, xs, coef, ypart, bars, total;
};

__host__ __device__ inline RowsLayout rows_layout(int fmt, int M, int stages, int win) {
    const int slot = fmt == 8 ? kQ8GroupBytes : kQ4Bytes;
    RowsLayout L;
    int off = 0;
    L.ring = off;
    off += stages * kRowsR * slot;
    L.xh = off;
    off += M * (win * kGroup + 32) * 2;
    L.xs = off;
    off += fmt == 4 ? win * 8 * 8 * 4 : 0;
    L.coef = off;
    off += fmt == 4 ? kWarpsR * 16 * 8 * 4 : 0;
    L.ypart = off;
    off += kWarpsR * kRowsR * 8 * 4;
    off = (off + 15) & ~15;
    L.bars = off;
    off += 2 * stages * 8;
    L.total = off;
    return L;
}

struct RowsParams {
    float *Y;
    const uint16_t *X;
    int M, N, K;
    int nchunks;  // K / 256
    int stages;   // ring depth
    int win;      // activation window in chunks (a multiple of 8, or nchunks)
};

template <int kFmt>
__device__ __forceinline__ void rows_stage_x(const RowsParams &p, __half *xh, float *xs, int xstride,
                                             int w0, int wn, int tid) {
    constexpr int kMT = 8;
    const int ngr = (wn * kGroup) / 8;
    const int kw = w0 * kGroup;
    for (int idx = tid; idx < p.M * ngr; idx += kWarpsR * 32) {
        const int m = idx / ngr, kg = idx - m * ngr;
        const uint4 v = __ldg(reinterpret_cast<const uint4 *>(p.X + (int64_t)m * p.K + kw + 8 * kg));
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
        if constexpr (kFmt == 4) {
            const float2 s02 = __half22float2(h02), s13 = __half22float2(h13);
            const float2 s46 = __half22float2(h46), s57 = __half22float2(h57);
            float sum = ((s02.x + s13.x) + (s02.y + s13.y)) + ((s46.x + s57.x) + (s46.y + s57.y));
            sum += __shfl_xor_sync(0xffffffffu, sum, 1);
            sum += __shfl_xor_sync(0xffffffffu, sum, 2);
            if ((kg & 3) == 0) xs[(kg >> 2) * kMT + m] = sum;
        }
    }
}

// One CTA per 16-row tile.  Chunk i of the tile goes to stage i % stages
// and to consumer warp i % 8.
template <int kFmt>
__global__ void __launch_bounds__(kThreadsR)
gemv_rows_kernel(const __grid_constant__ CUtensorMap wmap, const RowsParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int kCB = kFmt == 8 ? kQ8GroupBytes : kQ4Bytes;
    constexpr int kNT = 1;
    constexpr int kMT = 8;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int row0 = blockIdx.x * kRowsR;
    const int nch = p.nchunks;
    const int xstride = p.win * kGroup + 32;
    const RowsLayout L = rows_layout(kFmt, p.M, p.stages, p.win);
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
            mbar_init(empty_bar(s), 1);
        }
        fence_mbar_init();
    }
    if constexpr (kFmt == 4)
        for (int idx = tid; idx < p.win * 8 * kMT; idx += kThreadsR) xs[idx] = 0.f;
    if (warp == kWarpsR && lane == 0) {
        // descriptor fetch and L2 prefetch of the first stages (safe before
        // the dependency wait: nothing lands in shared memory)
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&wmap)) : "memory");
        for (int i = 0; i < nch && i < p.stages; ++i) tma_prefetch_l2_2d(&wmap, i * (kCB / 2), row0);
    }
    __syncthreads();
    // programmatic dependent launch: see gemv.cu
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (warp == kWarpsR) {
        // ---------------- producer
        if (lane == 0) {
            for (int i = 0; i < nch; ++i) {
                const int s = i % p.stages;
                if (i >= p.stages && !mbar_wait(empty_bar(s), ((i / p.stages) - 1) & 1, kErrGemvEmptyWait))
                    break;  // bug path: consumers then time out on their full barriers
                mbar_arrive_expect_tx(full_bar(s), (uint32_t)(kRowsR * kCB));
                tma_load_2d(smem_addr(ring + s * kRowsR * kCB), &wmap, i * (kCB / 2), row0, full_bar(s));
            }
        }
    } else {
        // ---------------- consumers: warp w takes chunks w, w + 8, ...
        const int g = lane >> 2, t = lane & 3;
        float acc[kNT][4] = {{0.f, 0.f, 0.f, 0.f}};
        const __half *xrow = xh + g * xstride;
        const int gvalid = p.M - g;
        float *cw = coef + warp * 16 * 8;
        bool ok = true;  // warp-uniform, see gemv.cu
        for (int w0 = 0; w0 < nch; w0 += p.win) {
            const int wn = min(p.win, nch - w0);
            if (w0 > 0) named_bar_sync(1, kWarpsR * 32);
            rows_stage_x<kFmt>(p, xh, xs, xstride, w0, wn, tid);
            named_bar_sync(1, kWarpsR * 32);
            for (int i = w0 + warp; i < w0 + wn; i += kWarpsR) {
                const int s = i % p.stages, li = i - w0;
                if (ok) ok = mbar_wait_warp(full_bar(s), (i / p.stages) & 1, kErrGemvFullWait);
                if (!ok) continue;
                const uint8_t *base = ring + s * kRowsR * kCB;
                const uint8_t *r0 = base + g * kCB;
                const uint8_t *r1 = base + (g + 8) * kCB;
                const __half *xr = xrow + li * kGroup;
                if constexpr (kFmt == 8) {
                    q8_block<0, kNT>(r0, r1, xr, xstride, xs, li * 8 + 0, t, gvalid, acc);
                    q8_block<1, kNT>(r0, r1, xr, xstride, xs, li * 8 + 1, t, gvalid, acc);
                    q8_block<2, kNT>(r0, r1, xr, xstride, xs, li * 8 + 2, t, gvalid, acc);
                    q8_block<3, kNT>(r0, r1, xr, xstride, xs, li * 8 + 3, t, gvalid, acc);
                    q8_block<4, kNT>(r0, r1, xr, xstride, xs, li * 8 + 4, t, gvalid, acc);
                    q8_block<5, kNT>(r0, r1, xr, xstride, xs, li * 8 + 5, t, gvalid, acc);
                    q8_block<6, kNT>(r0, r1, xr, xstride, xs, li * 8 + 6, t, gvalid, acc);
                    q8_block<7, kNT>(r0, r1, xr, xstride, xs, li * 8 + 7, t, gvalid, acc);
                } else {
                    q4k_half<kNT>(base, r0, r1, xr, xstride, xs, li, cw, lane, g, t, gvalid, 0, acc);
                    q4k_half<kNT>(base, r0, r1, xr, xstride, xs, li, cw, lane, g, t, gvalid, 1, acc);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(empty_bar(s));
            }
        }
        float *yp = ypart + warp * kRowsR * kMT;
        *reinterpret_cast<float2 *>(yp + g * kMT + 2 * t) = make_float2(acc[0][0], acc[0][1]);
        *reinterpret_cast<float2 *>(yp + (g + 8) * kMT + 2 * t) = make_float2(acc[0][2], acc[0][3]);
        named_bar_sync(1, kWarpsR * 32);
        // fixed-order sum of the eight warps' partials
        for (int idx = tid; idx < kRowsR * p.M; idx += kWarpsR * 32) {
            const int r = idx / p.M, m = idx - r * p.M;
            if (row0 + r < p.N) {
                float sum = 0.f;
#pragma unroll
                for (int w = 0; w < kWarpsR; ++w) sum += ypart[(w * kRowsR + r) * kMT + m];
                p.Y[(int64_t)m * p.N + row0 + r] = sum;
            }
        }
    }
}

#ifndef QMM_ROWS_CARVEOUT  // preferred shared-memory carveout in %, -1 = driver default
#define QMM_ROWS_CARVEOUT -1
#endif
#ifndef QMM_ROWS_MAX_STAGES_Q8
#define QMM_ROWS_MAX_STAGES_Q8 16
#endif
#ifndef QMM_ROWS_MAX_STAGES_Q4
#define QMM_ROWS_MAX_STAGES_Q4 32
#endif

// Ring depth.  Chunk i goes to warp i % 8 and stage i % stages; a stage may
// only be reused by the warp that used it before (an mbarrier parity wait
// cannot tell phase k from phase k + 2), so the depth is a multiple of 8:
// 16 (Q8_0) or 32 (Q4_K), lowered (to at least 8) until the grid fits one
// wave of resident CTAs; one CTA per tile (a persistent loop over tiles
// measured slower on the decode shapes).
bool gemv_rows_plan(int fmt, int M, int N, int K, int sms, RowsParams &p, int &smem, int &grid) {
    const int nch = K / kGroup;
    const int ntiles = (N + kRowsR - 1) / kRowsR;
    // window: all of K while M * K <= 64 chunks of binary16 (32 KB), else the
    // largest multiple of 8 chunks within that budget (at least 8)
    int win = nch;
    if (M * nch > 64) {
        win = (64 / M) / 8 * 8;
        if (win < 8) win = 8;
    }
    int st = fmt == 8 ? QMM_ROWS_MAX_STAGES_Q8 : QMM_ROWS_MAX_STAGES_Q4;
    while (true) {
        const int sm = rows_layout(fmt, M, st, win).total;
        const int by_smem = (227 * 1024) / (sm + 1024);
        const int by_warps = 64 / (kThreadsR / 32);
        const int per_sm = by_smem < by_warps ? by_smem : by_warps;
        if (st <= 8 || ntiles <= sms * per_sm) break;
        st -= 8;
    }
    p.stages = st;
    p.win = win;
    smem = rows_layout(fmt, M, st, win).total;
    grid = ntiles;
    return true;
}

template <int kFmt>
static cudaError_t launch_rows_t(const void *W, const RowsParams &p, int smem, int grid,
                                 cudaStream_t stream) {
    constexpr int kCB = kFmt == 8 ? kQ8GroupBytes : kQ4Bytes;
    const int64_t row_bytes = (int64_t)p.nchunks * kCB;
    CUtensorMap wmap;
    cudaError_t e = encode_tmap_2d(&wmap, W, CU_TENSOR_MAP_DATA_TYPE_UINT16, (uint64_t)(row_bytes / 2),
                                   (uint64_t)p.N, (uint64_t)row_bytes, kCB / 2, kRowsR);
    if (e != cudaSuccess) return e;
    static bool attr_set = false;
    if (!attr_set) {
        e = cudaFuncSetAttribute(gemv_rows_kernel<kFmt>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 227 * 1024);
        if (e != cudaSuccess) return e;
#if QMM_ROWS_CARVEOUT >= 0
        e = cudaFuncSetAttribute(gemv_rows_kernel<kFmt>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 QMM_ROWS_CARVEOUT);
        if (e != cudaSuccess) return e;
#endif
        attr_set = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(kThreadsR, 1, 1);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gemv_rows_kernel<kFmt>, wmap, p);
}

cudaError_t launch_gemv_rows(int fmt, const void *W, const uint16_t *X, float *Y, int M, int N, int K,
                             int sms, cudaStream_t stream) {
    RowsParams p;
    p.Y = Y;
    p.X = X;
    p.M = M;
    p.N = N;
    p.K = K;
    p.nchunks = K / kGroup;
    int smem = 0, grid = 1;
    gemv_rows_plan(fmt, M, N, K, sms, p, smem, grid);
    return fmt == 8 ? launch_rows_t<8>(W, p, smem, grid, stream)
                    : launch_rows_t<4>(W, p, smem, grid, stream);
}

}  // namespace qmm
