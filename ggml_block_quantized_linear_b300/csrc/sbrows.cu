// sbrows.cu -- decode matmul at M = 1 for the superblock formats whose
// superblocks are not 16-byte aligned inside a row: Q6_K (210 bytes, the
// output-head type of a Q4K model), Q3_K (110) and Q2_K (84).
//
// The row-tile kernel (gemv_rows.cu) stages 16 rows x 2 superblocks, which
// needs 16-byte multiples; eight superblocks of these formats are (1680 /
// 880 / 672 bytes).  So a stage here is one TMA box of 8 rows x 8
// superblocks, streamed by one producer thread into a ring of shared-memory
// stages deep enough to keep ~70 KB in flight per CTA; the token's bf16
// activations stay resident in shared memory (one bulk copy per CTA).  Eight
// consumer warps each own one row of a box and decode it with the CUDA-core
// lane decoders of q6k.cu and kquant.cu (lane l: weights 8l .. 8l + 7 of a
// superblock), reading the superblocks from shared memory instead of global
// memory.  A row's sum is formed as in the direct-load kernels at one token
// (per lane over the superblocks in order, exact codes with the sub-block
// scale applied once per superblock, then a fixed butterfly across the
// lanes), so the results are the same bits.
// CTAs are persistent over 8-row tiles (CTA b takes tiles b, b + G, ...);
// every wait is bounded (common.cuh); programmatic dependent launch as in
// the other decode kernels.
#include "common.cuh"

namespace qmm {

constexpr int kSbTileRows = 8;  // rows per tile: one per consumer warp
constexpr int kSbSeg = 8;       // superblocks per stage row
constexpr int kSbWarps = 8;
constexpr int kSbThreads = (kSbWarps + 1) * 32;  // + the producer warp
constexpr int kSbRingBytes = 72 * 1024;           // ring per CTA (two CTAs per SM)
constexpr int kSbMaxXBytes = 64 * 1024;           // resident activations: K <= 32768

__host__ __device__ constexpr int sb_bytes(int fmt) { return fmt == 6 ? 210 : fmt == 3 ? 110 : 84; }
// a box row in shared memory, and a stage (rounded to 128 bytes)
__host__ __device__ constexpr int sb_row_pitch(int fmt) { return kSbSeg * sb_bytes(fmt); }
__host__ __device__ constexpr int sb_stage_bytes(int fmt) {
    return (kSbTileRows * sb_row_pitch(fmt) + 127) / 128 * 128;
}
__host__ __device__ constexpr int sb_stages(int fmt) {
    return kSbRingBytes / sb_stage_bytes(fmt) > 16 ? 16 : kSbRingBytes / sb_stage_bytes(fmt);
}

struct SbParams {
    float *Y;
    const uint16_t *X;
    int N, K;
    int nsb;     // superblocks per row (K / 256)
    int nseg;    // stages per tile (ceil(nsb / 8))
    int ntiles;  // ceil(N / 8)
};

// One superblock of one row against the token: lane l's 8 weights times the
// activations at xsb (the superblock's 256 bf16 values in shared memory),
// added to acc in the one-token direct-load kernels' order.
template <int kFmt>
__device__ __forceinline__ void sb_lane_dot(const uint8_t *blk, const uint16_t *xsb, int lane, float &acc) {
    if constexpr (kFmt == 6) {
        float c[8];
        q6_lane_codes<true>(blk, lane, c);
        const float S = q6_lane_scale(blk, lane);
        const int koff = 128 * (lane >> 4) + 32 * ((lane >> 2) & 3) + 8 * (lane & 3);
        const uint4 xv = *reinterpret_cast<const uint4 *>(xsb + koff);
        const uint32_t w[4] = {xv.x, xv.y, xv.z, xv.w};
        acc = fmaf(S, q6_codes_dot(c, w), acc);
    } else {
        const KqCodes kc = kq_lane_codes<kFmt>(kq_lane_load<kFmt, true>(blk, lane), lane);
        const uint4 xv = *reinterpret_cast<const uint4 *>(xsb + 8 * lane);
        const uint32_t w[4] = {xv.x, xv.y, xv.z, xv.w};
        acc = kq_codes_dot<kFmt>(kc, w, acc);
    }
}

template <int kFmt>
__global__ void __launch_bounds__(kSbThreads, 2)
qmm_sbrows_kernel(const __grid_constant__ CUtensorMap wmap, const SbParams p) {
    constexpr int kB = sb_bytes(kFmt), kPitch = sb_row_pitch(kFmt);
    constexpr int kStage = sb_stage_bytes(kFmt), kNst = sb_stages(kFmt);
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t *ring = smem;
    uint16_t *xs = reinterpret_cast<uint16_t *>(smem + kNst * kStage);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t bar0 = smem_addr(smem + kNst * kStage + p.K * 2);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (kNst + s); };
    const uint32_t xfull = bar0 + 16u * kNst;
    if (tid == 0) {
        for (int s = 0; s < kNst; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), kSbWarps);
        }
        mbar_init(xfull, 1);
        fence_mbar_init();
    }
    if (warp == kSbWarps && lane == 0) {
        // descriptor fetch and L2 prefetch of the first tile's leading stages
        // (nothing lands in shared memory: safe before the dependency wait)
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&wmap)) : "memory");
        for (int j = 0; j < p.nseg && j < kNst; ++j)
            tma_prefetch_l2_2d(&wmap, j * (kPitch / 8), (int)blockIdx.x * kSbTileRows);
        bulk_prefetch_l2(p.X, (uint32_t)(p.K * 2));
    }
    __syncthreads();
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (warp == kSbWarps) {
        // ---------------- producer (one thread): the activations, then the stages in order
        if (lane == 0) {
            mbar_arrive_expect_tx(xfull, (uint32_t)(p.K * 2));
            bulk_g2s(smem_addr(xs), p.X, (uint32_t)(p.K * 2), xfull);
            int it = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < p.ntiles; tile += gridDim.x) {
                for (int seg = 0; seg < p.nseg; ++seg, ++it) {
                    const int s = it % kNst;
                    if (it >= kNst && !mbar_wait(empty_bar(s), ((it / kNst) - 1) & 1, kErrGemvEmptyWait)) {
                        ok = false;  // bug path: the consumers then time out on their full barriers
                        break;
                    }
                    // a box may run past the row's end or past N (zero filled); its bytes all count
                    mbar_arrive_expect_tx(full_bar(s), (uint32_t)(kSbTileRows * kPitch));
                    tma_load_2d(smem_addr(ring + s * kStage), &wmap, seg * (kPitch / 8), tile * kSbTileRows,
                                full_bar(s));
                }
            }
        }
    } else {
        // ---------------- consumers: warp w takes row w of every box
        bool ok = mbar_wait_warp(xfull, 0, kErrGemvFullWait);  // warp-uniform
        int it = 0;
        for (int tile = blockIdx.x; tile < p.ntiles; tile += gridDim.x) {
            float acc = 0.f;
            for (int seg = 0; seg < p.nseg; ++seg, ++it) {
                const int s = it % kNst;
                if (ok) ok = mbar_wait_warp(full_bar(s), (it / kNst) & 1, kErrGemvFullWait);
                if (ok) {
                    const uint8_t *rowp = ring + s * kStage + warp * kPitch;
                    const int sb0 = seg * kSbSeg;
                    const uint16_t *xsb = xs + sb0 * 256;
                    if (sb0 + kSbSeg <= p.nsb) {
#pragma unroll
                        for (int j = 0; j < kSbSeg; ++j) sb_lane_dot<kFmt>(rowp + j * kB, xsb + j * 256, lane, acc);
                    } else {
                        for (int j = 0; sb0 + j < p.nsb; ++j)
                            sb_lane_dot<kFmt>(rowp + j * kB, xsb + j * 256, lane, acc);
                    }
                }
                __syncwarp();
                if (ok && lane == 0) mbar_arrive(empty_bar(s));
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
            const int n = tile * kSbTileRows + warp;
            if (ok && lane == 0 && n < p.N) p.Y[n] = acc;
        }
    }
}

// M = 1, a row a 16-byte multiple (TMA strides), resident activations.
bool sbrows_supported(int fmt, int M, int K) {
    if (fmt != 6 && fmt != 3 && fmt != 2) return false;
    const int64_t row_bytes = (int64_t)(K / 256) * sb_bytes(fmt);
    return M == 1 && row_bytes % 16 == 0 && (int64_t)K * 2 <= kSbMaxXBytes;
}

template <int kFmt>
static cudaError_t launch_sbrows_t(const void *W, const uint16_t *X, float *Y, int N, int K, int sms,
                                   cudaStream_t stream) {
    constexpr int kNst = sb_stages(kFmt);
    static std::atomic<uint64_t> done{0};
    const void *fn = reinterpret_cast<const void *>(qmm_sbrows_kernel<kFmt>);
    cudaError_t e = set_smem_limit_once(fn, 227 * 1024, done);
    if (e != cudaSuccess) return e;
    SbParams p;
    p.Y = Y;
    p.X = X;
    p.N = N;
    p.K = K;
    p.nsb = K / 256;
    p.nseg = (p.nsb + kSbSeg - 1) / kSbSeg;
    p.ntiles = (N + kSbTileRows - 1) / kSbTileRows;
    const int smem = kNst * sb_stage_bytes(kFmt) + K * 2 + (2 * kNst + 1) * 8;
    int occ = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, qmm_sbrows_kernel<kFmt>, kSbThreads, (size_t)smem);
    if (e != cudaSuccess) return e;
    if (occ < 1) occ = 1;
    const int64_t cap = (int64_t)sms * occ;
    const int grid = (int)(p.ntiles < cap ? p.ntiles : cap);
    const int64_t row_bytes = (int64_t)p.nsb * sb_bytes(kFmt);
    CUtensorMap wmap;
    e = encode_tmap_2d(&wmap, W, CU_TENSOR_MAP_DATA_TYPE_UINT64, (uint64_t)(row_bytes / 8), (uint64_t)N,
                       (uint64_t)row_bytes, (uint32_t)(sb_row_pitch(kFmt) / 8), kSbTileRows);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(kSbThreads, 1, 1);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, qmm_sbrows_kernel<kFmt>, wmap, p);
}

cudaError_t launch_sbrows(int fmt, const void *W, const uint16_t *X, float *Y, int N, int K, int sms,
                          cudaStream_t stream) {
    if (fmt == 6) return launch_sbrows_t<6>(W, X, Y, N, K, sms, stream);
    if (fmt == 3) return launch_sbrows_t<3>(W, X, Y, N, K, sms, stream);
    return launch_sbrows_t<2>(W, X, Y, N, K, sms, stream);
}

}  // namespace qmm
