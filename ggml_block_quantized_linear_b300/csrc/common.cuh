// common.cuh -- shared device helpers of the qmm CUDA library (sm_103a):
// shared-memory addresses, mbarriers with bounded waits, 1-D bulk copies,
// thread-block-cluster barriers and distributed shared memory, the legacy
// warp-level MMA used by the decode kernel, and the device error word.
#pragma once

#include <cuda.h>  // CUtensorMap (types only; the driver is reached through the runtime)
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>

#include <atomic>

namespace qmm {

// Block geometry of the two formats (see include/qmm.h for the layouts).
constexpr int kQ8Weights = 32;
constexpr int kQ8Bytes = 34;
constexpr int kQ4Weights = 256;
constexpr int kQ4Bytes = 144;
// Every kernel walks the weights in groups of 256 (8 Q8_0 blocks = 272 bytes,
// one Q4_K superblock = 144 bytes); both are multiples of 16 bytes.
constexpr int kGroup = 256;
constexpr int kQ8GroupBytes = 272;
// FP8 E4M3 with a scale per row: a packed row is K codes, the fp32 row scale
// and 12 zero bytes (format value 80).
constexpr int kFp8 = 80;
constexpr int kFp8RowPad = 16;

// Device error word: nonzero codes are written by kernels whose bounded wait
// ran out (see qmm_device_error_take).  The library is one translation unit
// (qmm_lib.cu), so this is its only definition.
__device__ int g_device_error = 0;
// The codes match qmm_device_error in include/qmm.h.
enum DeviceError : int {
    kErrNone = 0,
    kErrGemvFullWait = 101,
    kErrGemvEmptyWait = 102,
    kErrGemmWait = 201,
    kErrBadId = 301,
    kErrSelftestTimeout = 901,
    kErrSelftestUnexpected = 902,
};

__device__ __forceinline__ void record_error(int code) { atomicCAS(&g_device_error, 0, code); }

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait limit of every spin on an mbarrier: about two seconds.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
#ifndef QMM_TRYWAIT_HINT_NS
#define QMM_TRYWAIT_HINT_NS 0
#endif
// One mbarrier.try_wait: the hardware may suspend the thread for a short,
// system-dependent time (or up to an explicit hint, when one is compiled in)
// until the phase completes.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
#if QMM_TRYWAIT_HINT_NS > 0
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(QMM_TRYWAIT_HINT_NS)
        : "memory");
#else
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
#endif
    return ok != 0;
}
// Bounded wait for the phase with the given parity to complete.  Returns
// false (after recording `err`) if it has not completed within limit_ns.
__device__ __forceinline__ bool mbar_wait_limit(uint32_t bar, uint32_t parity, int err, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t i = 0;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 255u) == 255u && global_timer_ns() - t0 > limit_ns) {
            record_error(err);
            return false;
        }
    }
}
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int err) {
    return mbar_wait_limit(bar, parity, err, kWaitLimitNs);
}

// mbar_wait by a whole warp, with a warp-uniform answer (true only if every
// lane saw the phase complete), so that the warp never diverges around
// warp-synchronous instructions after a timeout.
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity, int err) {
    const bool ok = mbar_wait(bar, parity, err);
    return __all_sync(0xffffffffu, ok) != 0;
}

// 1-D bulk copy global -> shared (this CTA), completing on an mbarrier.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes,
                                         uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// 2-D tiled tensor copy global -> shared (this CTA), completing on an
// mbarrier.  (x, y) are element coordinates of the box's first element; x *
// element size must be a multiple of 16 bytes.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

// Prefetch a 2-D box of a tensor into L2 (no shared-memory destination).
__device__ __forceinline__ void tma_prefetch_l2_2d(const CUtensorMap *map, int x, int y) {
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y)
                 : "memory");
}

// Prefetch `bytes` (a multiple of 16) of global memory at a 16-byte-aligned
// address into L2.  Safe before a programmatic-dependency wait: L2 is the
// point of coherence, so a later write by the previous kernel updates the
// prefetched lines.
__device__ __forceinline__ void bulk_prefetch_l2(const void *src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(src)),
                 "r"(bytes)
                 : "memory");
}

// Host: raise a kernel's dynamic shared-memory limit once per device (the
// attribute belongs to the current context, so each device needs its own
// call); `done` is the caller's per-kernel bitmask of devices already set.
inline cudaError_t set_smem_limit_once(const void *kernel, int bytes, std::atomic<uint64_t> &done) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_acq_rel);
    return e;
}

// Host: encode a 2-D tiled tensor map (row-major [dim1][dim0] of `dtype`,
// row pitch `stride1_bytes`, box [box1][box0], no swizzle, zero fill out of
// bounds).  The driver function is looked up once through the runtime.
inline cudaError_t encode_tmap_2d(CUtensorMap *map, const void *base, CUtensorMapDataType dtype,
                                  uint64_t dim0, uint64_t dim1, uint64_t stride1_bytes,
                                  uint32_t box0, uint32_t box1,
                                  CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_NONE) {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (fn == nullptr) {
        cudaDriverEntryPointQueryResult q;
        void *p = nullptr;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                                         cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || p == nullptr)
            return e != cudaSuccess ? e : cudaErrorNotSupported;
        fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    const cuuint64_t dims[2] = {dim0, dim1};
    const cuuint64_t strides[1] = {stride1_bytes};
    const cuuint32_t box[2] = {box0, box1};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, dtype, 2, const_cast<void *>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// ------------------------------------------------------------------ cluster
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_nctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}
// Full cluster barrier (every thread of every CTA of the cluster arrives).
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}
__device__ __forceinline__ float ld_dsmem_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

// --------------------------------------------------------------- warp MMA
// D = A * B + C, m16n8k16, A row-major f16, B column-major f16, fp32 accum.
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                              uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Named barrier over `nthreads` threads (a multiple of 32).
__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Pairs of fp32 values in one 64-bit register: sm_100-family GPUs issue
// add / sub / fma on .f32x2 operands once for both lanes, each lane rounded
// exactly like the scalar instruction (IEEE, round to nearest even).
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
    return r;
}
// (a & b) | c in one LOP3.
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
    return r;
}

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b16) {
    return __uint_as_float(b16 << 16);
}

// Two E4M3 codes (low byte first) -> their values as a binary16 pair, exactly.
__device__ __forceinline__ uint32_t e4m3x2_to_h2(uint32_t two_codes) {
    // the packed conversion (exact: every E4M3 value is a binary16 value), its
    // 32-bit result used as is
    uint32_t r;
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, lo;\n\t}"
        : "=r"(r)
        : "r"(two_codes));
    return r;
}

}  // namespace qmm
