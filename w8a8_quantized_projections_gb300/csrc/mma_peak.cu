// mma_peak.cu -- dense tensor-core rate microbenchmarks: the denominators of
// the GEMMs' roofline fractions, measured on the device the library runs on.
//
// Three instruction routes:
//   kind 0  tcgen05.mma.cta_group::2.kind::f16, bf16 operands, fp32 accumulator
//           (the route of the INT8 GEMMs, which multiply int8 codes exactly as
//           fp16, and of the LoRA products)
//   kind 1  tcgen05.mma.cta_group::2.kind::f8f6f4, e4m3 operands, fp32
//           accumulator (the FP8 GEMMs)
//   kind 2  mma.sync.m16n8k32 s8 x s8 -> s32 (the legacy integer tensor path;
//           sm_103a has no tcgen05 integer MMA)
//
// The tcgen05 kernels run one CTA pair per two SMs, each pair issuing
// 256 x 256 MMAs from one elected thread over two shared-memory operand stages
// (the 128-byte swizzled K-major tiles the GEMMs use) into two TMEM
// accumulators in turn, with no copies: the tensor pipe's issue and
// operand-read rate alone.  The mma.sync kernel keeps its operands in
// registers and runs independent accumulator chains in every warp.
// Each kind is timed with CUDA events over one launch after a warm-up launch;
// the rate is the multiply-add count x 2 over that time.
#include <cstdint>
#include <cstdio>

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/clef.h"
#include "clef_kernels.h"
#include "clef_ptx.cuh"

namespace clef {
namespace {

constexpr int kPeakStage = 128 * 128;            // one operand tile: 128 rows of 128 bytes
// A and B of two stages (64 KB, 1024-aligned) are used; the request is large
// enough that no two CTAs share an SM, so each CTA's 512-column TMEM
// allocation never waits for another CTA's
constexpr int kPeakSmem = 160 * 1024;
constexpr int kPeakThreads = 128;

// Where the mma.sync kernel's folded result would go (it never does; the
// store only keeps the compiler from dropping the work).
__device__ int g_peak_sink[256];

__device__ __forceinline__ uint32_t peak_cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void peak_cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
                 ::: "memory");
}

template <int KIND>
__device__ __forceinline__ void peak_mma2(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    if constexpr (KIND == 1)
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}\n"
            ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(acc) : "memory");
    else
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}\n"
            ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(acc) : "memory");
}

// Every operand byte is a small finite value in either format: 0x38 is 1.0 in
// e4m3 and, paired, 0x3838 is 4.4e-5 in bf16.
template <int KIND>
__global__ void __launch_bounds__(kPeakThreads, 1) mma_peak_kernel(int iters, unsigned int *status,
                                                                   uint64_t limit_ns) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t done;
    __shared__ uint32_t tmem_slot;
    const uint32_t base = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + (((base + 1023u) & ~1023u) - base);
    const int warp = threadIdx.x >> 5;
    const uint32_t rank = peak_cluster_rank();

    for (int i = threadIdx.x; i < 4 * kPeakStage / 16; i += kPeakThreads)
        reinterpret_cast<uint4 *>(smem)[i] = make_uint4(0x38383838u, 0x38383838u, 0x38383838u, 0x38383838u);
    fence_proxy_async_smem();
    if (threadIdx.x == 0) {
        mbar_init(&done, 1);
        fence_barrier_init();
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(smem_u32(&tmem_slot)), "r"(512) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    peak_cluster_sync();
    tc_fence_after();

    if (rank == 0 && threadIdx.x == 32) {
        // the pair's accumulators: M = 256 (128 rows per CTA), N = 256
        constexpr uint32_t idesc = idesc_f32acc(KIND == 1 ? 0u : 1u, KIND == 1 ? 0u : 1u, 256, 256);
        const uint32_t tmem = tmem_slot;
        const uint32_t s0 = smem_u32(smem);
        for (int it = 0; it < iters; ++it) {
            const uint32_t a = s0 + (uint32_t)(it & 1) * (2 * kPeakStage);
            const uint32_t b = a + kPeakStage;
            const uint32_t d = tmem + (uint32_t)(it & 1) * 256u;
#pragma unroll
            for (int k = 0; k < 4; ++k)
                peak_mma2<KIND>(d, sdesc_sw128(a + 32 * k), sdesc_sw128(b + 32 * k), idesc, k > 0 ? 1u : 0u);
        }
        // both CTAs' barriers: the peer's operands are read until the last MMA ends
        asm volatile(
            "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
            " [%0], %1;" ::"r"(smem_u32(&done)), "h"((uint16_t)3) : "memory");
    }
    if (threadIdx.x == 0) {
        const uint32_t a = smem_u32(&done);
        const uint64_t t0 = globaltimer_ns();
        for (uint32_t it = 0;; ++it) {
            uint32_t ok;
            asm volatile(
                "{\n\t.reg .pred p;\n\t"
                "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
                "selp.u32 %0, 1, 0, p;\n\t}\n"
                : "=r"(ok) : "r"(a), "r"(0u) : "memory");
            if (ok) break;
            if ((it & 63u) == 63u && globaltimer_ns() - t0 > limit_ns) {
                record_status(status, kStatusTimeout | (kSiteDrain << 8));
                break;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    peak_cluster_sync();
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_slot), "r"(512)
                     : "memory");
    }
}

// mma.sync s8: eight independent m16n8k32 accumulator chains per warp on
// register operands; the result is folded into one word per thread and
// stored only when impossible, so the compiler keeps the work.
__global__ void __launch_bounds__(256) mma_s8_peak_kernel(int iters) {
    uint32_t a0 = 0x01020304u ^ threadIdx.x, a1 = 0x05060708u, a2 = 0x090A0B0Cu, a3 = 0x0D0E0F10u;
    uint32_t b0 = 0x11121314u, b1 = 0x15161718u ^ blockIdx.x;
    int acc[8][4] = {};
#pragma unroll 1
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int c = 0; c < 8; ++c)
            asm volatile(
                "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                "{%0,%1,%2,%3};"
                : "+r"(acc[c][0]), "+r"(acc[c][1]), "+r"(acc[c][2]), "+r"(acc[c][3])
                : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
    int f = 0;
#pragma unroll
    for (int c = 0; c < 8; ++c) f ^= acc[c][0] ^ acc[c][1] ^ acc[c][2] ^ acc[c][3];
    if (f == 0x7FFFFFFF) g_peak_sink[threadIdx.x] = f;
}

// Launches as many CTA pairs as can be resident at once (*pairs is set to
// that count), so that every pair runs in the one wave that is timed.
template <int KIND>
cudaError_t launch_tc_peak(int num_sms, int *pairs, int iters, unsigned int *status, uint64_t limit_ns,
                           cudaStream_t st) {
    auto kern = mma_peak_kernel<KIND>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kPeakSmem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(2 * (num_sms / 2), 1, 1);
    cfg.blockDim = dim3(kPeakThreads, 1, 1);
    cfg.dynamicSmemBytes = kPeakSmem;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
    if (e != cudaSuccess) return e;
    *pairs = n < num_sms / 2 ? n : num_sms / 2;
    if (*pairs <= 0) return cudaErrorInvalidConfiguration;
    cfg.gridDim = dim3(2 * *pairs, 1, 1);
    return cudaLaunchKernelEx(&cfg, kern, iters, status, limit_ns);
}

}  // namespace
}  // namespace clef

using namespace clef;

extern "C" int clef_mma_peak(int kind, int64_t iters, double *tflops) {
    if (!tflops) {
        internal_set_error("invalid argument: null pointer");
        return CLEF_ERR_INVALID_ARG;
    }
    if (kind < 0 || kind > 2 || iters <= 0 || iters > (1 << 24)) {
        internal_set_error("invalid argument: kind must be 0..2 and iters in (0, 2^24]");
        return CLEF_ERR_INVALID_ARG;
    }
    int num_sms = 0;
    unsigned int *status = nullptr;
    int rc = internal_device(&num_sms, &status);
    if (rc) return rc;
    cudaStream_t st = nullptr;
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    cudaError_t e = cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreate(&e0);
    if (e == cudaSuccess) e = cudaEventCreate(&e1);
    int pairs = 0;
    const int s8_blocks = num_sms * 4;
    const uint64_t limit = 10000000000ull;   // 10 s: far beyond any launch here
    auto run = [&](int n) -> cudaError_t {
        if (kind == 0) return launch_tc_peak<0>(num_sms, &pairs, n, status, limit, st);
        if (kind == 1) return launch_tc_peak<1>(num_sms, &pairs, n, status, limit, st);
        mma_s8_peak_kernel<<<s8_blocks, 256, 0, st>>>(n);
        return cudaGetLastError();
    };
    float ms = 0.0f;
    if (e == cudaSuccess) e = run((int)(iters < 64 ? iters : 64));   // warm-up
    if (e == cudaSuccess) e = cudaEventRecord(e0, st);
    if (e == cudaSuccess) e = run((int)iters);
    if (e == cudaSuccess) e = cudaEventRecord(e1, st);
    if (e == cudaSuccess) e = cudaEventSynchronize(e1);
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, e0, e1);
    if (e0) cudaEventDestroy(e0);
    if (e1) cudaEventDestroy(e1);
    if (st) cudaStreamDestroy(st);
    if (e != cudaSuccess) return internal_cuda_error(e, "mma peak microbenchmark");
    double flops;
    if (kind == 2)
        flops = 2.0 * 16 * 8 * 32 * 8.0 * (double)iters * (double)s8_blocks * 8.0;   // 8 warps x 8 chains
    else
        flops = 2.0 * 256 * 256 * (kind == 1 ? 128 : 64) * (double)iters * (double)pairs;
    *tflops = flops / (ms * 1e-3) / 1e12;
    return CLEF_OK;
}
