// copy_sm.cu -- clef_copy_sm: a byte copy whose loads and stores are issued
// by a few CTAs instead of a copy engine.
//
// A step that takes its activations from host memory moves them over the
// CPU-GPU link while the previous step computes.  Copy-engine transfers from
// page-locked host memory were measured to stall for 20-180 ms, on some GB300
// boxes about every half second (with or without other work running, in
// whole or in 16-64 MB pieces, on one stream or two) and on others rarely;
// loads issued by SMs over the same link ran at the same 211 GB/s without a
// stall on every box tried.  The copy therefore runs as
// a kernel on a few SMs, beside the compute: the compute launches leave those
// SMs free when the caller sets an SM budget (clef_set_sm_budget), because a
// persistent GEMM CTA takes a whole SM and no copy CTA could be resident
// beside it.
//
// Addresses are whatever the device can read or write: device memory, or
// page-locked host memory (allocated or registered with CUDA), reached
// through its device mapping.  Other host memory is refused on the host,
// unless the device reads pageable memory directly.  The CTAs come in
// clusters of two where their count is even, so that they occupy whole SM
// pairs and leave the pairs the GEMMs are launched on.
#include <cstdint>

#include <cuda_runtime.h>

#include "../../include/clef.h"
#include "clef_kernels.h"

namespace clef {

namespace {

constexpr int kCopyThreads = 1024;
constexpr int kCopyUnroll = 8;   // 16-byte loads in flight per thread
constexpr int kCopyMaxCtas = 64;

// Grid-stride over 16-byte words: a warp's loads and stores cover 512
// contiguous bytes each, and every thread keeps kCopyUnroll loads in flight
// (4 CTAs: 512 KB, about what the link's latency needs at full rate).  Loads
// and stores are streaming (the data passes through once).
__global__ void __launch_bounds__(kCopyThreads, 1)
copy_sm_kernel(uint4 *__restrict__ dst, const uint4 *__restrict__ src, int64_t n16) {
    const int64_t stride = (int64_t)gridDim.x * kCopyThreads;
    int64_t i = (int64_t)blockIdx.x * kCopyThreads + threadIdx.x;
    for (; i + (kCopyUnroll - 1) * stride < n16; i += kCopyUnroll * stride) {
        uint4 v[kCopyUnroll];
#pragma unroll
        for (int u = 0; u < kCopyUnroll; ++u) v[u] = __ldcs(src + i + u * stride);
#pragma unroll
        for (int u = 0; u < kCopyUnroll; ++u) __stcs(dst + i + u * stride, v[u]);
    }
    for (; i < n16; i += stride) __stcs(dst + i, __ldcs(src + i));
}

int fail(const char *msg) {
    internal_set_error(msg);
    return CLEF_ERR_INVALID_ARG;
}

// The address the kernel dereferences for p: device and managed memory as
// they are, page-locked host memory through its device mapping, and other
// host memory only where the device reads pageable memory directly.  nullptr
// where the device cannot reach p (the call is then refused instead of
// faulting on the GPU).
const void *device_address(const void *p, bool pageable_ok) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();   // a failed query leaves its error behind: clear it
        return pageable_ok ? p : nullptr;
    }
    if (at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged) return p;
    if (at.type == cudaMemoryTypeHost) return at.devicePointer;
    return pageable_ok ? p : nullptr;
}

}  // namespace

}  // namespace clef

using namespace clef;

extern "C" int clef_copy_sm(void *dst, const void *src, int64_t bytes, int ctas, void *stream) {
    if (bytes < 0 || bytes % 16 != 0) return fail("invalid argument: bytes must be a non-negative multiple of 16");
    if (ctas < 1 || ctas > kCopyMaxCtas) return fail("invalid argument: ctas must be in 1..64");
    if (bytes == 0) return CLEF_OK;
    if (!dst || !src) return fail("invalid argument: null pointer");
    if ((reinterpret_cast<uintptr_t>(dst) | reinterpret_cast<uintptr_t>(src)) & 15u)
        return fail("invalid argument: dst and src must be 16-byte aligned");
    const uintptr_t d0 = reinterpret_cast<uintptr_t>(dst), s0 = reinterpret_cast<uintptr_t>(src);
    if (d0 < s0 + (uint64_t)bytes && s0 < d0 + (uint64_t)bytes)
        return fail("invalid argument: the source and destination ranges overlap");
    int num_sms = 0;
    unsigned int *status = nullptr;
    int rc = internal_device(&num_sms, &status);   // device checks (sm_103) first
    if (rc) return rc;
    int dev = 0, pageable = 0;
    if (cudaGetDevice(&dev) == cudaSuccess)
        cudaDeviceGetAttribute(&pageable, cudaDevAttrPageableMemoryAccess, dev);
    const void *dsrc = device_address(src, pageable != 0);
    void *ddst = const_cast<void *>(device_address(dst, pageable != 0));
    if (!dsrc || !ddst)
        return fail("invalid argument: host memory must be page-locked (cudaHostAlloc or cudaHostRegister)");
    if ((reinterpret_cast<uintptr_t>(ddst) | reinterpret_cast<uintptr_t>(dsrc)) & 15u)
        return fail("invalid argument: the device addresses must be 16-byte aligned");
    const int64_t n16 = bytes / 16;
    // no more CTAs than 16-byte words per thread-round, and clusters of two
    // where the count allows
    int grid = ctas;
    if ((int64_t)grid * kCopyThreads > n16) grid = (int)((n16 + kCopyThreads - 1) / kCopyThreads);
    const int cluster = (grid % 2 == 0) ? 2 : 1;
    cudaError_t e = launch_kernel(copy_sm_kernel, dim3(grid), dim3(kCopyThreads), 0,
                                  static_cast<cudaStream_t>(stream), cluster, false, static_cast<uint4 *>(ddst),
                                  static_cast<const uint4 *>(dsrc), n16);
    if (e != cudaSuccess) return internal_cuda_error(e, "copy launch");
    return CLEF_OK;
}
