// swiglu.cu -- the unfused MLP product (fuse_mlp off in the "Loading CLEF
// INT8" usage notes): gate and up values already rounded to bf16 and stored
// side by side, h = bf16(silu(g) * u).  HBM-bound: 16-byte loads of eight
// gate and eight up values, one 16-byte store, grid-stride over groups of 8.
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "clef_kernels.h"
#include "clef_ptx.cuh"

namespace clef {

namespace {

__device__ __forceinline__ float lo16(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi16(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// silu(g) * u = g / (1 + exp(-g)) * u in fp32 with the hardware exp2 and
// reciprocal approximations (a few fp32 ulps; the bf16 result stays within
// one ulp of the correctly rounded value).  Denominators above 2^126 are
// scaled by 2^-64 with the numerator, exactly, to keep the fast quotient in
// its accurate range.  The fused LoRA gate/up kernel uses the same sequence.
__device__ __forceinline__ float silu_mul(float g, float u) {
    const float d = __fadd_rn(1.0f, __expf(-g));
    const float sc = d > 0x1p126f ? 0x1p-64f : 1.0f;
    return __fmul_rn(__fdividef(g * sc, d * sc), u);
}

__device__ __forceinline__ uint32_t pack(float lo, float hi) {
    __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&p);
}

__global__ void __launch_bounds__(256) swiglu_bf16_kernel(const uint16_t *__restrict__ y_gu,
                                                          int64_t M, int64_t N, int64_t ldg,
                                                          uint16_t *__restrict__ h, int64_t ldh) {
    const int64_t groups_per_row = N / 8;
    const int64_t total = M * groups_per_row;
    pdl_wait();
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t m = i / groups_per_row, n = (i - m * groups_per_row) * 8;
        const uint4 g = __ldg(reinterpret_cast<const uint4 *>(y_gu + m * ldg + n));
        const uint4 u = __ldg(reinterpret_cast<const uint4 *>(y_gu + m * ldg + N + n));
        const uint32_t gw[4] = {g.x, g.y, g.z, g.w}, uw[4] = {u.x, u.y, u.z, u.w};
        uint32_t o[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
            o[k] = pack(silu_mul(lo16(gw[k]), lo16(uw[k])), silu_mul(hi16(gw[k]), hi16(uw[k])));
        *reinterpret_cast<uint4 *>(h + m * ldh + n) = make_uint4(o[0], o[1], o[2], o[3]);
    }
    pdl_launch_dependents();
}

}  // namespace

cudaError_t launch_swiglu_bf16(const uint16_t *y_gu, int64_t M, int64_t N, int64_t ldg,
                               uint16_t *h, int64_t ldh, cudaStream_t st) {
    const int64_t total = M * (N / 8);
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    int64_t blocks = (total + 255) / 256;
    const int64_t cap = (int64_t)sms * 8;  // 8 resident blocks of 256 threads per SM
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    return launch_kernel(swiglu_bf16_kernel, dim3((unsigned)blocks), dim3(256), 0, st, 1, true, y_gu, M, N, ldg, h,
                         ldh);
}

}  // namespace clef
