// quant_act.cu -- per-token activation quantizer (HBM-bound).
//
// One CTA per row.  Each thread owns one 32-element chunk of the row (two
// chunks for rows longer than 32768): four 16-byte loads of bf16, widened to
// fp32 in registers.  A 128-block of the row spans four neighbouring lanes,
// so the Walsh-Hadamard butterfly runs its strides 1..16 inside a thread and
// strides 32 and 64 as lane exchanges (xor 1, xor 2), in the fixed order
// 1, 2, 4, ..., 64 with explicitly rounded fp32 add/sub (no contraction),
// then one multiply by fp32(1/sqrt(128)).  The row's absmax is a warp-shuffle
// max plus one shared-memory step; codes are written as two 16-byte stores
// per chunk.  Reads 2 B and writes 1 B per element, plus a 4 B scale per row.
//
// What it computes follows the "CLEF Calibrated INT8 ConvRot" model card
// (note under the latency table: activations are rotated and quantized to
// INT8 before the integer GEMMs; the rotation is read as the block-128
// Walsh-Hadamard transform) and the "clef-flash-FP8" model card
// (Quantization table: FP8 activations, per token, dynamic).
#include <cstdint>
#include <cuda_runtime.h>

#include "clef_kernels.h"

namespace clef {

namespace {

constexpr unsigned kFull = 0xFFFFFFFFu;

__device__ __forceinline__ float hadamard_c() { return __uint_as_float(0x3DB504F3u); }

// Packed fp32 pairs (sm_100 family): each lane of add/sub/mul/fma.rn.f32x2 is
// the IEEE round-to-nearest-even operation on that lane alone, so results are
// bit-identical to the scalar operations while issuing half as many.
__device__ __forceinline__ uint64_t f2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void unf2(uint64_t p, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(p));
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t sub2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

// Rotate this thread's 32 values as part of a 128-block spread over lanes
// (lane & 3) = 0..3 holding block positions 32*(lane & 3) + j.  The values are
// held as pairs p[k] = (v[k], v[k+16]): strides 1..8 pair p[k] with p[k+h] in
// both halves at once, stride 16 is the pair's own two halves, and strides 32
// and 64 exchange with lanes xor 1 and xor 2.
__device__ __forceinline__ void wht128_lanes(float (&v)[32], int lane) {
    uint64_t p[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) p[k] = f2(v[k], v[k + 16]);
#pragma unroll
    for (int h = 1; h < 16; h <<= 1) {
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            if ((k & h) == 0) {
                const uint64_t a = p[k], b = p[k + h];
                p[k] = add2(a, b);
                p[k + h] = sub2(a, b);
            }
        }
    }
#pragma unroll
    for (int k = 0; k < 16; ++k) {   // stride 16
        float a, b;
        unf2(p[k], a, b);
        v[k] = __fadd_rn(a, b);
        v[k + 16] = __fsub_rn(a, b);
    }
#pragma unroll
    for (int s = 1; s <= 2; s <<= 1) {   // strides 32 and 64
        // The lane holding index i computes v[i] + v[i+h]; its partner holding
        // i+h computes v[i] - v[i+h].  Both are one fma with an exact +-1
        // product, so each is the single rounded add or subtract itself.
        const float sg = (lane & s) ? -1.0f : 1.0f;
        const uint64_t sgn = f2(sg, sg);
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            const float oa = __shfl_xor_sync(kFull, v[k], s);
            const float ob = __shfl_xor_sync(kFull, v[k + 16], s);
            const uint64_t r = fma2(sgn, f2(v[k], v[k + 16]), f2(oa, ob));
            unf2(r, v[k], v[k + 16]);
        }
    }
    const float c = hadamard_c();
    const uint64_t c2 = f2(c, c);
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        const uint64_t r = mul2(f2(v[k], v[k + 16]), c2);
        unf2(r, v[k], v[k + 16]);
    }
}

__device__ __forceinline__ void load_chunk(const uint16_t *p, float (&v)[32]) {
    const uint4 *p4 = reinterpret_cast<const uint4 *>(p);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint4 w = __ldg(p4 + i);
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            v[8 * i + 2 * k] = __uint_as_float(ws[k] << 16);
            v[8 * i + 2 * k + 1] = __uint_as_float(ws[k] & 0xFFFF0000u);
        }
    }
}

// Four int32 codes (each already within [-127, 127]) packed as bytes q0..q3,
// two conversions with saturation: hi = {q2, q3}, then {q0, q1} below it.
__device__ __forceinline__ uint32_t pack_s8x4(int q0, int q1, int q2, int q3) {
    uint32_t hi, w;
    asm("cvt.pack.sat.s8.s32.b32 %0, %1, %2, %3;" : "=r"(hi) : "r"(q3), "r"(q2), "r"(0));
    asm("cvt.pack.sat.s8.s32.b32 %0, %1, %2, %3;" : "=r"(w) : "r"(q1), "r"(q0), "r"(hi));
    return w;
}

__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// MAXT / MINB: launch bounds.  Rows of up to 18,432 elements (576 threads)
// are compiled for two resident CTAs per SM, so two rows stream at once.
template <int MODE, int C, int MAXT, int MINB>
__global__ void __launch_bounds__(MAXT, MINB) quant_act_kernel(const uint16_t *__restrict__ x,
                                                         int64_t K, int64_t ldx,
                                                         uint8_t *__restrict__ q,
                                                         float *__restrict__ scale) {
    constexpr bool kRotate = (MODE == kActInt8H128 || MODE == kActFp8H128);
    constexpr bool kInt8 = (MODE == kActInt8H128);
    __shared__ float red[32];

    const int64_t m = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nchunk = (int)(K >> 5);
    const uint16_t *xr = x + m * ldx;

    float v[C][32];
    float amax = 0.0f;
#pragma unroll
    for (int c = 0; c < C; ++c) {
        const int ch = tid + c * blockDim.x;
        if (ch < nchunk) {
            load_chunk(xr + 32 * (int64_t)ch, v[c]);
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) v[c][j] = 0.0f;
        }
        // Whole 128-blocks are active or inactive together (nchunk % 4 == 0
        // in the rotated modes), and every lane of the warp exists.
        if (kRotate) wht128_lanes(v[c], lane);
#pragma unroll
        for (int j = 0; j < 32; ++j) amax = fmaxf(amax, fabsf(v[c][j]));
    }
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, s));
    if (lane == 0) red[warp] = amax;
    __syncthreads();
    if (warp == 0) {
        const int nw = (int)(blockDim.x >> 5);
        float a = lane < nw ? red[lane] : 0.0f;
#pragma unroll
        for (int s = 16; s > 0; s >>= 1) a = fmaxf(a, __shfl_xor_sync(kFull, a, s));
        if (lane == 0) red[0] = a;
    }
    __syncthreads();
    amax = red[0];

    const float qmax = kInt8 ? 127.0f : 448.0f;
    const bool zero_row = !(amax > 0.0f);
    const float r = zero_row ? 0.0f : __fdiv_rn(qmax, amax);  // zero row: every v * 0 = 0
    if (tid == 0) scale[m] = zero_row ? 0.0f : __fdiv_rn(amax, qmax);

    uint8_t *qr = q + m * K;
#pragma unroll
    for (int c = 0; c < C; ++c) {
        const int ch = tid + c * blockDim.x;
        if (ch >= nchunk) continue;
        uint32_t w[8];
        if (kInt8) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                // |v * r| <= 127 * (1 + 2^-23) for every v of the row, so the
                // round-half-even conversion never leaves [-127, 127].
                const uint64_t r2 = f2(r, r);
                float u[4];
                unf2(mul2(f2(v[c][4 * i], v[c][4 * i + 1]), r2), u[0], u[1]);
                unf2(mul2(f2(v[c][4 * i + 2], v[c][4 * i + 3]), r2), u[2], u[3]);
                w[i] = pack_s8x4(__float2int_rn(u[0]), __float2int_rn(u[1]), __float2int_rn(u[2]),
                                 __float2int_rn(u[3]));
            }
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                if (zero_row) {
                    w[i] = 0u;
                } else {
                    const float *u = &v[c][4 * i];
                    w[i] = e4m3x2(__fmul_rn(u[0], r), __fmul_rn(u[1], r)) |
                           (e4m3x2(__fmul_rn(u[2], r), __fmul_rn(u[3], r)) << 16);
                }
            }
        }
        uint4 *dst = reinterpret_cast<uint4 *>(qr + 32 * (int64_t)ch);
        dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
        dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
    }
}

template <int MODE>
cudaError_t launch_mode(const uint16_t *x, int64_t M, int64_t K, int64_t ldx, uint8_t *q,
                        float *scale, cudaStream_t st) {
    const int64_t nchunk = K / 32;
    if (nchunk <= 576) {
        const int T = (int)((nchunk + 31) / 32 * 32);
        quant_act_kernel<MODE, 1, 576, 2><<<(unsigned)M, T, 0, st>>>(x, K, ldx, q, scale);
    } else if (nchunk <= 1024) {
        const int T = (int)((nchunk + 31) / 32 * 32);
        quant_act_kernel<MODE, 1, 1024, 1><<<(unsigned)M, T, 0, st>>>(x, K, ldx, q, scale);
    } else {
        const int64_t per = (nchunk + 1) / 2;
        const int T = (int)((per + 31) / 32 * 32);
        quant_act_kernel<MODE, 2, 1024, 1><<<(unsigned)M, T, 0, st>>>(x, K, ldx, q, scale);
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_quant_act(int mode, const uint16_t *x, int64_t M, int64_t K, int64_t ldx,
                             uint8_t *q, float *scale, cudaStream_t st) {
    switch (mode) {
        case kActInt8H128: return launch_mode<kActInt8H128>(x, M, K, ldx, q, scale, st);
        case kActFp8: return launch_mode<kActFp8>(x, M, K, ldx, q, scale, st);
        case kActFp8H128: return launch_mode<kActFp8H128>(x, M, K, ldx, q, scale, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace clef
