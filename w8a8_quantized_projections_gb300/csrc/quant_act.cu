// quant_act.cu -- per-token activation quantizer (HBM-bound).
//
// Two kernels compute the same thing.  The staged kernel (rows whose length
// is a multiple of 64 and fits the shared-memory ring, which covers every
// projection width of the workloads) is persistent: each CTA owns a ring of
// row slots in shared memory that TMA fills several rows ahead (128-byte
// swizzled, so that the threads' 16-byte reads are free of bank conflicts),
// and several CTAs share an SM, so HBM sees a steady stream of row reads
// while earlier rows are rotated and coded.  The fallback kernel runs one
// CTA per row with direct 16-byte loads.
//
// In both, each thread owns one 32-element chunk of the row (two chunks for
// rows longer than 32768 in the fallback; the staged kernel gives rows of
// 8,192 to 12,288 elements 64 per thread): 16-byte pieces of bf16, widened
// to fp32 in registers.  A 128-block of the row spans four (two) neighbouring
// lanes, so the Walsh-Hadamard butterfly runs its strides 1..16 (1..32) inside
// a thread and the rest as lane exchanges (xor 1, xor 2), in the fixed order
// 1, 2, 4, ..., 64 with explicitly rounded fp32 add/sub (no contraction),
// then one multiply by fp32(1/sqrt(128)).  The row's absmax is a warp
// reduction (redux.sync on the bit patterns) per warp, then one over the
// warps' partials through shared memory; codes are written as 16-byte stores.
// Reads 2 B and writes 1 B per element, plus a 4 B scale per row.
//
// What it computes follows the "CLEF Calibrated INT8 ConvRot" model card
// (note under the latency table: activations are rotated and quantized to
// INT8 before the integer GEMMs; the rotation is read as the block-128
// Walsh-Hadamard transform) and the "clef-flash-FP8" model card
// (Quantization table: FP8 activations, per token, dynamic).
#include <cstdint>
#include <cuda_runtime.h>

#include "clef_kernels.h"
#include "clef_ptx.cuh"

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

// The same rotation on E = 2 NP consecutive values (E = 32 or 64) held as NP
// natural pairs p[i] = (v[2i], v[2i+1]) (the load's bf16 order); a 128-block
// spans 128 / E neighbouring lanes.  Stride 1 pairs the two halves of each
// pair, strides 2 .. E/2 pair p[i] with p[i + h/2] lane-wise, and the strides
// E .. 64 exchange whole pairs with lanes xor 1, xor 2.  Each output is the
// same fp32 add or subtract of the same two values in the same stage order as
// wht128_lanes.
template <int NP, bool kStride1Done>
__device__ __forceinline__ void wht128_pairs(uint64_t (&p)[NP], int lane) {
    static_assert(NP == 16 || NP == 32, "32 or 64 values per thread");
#pragma unroll
    for (int i = 0; i < NP; ++i) {   // stride 1
        if (kStride1Done) break;
        float a, b;
        unf2(p[i], a, b);
        p[i] = f2(__fadd_rn(a, b), __fsub_rn(a, b));
    }
#pragma unroll
    for (int hp = 1; hp < NP; hp <<= 1) {   // strides 2 .. E/2
#pragma unroll
        for (int k = 0; k < NP; ++k) {
            if ((k & hp) == 0) {
                const uint64_t a = p[k], b = p[k + hp];
                p[k] = add2(a, b);
                p[k + hp] = sub2(a, b);
            }
        }
    }
#pragma unroll
    for (int s = 1; 2 * NP * s <= 64; s <<= 1) {   // strides E .. 64 across lanes
        const float sg = (lane & s) ? -1.0f : 1.0f;
        const uint64_t sgn = f2(sg, sg);
#pragma unroll
        for (int k = 0; k < NP; ++k) {
            float a, b;
            unf2(p[k], a, b);
            const float oa = __shfl_xor_sync(kFull, a, s);
            const float ob = __shfl_xor_sync(kFull, b, s);
            p[k] = fma2(sgn, p[k], f2(oa, ob));
        }
    }
    const float c = hadamard_c();
    const uint64_t c2 = f2(c, c);
#pragma unroll
    for (int k = 0; k < NP; ++k) p[k] = mul2(p[k], c2);
}

// The stride-1 butterfly of the bf16 pair (v0, v1) held in w (v0 in the low
// half), straight from bf16 by mixed-precision add/sub (each the single
// rounded fp32 operation on the widened values): (v0 + v1, v1 - v0).  The
// second lane is the negated difference; every later stage pairs such lanes
// only with each other, and fp32 add, subtract and multiply commute with
// negation except for the sign of an exact zero, so the whole odd lane comes
// out negated in magnitude-exact form and the codes take the multiplier -r
// there.  (INT8 codes do not see the sign of a zero.)
__device__ __forceinline__ uint64_t stride1_bf16(uint32_t w) {
    const float v0 = __uint_as_float(w << 16);
    float s, d;
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
        "add.rn.f32.bf16 %0, h, %3;\n\tsub.rn.f32.bf16 %1, h, %3;\n\t}"
        : "=f"(s), "=f"(d) : "r"(w), "f"(v0));
    return f2(s, d);
}

// Warp-wide maximum of non-negative finite-or-infinite floats: their bit
// patterns order like unsigned integers.
__device__ __forceinline__ float warp_max_nonneg(float a) {
    uint32_t m;
    asm volatile("redux.sync.max.u32 %0, %1, 0xffffffff;" : "=r"(m) : "r"(__float_as_uint(a)));
    return __uint_as_float(m);
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

// Codes of one 32-element chunk (r = qmax / amax of the row), written as two
// 16-byte stores.
// kClamp (static scales, INT8): values may exceed the code range; the
// saturating pack gives -128 below it, raised to -127 by a signed-byte max.
template <bool kInt8, bool kClamp = false>
__device__ __forceinline__ void store_codes(const float (&v)[32], float r, bool zero_row,
                                            uint8_t *dst8) {
    uint32_t w[8];
    if (kInt8) {
        const uint64_t r2 = f2(r, r);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            // |v * r| <= 127 * (1 + 2^-23) for every v of the row, so the
            // round-half-even conversion never leaves [-127, 127].
            float u[4];
            unf2(mul2(f2(v[4 * i], v[4 * i + 1]), r2), u[0], u[1]);
            unf2(mul2(f2(v[4 * i + 2], v[4 * i + 3]), r2), u[2], u[3]);
            w[i] = pack_s8x4(__float2int_rn(u[0]), __float2int_rn(u[1]), __float2int_rn(u[2]),
                             __float2int_rn(u[3]));
            if (kClamp) w[i] = __vmaxs4(w[i], 0x81818181u);
        }
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (zero_row) {
                w[i] = 0u;
            } else {
                const float *u = &v[4 * i];
                w[i] = e4m3x2(__fmul_rn(u[0], r), __fmul_rn(u[1], r)) |
                       (e4m3x2(__fmul_rn(u[2], r), __fmul_rn(u[3], r)) << 16);
            }
        }
    }
    uint4 *dst = reinterpret_cast<uint4 *>(dst8);
    dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
    dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
}

// Codes of 32 values held as natural pairs (as store_codes).
template <bool kInt8, bool kClamp = false>
__device__ __forceinline__ void store_codes_pairs(const uint64_t *p, uint64_t r2, bool zero_row,
                                                  uint8_t *dst8) {
    uint32_t w[8];
    if (kInt8) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            float u[4];
            unf2(mul2(p[2 * i], r2), u[0], u[1]);
            unf2(mul2(p[2 * i + 1], r2), u[2], u[3]);
            w[i] = pack_s8x4(__float2int_rn(u[0]), __float2int_rn(u[1]), __float2int_rn(u[2]),
                             __float2int_rn(u[3]));
            if (kClamp) w[i] = __vmaxs4(w[i], 0x81818181u);
        }
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (zero_row) {
                w[i] = 0u;
            } else {
                float u[4];
                unf2(mul2(p[2 * i], r2), u[0], u[1]);
                unf2(mul2(p[2 * i + 1], r2), u[2], u[3]);
                w[i] = e4m3x2(u[0], u[1]) | (e4m3x2(u[2], u[3]) << 16);
            }
        }
    }
    uint4 *dst = reinterpret_cast<uint4 *>(dst8);
    dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
    dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
}

// MAXT / MINB: launch bounds.  Rows of up to 18,432 elements (576 threads)
// are compiled for two resident CTAs per SM, so two rows stream at once.
template <int MODE, int C, int MAXT, int MINB>
__global__ void __launch_bounds__(MAXT, MINB) quant_act_kernel(const uint16_t *__restrict__ x,
                                                         int64_t K, int64_t ldx,
                                                         uint8_t *__restrict__ q,
                                                         float *__restrict__ scale,
                                                         float static_r, float static_s) {
    constexpr bool kRotate = (MODE == kActInt8H128 || MODE == kActFp8H128);
    constexpr bool kInt8 = (MODE == kActInt8H128);
    __shared__ float red[32];

    const int64_t m = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nchunk = (int)(K >> 5);
    const uint16_t *xr = x + m * ldx;
    pdl_wait();   // the row may come from the stream's previous kernel

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
    amax = warp_max_nonneg(amax);
    if (lane == 0) red[warp] = amax;
    __syncthreads();
    amax = warp_max_nonneg(lane < (int)(blockDim.x >> 5) ? red[lane] : 0.0f);

    const float qmax = kInt8 ? 127.0f : 448.0f;
    const bool stat = static_r > 0.0f;   // static scale: the row's amax is not used
    const bool zero_row = !stat && !(amax > 0.0f);
    const float r = stat ? static_r : (zero_row ? 0.0f : __fdiv_rn(qmax, amax));
    if (tid == 0) scale[m] = stat ? static_s : (zero_row ? 0.0f : __fdiv_rn(amax, qmax));

    uint8_t *qr = q + m * K;
#pragma unroll
    for (int c = 0; c < C; ++c) {
        const int ch = tid + c * blockDim.x;
        if (ch >= nchunk) continue;
        if (stat) store_codes<kInt8, kInt8>(v[c], r, false, qr + 32 * (int64_t)ch);
        else store_codes<kInt8>(v[c], r, zero_row, qr + 32 * (int64_t)ch);
    }
    pdl_launch_dependents();
}

// ---------------------------------------------------------------- staged kernel

constexpr int kMaxSlots = 8;

// 3-D tile load (row view [M][K/64][64] of bf16) into shared memory.
__device__ __forceinline__ void tma_load_3d(void *smem_dst, const CUtensorMap *m, int32_t c0,
                                            int32_t c1, int32_t c2, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];"
        ::"r"(smem_u32(smem_dst)), "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(c2),
          "r"(smem_u32(bar))
        : "memory");
}

// Persistent quantizer.  CTA b handles rows b, b + G, b + 2G, ... (G = grid
// size); slot it % nslot of its ring holds the row of iteration it.  A row
// is K/64 128-byte lines of 64 bf16, copied as nbox boxes of box_rows lines
// with the 128-byte swizzle: 16-byte unit u of line l lands at unit
// u ^ (l & 7).  Thread t owns chunk t (32 elements), the half t & 1 of line
// t >> 1, so its four pieces sit at units (4 (t & 1) + j) ^ ((t >> 1) & 7):
// every quarter-warp's eight 16-byte reads hit eight different bank groups.
// One block barrier per row: it publishes the warps' absmax (double-buffered
// by row parity) and certifies that every thread has read the slot, after
// which thread 0 refills it with the row nslot iterations ahead.
template <int MODE, int E, int MAXT, int MINB>
__global__ void __launch_bounds__(MAXT, MINB)
quant_staged_kernel(const __grid_constant__ CUtensorMap tmx, int M, int K, int nslot,
                    uint32_t slot_stride, int nbox, int box_rows, uint8_t *__restrict__ q,
                    float *__restrict__ scale, unsigned int *status, uint64_t limit_ns,
                    float static_r, float static_s) {
    constexpr bool kRotate = (MODE == kActInt8H128 || MODE == kActFp8H128);
    constexpr bool kInt8 = (MODE == kActInt8H128);
    extern __shared__ uint8_t dyn[];
    __shared__ uint64_t full[kMaxSlots];
    __shared__ float red[2][32];
    __shared__ int abort_flag;

    const uint32_t base = smem_u32(dyn);
    uint8_t *ring = dyn + (((base + 1023u) & ~1023u) - base);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nw = (int)(blockDim.x >> 5);
    const int nchunk = K / E;
    const uint32_t row_bytes = (uint32_t)K * 2u;

    if (tid == 0) {
        for (int s = 0; s < nslot; ++s) mbar_init(&full[s], 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    pdl_wait();   // the rows may come from the stream's previous kernel
    WaitCtx w;
    w.limit_ns = limit_ns;
    w.abort = &abort_flag;
    w.status = status;

    auto issue = [&](int slot, int m) {
        uint8_t *dst = ring + (uint32_t)slot * slot_stride;
        mbar_arrive_expect_tx(&full[slot], row_bytes);
        for (int b = 0; b < nbox; ++b)
            tma_load_3d(dst + (uint32_t)(b * box_rows) * 128u, &tmx, 0, b * box_rows, m, &full[slot]);
    };
    if (tid == 0) {
        tma_prefetch_desc(&tmx);
        for (int s = 0; s < nslot; ++s) {
            const int m = (int)blockIdx.x + s * (int)gridDim.x;
            if (m < M) issue(s, m);
        }
    }

    // E = 32: thread t reads half t & 1 of line t >> 1 (four 16-byte units);
    // E = 64: the whole line t (eight units).  Either way a quarter-warp's
    // eight reads of one step hit eight different bank groups.
    constexpr int kU = E / 8;   // 16-byte units per thread
    // stride 1 straight from bf16 with the odd lanes negated (INT8 only: the
    // FP8 codes keep the sign of a zero)
    constexpr bool kFold = kRotate && kInt8;
    const bool active = tid < nchunk;
    // a thread past the row's end reads line 0 (its values are left out of
    // the max and its codes are not stored)
    const uint32_t line = active ? (uint32_t)(E == 64 ? tid : tid >> 1) : 0u;
    uint32_t off[kU];
#pragma unroll
    for (int j = 0; j < kU; ++j)
        off[j] = line * 128u + (((uint32_t)((E == 64 ? 0 : (tid & 1) * 4) + j) ^ (line & 7u)) << 4);

    int it = 0, slot = 0;
    uint32_t phase = 0, src = smem_u32(ring);
    for (int m = (int)blockIdx.x; m < M; m += (int)gridDim.x, ++it) {
        mbar_wait(&full[slot], phase, w, kSiteQuantFull);
        uint64_t p[E / 2];   // the thread's E values as natural pairs (v[2i], v[2i+1])
#pragma unroll
        for (int j = 0; j < kU; ++j) {
            uint32_t a0, a1, a2, a3;
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(a0), "=r"(a1), "=r"(a2), "=r"(a3) : "r"(src + off[j]));
            const uint32_t ws[4] = {a0, a1, a2, a3};
#pragma unroll
            for (int k = 0; k < 4; ++k)
                p[4 * j + k] = kFold ? stride1_bf16(ws[k])
                                     : f2(__uint_as_float(ws[k] << 16), __uint_as_float(ws[k] & 0xFFFF0000u));
        }
        // whole 128-blocks are active or inactive together (K % 128 == 0 in
        // the rotated modes), and every lane of the warp exists
        if (kRotate) wht128_pairs<E / 2, kFold>(p, lane);
        float amax = 0.0f;
#pragma unroll
        for (int j = 0; j < E / 2; ++j) {
            float a, b;
            unf2(p[j], a, b);
            amax = fmaxf(amax, fmaxf(fabsf(a), fabsf(b)));
        }
        if (!active) amax = 0.0f;
        amax = warp_max_nonneg(amax);
        if (lane == 0) red[it & 1][warp] = amax;
        __syncthreads();
        if (abort_flag) break;
        if (tid == 0) {
            const int mn = m + nslot * (int)gridDim.x;
            if (mn < M) {
                fence_proxy_async_smem();
                issue(slot, mn);
            }
        }
        // the nw partial maxima: lane l reads partial l, one warp reduction
        amax = warp_max_nonneg(lane < nw ? red[it & 1][lane] : 0.0f);

        const float qmax = kInt8 ? 127.0f : 448.0f;
        const bool stat = static_r > 0.0f;   // static scale: the row's amax is not used
        const bool zero_row = !stat && !(amax > 0.0f);
        const float r = stat ? static_r : (zero_row ? 0.0f : __fdiv_rn(qmax, amax));
        if (tid == 0) scale[m] = stat ? static_s : (zero_row ? 0.0f : __fdiv_rn(amax, qmax));
        const uint64_t r2 = f2(r, kFold ? -r : r);
        if (active) {
            uint8_t *dst = q + (int64_t)m * K + E * tid;
#pragma unroll
            for (int g = 0; g < E / 32; ++g) {
                if (stat) store_codes_pairs<kInt8, kInt8>(p + 16 * g, r2, false, dst + 32 * g);
                else store_codes_pairs<kInt8>(p + 16 * g, r2, zero_row, dst + 32 * g);
            }
        }
        if (++slot == nslot) {
            slot = 0;
            phase ^= 1u;
            src = smem_u32(ring);
        } else {
            src += slot_stride;
        }
    }
    pdl_launch_dependents();   // this CTA's rows are done
    if (abort_flag && tid == 0) {
        // let the copies already issued into the ring land before the CTA exits
        for (int k = it; k < it + nslot; ++k) {
            const int m = (int)blockIdx.x + k * (int)gridDim.x;
            if (m >= M) break;
            const uint32_t a = smem_u32(&full[k % nslot]);
            const uint64_t t0 = globaltimer_ns();
            for (uint32_t n = 0;; ++n) {
                if (mbar_try_wait(a, (uint32_t)(k / nslot) & 1u)) break;
                if ((n & 63u) == 63u && globaltimer_ns() - t0 > 200000000ull) {
                    record_status(status, kStatusTimeout | (kSiteDrain << 8));
                    break;
                }
            }
        }
    }
}

// Staged launch plan: slots per CTA and CTAs per SM for a row of K elements,
// or false when the row does not suit the staged kernel.
struct StagedPlan {
    int threads, nslot, nbox, box_rows, ctas_per_sm;
    uint32_t slot_stride, smem;
};

// E: elements per thread (32, or 64 for long rows: fewer warps meet at each
// row's barrier and one lane exchange of the rotation stays in registers)
bool staged_plan(int64_t K, int E, StagedPlan &p) {
    if (K % 64 != 0 || K / 32 > 1024) return false;
    const int lines = (int)(K / 64);
    int nbox = (lines + 255) / 256;
    // several boxes per row start on 1024-byte boundaries (whole swizzle atoms)
    while (nbox <= 8 && nbox > 1 && (lines % nbox != 0 || (lines / nbox) % 8 != 0)) ++nbox;
    if (nbox > 8) return false;
    p.nbox = nbox;
    p.box_rows = lines / nbox;
    p.threads = (int)((K / E + 31) / 32 * 32);
    p.slot_stride = (uint32_t)((K * 2 + 1023) / 1024 * 1024);
    // about 1,152 threads per SM with 32 values each (registers for 56 per
    // thread) or 640 with 64 (about 100), and 220 KB of ring
    const uint32_t budget = 220u * 1024u;
    int want = (E == 64 ? 640 : 1152) / p.threads;
    want = want < 1 ? 1 : (want > 8 ? 8 : want);
    for (int P = want; P >= 1; --P) {
        const uint32_t per = budget / (uint32_t)P;
        if (per < 1024u + 2u * p.slot_stride) continue;
        int S = (int)((per - 1024u) / p.slot_stride);
        if (S > kMaxSlots) S = kMaxSlots;
        p.nslot = S;
        p.ctas_per_sm = P;
        p.smem = (uint32_t)S * p.slot_stride + 1024u;
        return true;
    }
    return false;
}

template <int MODE, int E, int MAXT, int MINB>
cudaError_t launch_staged(const StagedPlan &p, const uint16_t *x, int64_t M, int64_t K,
                          int64_t ldx, uint8_t *q, float *scale, const QuantEnv &env,
                          cudaStream_t st) {
    CUtensorMap tm;
    const uint64_t dims[3] = {64, (uint64_t)(K / 64), (uint64_t)M};
    const uint64_t strides[2] = {128, (uint64_t)ldx * 2};
    const uint32_t box[3] = {64, (uint32_t)p.box_rows, 1};
    if (internal_make_tmap_nd(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, x, dims, strides, box,
                              CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    auto kern = quant_staged_kernel<MODE, E, MAXT, MINB>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem);
    if (e != cudaSuccess) return e;
    // resident CTAs per SM, cached per row length (K / 64 <= 512 here; one
    // table per instantiation)
    static int resident_by_lines[513] = {0};
    int resident = resident_by_lines[K / 64];
    if (resident == 0) {
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&resident, kern, p.threads, p.smem);
        if (e != cudaSuccess) return e;
        if (resident < 1) return cudaErrorInvalidConfiguration;
        resident_by_lines[K / 64] = resident;
    }
    const int per_sm = resident < p.ctas_per_sm ? resident : p.ctas_per_sm;
    const int64_t want = (int64_t)per_sm * env.num_sms;
    const int grid = (int)(M < want ? M : want);
    return launch_kernel(kern, dim3(grid), dim3(p.threads), p.smem, st, 1, true, tm, (int)M, (int)K, p.nslot,
                         p.slot_stride, p.nbox, p.box_rows, q, scale, env.status, env.wait_limit_ns,
                         env.static_r, env.static_s);
}

template <int MODE>
cudaError_t launch_mode(const uint16_t *x, int64_t M, int64_t K, int64_t ldx, uint8_t *q,
                        float *scale, const QuantEnv &env, cudaStream_t st) {
    StagedPlan p;
    // a few rows per SM or fewer: the per-row kernel starts sooner
    const bool want = env.staging == 2 || (env.staging == 1 && M >= 8 * (int64_t)env.num_sms);
    if (want) {
        // rows of 8,192 to 12,288 elements: 64 values per thread (24,032 rows:
        // K = 8192 116.7 -> 106.5 us, 12288 174.1 -> 172.0 us; at K = 17408,
        // with two CTAs of 9 warps per SM, 268.3 -> 282.6 us, so 32 there)
        if (K >= 8192 && K <= 12288 && staged_plan(K, 64, p))
            return launch_staged<MODE, 64, 320, 2>(p, x, M, K, ldx, q, scale, env, st);
        if (staged_plan(K, 32, p)) {
            if (p.threads <= 576) return launch_staged<MODE, 32, 576, 2>(p, x, M, K, ldx, q, scale, env, st);
            return launch_staged<MODE, 32, 1024, 1>(p, x, M, K, ldx, q, scale, env, st);
        }
    }
    const int64_t nchunk = K / 32;
    if (nchunk <= 576) {
        const int T = (int)((nchunk + 31) / 32 * 32);
        return launch_kernel(quant_act_kernel<MODE, 1, 576, 2>, dim3((unsigned)M), dim3(T), 0, st, 1, true, x, K, ldx,
                             q, scale, env.static_r, env.static_s);
    }
    if (nchunk <= 1024) {
        const int T = (int)((nchunk + 31) / 32 * 32);
        return launch_kernel(quant_act_kernel<MODE, 1, 1024, 1>, dim3((unsigned)M), dim3(T), 0, st, 1, true, x, K,
                             ldx, q, scale, env.static_r, env.static_s);
    }
    const int64_t per = (nchunk + 1) / 2;
    const int T = (int)((per + 31) / 32 * 32);
    return launch_kernel(quant_act_kernel<MODE, 2, 1024, 1>, dim3((unsigned)M), dim3(T), 0, st, 1, true, x, K, ldx, q,
                         scale, env.static_r, env.static_s);
}

}  // namespace

cudaError_t launch_quant_act(int mode, const uint16_t *x, int64_t M, int64_t K, int64_t ldx,
                             uint8_t *q, float *scale, const QuantEnv &env, cudaStream_t st) {
    switch (mode) {
        case kActInt8H128: return launch_mode<kActInt8H128>(x, M, K, ldx, q, scale, env, st);
        case kActFp8: return launch_mode<kActFp8>(x, M, K, ldx, q, scale, env, st);
        case kActFp8H128: return launch_mode<kActFp8H128>(x, M, K, ldx, q, scale, env, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace clef
