// gemm.cu -- persistent, warp-specialised tcgen05 GEMM for sm_103a with the
// fused epilogues of the W8A8 projection path.
//
// Tile: 128 output rows x BN columns, accumulated in TMEM (fp32), two
// accumulator buffers so that the epilogue of one tile (or K-chunk) overlaps
// the mainloop of the next.  Operands are K-major ("row . row^T"): A is the
// activation [M][K], B the weight [N][K].
//
// Warp roles (one CTA per SM, persistent over tiles in M-fastest order so
// that concurrently running CTAs share weight tiles in L2):
//   warp 0     TMA producer (one elected lane)
//   warp 1     TMEM allocator and MMA issuer (one elected lane)
//   warps 2-7  INT8 only: converters, widening int8 codes to fp16 in the
//              128-byte-swizzled K-major layout the tensor core reads
//   8 warps    epilogue (TMEM -> registers -> scales / bias / SwiGLU -> HBM);
//              warp w reads TMEM lanes 32*(w%4)..+31, two warps per lane
//              quadrant split the tile's columns
//
// INT8 route.  tcgen05 has no integer MMA on sm_103a, so INT8 codes are
// multiplied exactly on the fp16 path: every code in [-127, 127] is exact in
// fp16, every product (<= 16129) is exact in fp32, and a sum of at most 1024
// such products stays below 2^24, so every partial sum the tensor core forms
// is an exactly representable integer.  The K loop is therefore cut into
// chunks of 1024; each chunk's fp32 accumulator is converted to int32 by the
// epilogue warps (exact) and added to int32 totals held in registers.  The
// result is the exact int32 accumulator, whatever the summation order.
//
// Sources: "CLEF Calibrated INT8 ConvRot" model card, Benefits (kernels fuse
// calibrated scales, biases and MLP SwiGLU); "Loading CLEF INT8" usage
// notes (fuse_mlp paired gate/up epilogue; gate/up packed at load);
// "clef-flash-FP8" model card, Quantization table (FP8 W8A8 dynamic);
// TensorFold pull request 1364 (LoRA products on bf16 tensor cores,
// y = bf16(y + bf16(x A^T) B^T)).
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "clef_kernels.h"
#include "clef_ptx.cuh"

namespace clef {

namespace {

template <int OP, int EPI, int BN_>
struct Cfg {
    static constexpr int BM = 128;
    static constexpr int BN = BN_;
    static constexpr bool kI8 = (OP == kOpI8);
    // Every MMA operand k-block is 128 bytes of K: 64 fp16/bf16 or 128 e4m3.
    static constexpr int kOperandBytes = (OP == kOpF8) ? 1 : 2;
    static constexpr int BK = 128 / kOperandBytes;         // K elements per k-block
    static constexpr int kMmaPerKBlock = 4;                // each MMA consumes 32 bytes of K
    static constexpr int kAStage = BM * 128;               // 16 KB
    static constexpr int kBStage = BN * 128;
    static constexpr int kStage = kAStage + kBStage;
    // Raw int8 k-block (INT8 only): 64 codes = 64 bytes per row, no swizzle.
    static constexpr int kRawA = BM * 64, kRawB = BN * 64, kRawStage = kRawA + kRawB;
    static constexpr int kSmemBudget = 232448 - 1024 - 512;  // opt-in max - align slack - barriers
    // INT8: two fp16 operand stages (converter -> MMA hand-off) and five raw
    // int8 stages (enough TMA lookahead to cover L2/HBM latency).
    static constexpr int NRAW = kI8 ? 5 : 0;
    static constexpr int NSTAGE_RAWFREE = (kSmemBudget - NRAW * kRawStage) / kStage;
    static constexpr int NSTAGE = kI8 ? 2 : (NSTAGE_RAWFREE > 8 ? 8 : NSTAGE_RAWFREE);
    static constexpr int kChunkKBlocks = kI8 ? 16 : (1 << 30);  // 1024 K per exact chunk
    static constexpr int kConvWarps = kI8 ? 6 : 0;
    static constexpr int kEpiWarp0 = kI8 ? 8 : 4;
    static constexpr int kNumWarps = kEpiWarp0 + 8;
    static constexpr int kThreads = kNumWarps * 32;
    static constexpr int kTmemCols = 2 * BN;               // two accumulator buffers
    static constexpr int kColsPerThread = BN / 2;          // columns one epilogue thread owns
    static constexpr int kChunks32 = kColsPerThread / 32;
    static constexpr bool kSwiGLU = (EPI == kEpiSwiGLU);
    static constexpr int kOutColsPerTile = kSwiGLU ? BN / 2 : BN;
    static constexpr int kSmemBytes = NSTAGE * kStage + NRAW * kRawStage + 1024 + 512;
    static_assert(BN == 64 || BN == 128 || BN == 256, "tile width");
    static_assert(kTmemCols >= 32 && kTmemCols <= 512, "TMEM columns");
    static_assert(kSmemBytes <= 232448, "shared memory");
    static_assert(NSTAGE >= 2, "pipeline depth");
};

struct Barriers {
    uint64_t full[8], empty[8];
    uint64_t raw_full[6], raw_empty[6];
    uint64_t acc_full[2], acc_empty[2];
    uint64_t drain;
    uint32_t tmem_slot;
    int abort;
};
static_assert(sizeof(Barriers) <= 512, "barrier block");

// Time-limited wait that ignores the abort flag (used only while winding
// down, to let copies and MMAs already in flight finish).
__device__ __forceinline__ bool mbar_wait_drain(uint64_t *bar, uint32_t parity, uint64_t limit_ns,
                                                unsigned int *status) {
    const uint32_t a = smem_u32(bar);
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 0;; ++it) {
        if (mbar_try_wait(a, parity)) return true;
        if ((it & 63u) == 63u && globaltimer_ns() - t0 > limit_ns) {
            record_status(status, kStatusTimeout | (kSiteDrain << 8));
            return false;
        }
    }
}

__device__ __forceinline__ uint32_t sub_f16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// Four int8 codes -> two fp16x2 words, exactly: flip the sign bit to get the
// offset-binary byte u = q + 128, place it under the fp16 exponent of 1024
// (0x64uu encodes 1024 + u), then subtract 1152.
__device__ __forceinline__ void s8x4_to_f16x4(uint32_t w, uint32_t &lo, uint32_t &hi) {
    const uint32_t u = w ^ 0x80808080u;
    lo = sub_f16x2(prmt(u, 0x64646464u, 0x4140u), 0x64806480u);
    hi = sub_f16x2(prmt(u, 0x64646464u, 0x4342u), 0x64806480u);
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}

__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&p);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ float silu_mul(float g, float u) {
    const float d = __fadd_rn(1.0f, expf(-g));
    return __fmul_rn(__fdiv_rn(g, d), u);
}

// Epilogue value of one accumulator: ((acc * sa) * sb) + bias, each rounded.
__device__ __forceinline__ float scale_bias(float acc, float sa, float sb, const uint16_t *bias,
                                            int n) {
    float y = __fmul_rn(__fmul_rn(acc, sa), sb);
    if (bias) y = __fadd_rn(y, __uint_as_float((uint32_t)__ldg(bias + n) << 16));
    return y;
}

}  // namespace

namespace {

template <int OP, int EPI, int BN>
struct Gemm {
    using C = Cfg<OP, EPI, BN>;

    struct Ctx {
        uint8_t *stage;      // NSTAGE x (A tile, B tile), 1024-aligned
        uint8_t *raw;        // NRAW x (raw A, raw B) for INT8
        Barriers *bar;
        uint32_t tmem;
        int num_m, num_n, num_tiles, nkb;
        WaitCtx w;
    };

    static __device__ __forceinline__ void tile_coords(const Ctx &c, int t, int &mb, int &nb) {
        mb = t % c.num_m;
        nb = t / c.num_m;
    }

    // ---------------------------------------------------------------- producer
    static __device__ void producer(const Ctx &c, const CUtensorMap *tmA, const CUtensorMap *tmB,
                                    const GemmArgs &a, uint32_t (&fills)[8]) {
        static_assert(C::NRAW <= 8 && C::NSTAGE <= 8, "fill bookkeeping");
        uint32_t s = 0, ph = 0;
        const int nstage = C::kI8 ? C::NRAW : C::NSTAGE;
        for (int t = blockIdx.x; t < c.num_tiles; t += gridDim.x) {
            int mb, nb;
            tile_coords(c, t, mb, nb);
            const int row_a = mb * C::BM;
            for (int kb = 0; kb < c.nkb; ++kb) {
                uint64_t *empty = C::kI8 ? &c.bar->raw_empty[s] : &c.bar->empty[s];
                uint64_t *full = C::kI8 ? &c.bar->raw_full[s] : &c.bar->full[s];
                if (!mbar_wait(empty, ph ^ 1u, c.w, kSiteTmaEmpty)) return;
                if (C::kI8) {
                    uint8_t *ra = c.raw + s * C::kRawStage;
                    uint8_t *rb = ra + C::kRawA;
                    const int k0 = kb * 64;
                    mbar_arrive_expect_tx(full, C::kRawStage);
                    tma_load_2d(ra, tmA, k0, row_a, full);
                    if (C::kSwiGLU) {
                        tma_load_2d(rb, tmB, k0, nb * (BN / 2), full);
                        tma_load_2d(rb + (BN / 2) * 64, tmB, k0, a.n_half + nb * (BN / 2), full);
                    } else {
                        tma_load_2d(rb, tmB, k0, nb * BN, full);
                    }
                } else {
                    uint8_t *sa = c.stage + s * C::kStage;
                    uint8_t *sb = sa + C::kAStage;
                    const int k0 = kb * C::BK;
                    mbar_arrive_expect_tx(full, C::kStage);
                    tma_load_2d(sa, tmA, k0, row_a, full);
                    if (C::kSwiGLU) {
                        tma_load_2d(sb, tmB, k0, nb * (BN / 2), full);
                        tma_load_2d(sb + (BN / 2) * 128, tmB, k0, a.n_half + nb * (BN / 2), full);
                    } else {
                        tma_load_2d(sb, tmB, k0, nb * BN, full);
                    }
                }
                fills[s] = ph | 2u;  // bit 1: stage filled at least once; bit 0: parity
                if (++s == (uint32_t)nstage) { s = 0; ph ^= 1u; }
            }
        }
    }

    // Before the CTA exits: wait (time-limited) until every copy issued into
    // each stage has landed, so no TMA write targets a finished CTA.
    static __device__ void drain_copies(const Ctx &c, const uint32_t (&fills)[8], unsigned int *st) {
        const int nstage = C::kI8 ? C::NRAW : C::NSTAGE;
        for (int s = 0; s < nstage; ++s) {
            if (!(fills[s] & 2u)) continue;
            uint64_t *full = C::kI8 ? &c.bar->raw_full[s] : &c.bar->full[s];
            mbar_wait_drain(full, fills[s] & 1u, 200000000ull, st);
        }
    }

    // ---------------------------------------------------------------- converters
    // Each converter thread owns the same 16-byte raw pieces in every k-block:
    // piece = ctid & 3 of rows (ctid >> 2) + 48 j, j = 0..7 (A rows 0..127,
    // then B rows).  Because 48 is a multiple of 8, the 128-byte swizzle phase
    // (row & 7) of a thread's rows is constant, so all shared addresses are a
    // per-thread base plus compile-time offsets.
    static __device__ void converter(const Ctx &c, int ctid) {
        constexpr int kThr = (C::kI8 ? C::kConvWarps : 6) * 32;  // native ops never call this
        constexpr int kRows = C::BM + BN;
        constexpr int kPer = kRows * 4 / kThr;
        static_assert(!C::kI8 || kRows * 4 % kThr == 0, "converter tasks");
        static_assert(!C::kI8 || (kThr / 4) % 8 == 0, "constant swizzle phase");
        constexpr uint32_t kSrcStep = (kThr / 4) * 64, kDstStep = (kThr / 4) * 128;
        const int row0 = ctid >> 2, piece = ctid & 3, phase = row0 & 7;
        const uint32_t src0 = (uint32_t)(row0 * 64 + piece * 16);
        const uint32_t dst0 = (uint32_t)(row0 * 128 + (((2 * piece) ^ phase) << 4));
        const uint32_t dst1 = (uint32_t)(row0 * 128 + (((2 * piece + 1) ^ phase) << 4));
        const uint32_t raw_base = smem_u32(c.raw), stage_base = smem_u32(c.stage);
        const int lane = threadIdx.x & 31;
        uint32_t rs = 0, rph = 0, cs = 0, cph = 0;
        for (int t = blockIdx.x; t < c.num_tiles; t += gridDim.x) {
            for (int kb = 0; kb < c.nkb; ++kb) {
                if (!mbar_wait(&c.bar->raw_full[rs], rph, c.w, kSiteConvRaw)) return;
                if (!mbar_wait(&c.bar->empty[cs], cph ^ 1u, c.w, kSiteConvEmpty)) return;
                const uint32_t src = raw_base + rs * C::kRawStage + src0;
                const uint32_t dst = stage_base + cs * C::kStage;
                constexpr int kBatch = kPer >= 4 ? 4 : kPer;  // loads in flight per thread
#pragma unroll
                for (int j0 = 0; j0 < kPer; j0 += kBatch) {
                    uint4 w[kBatch];
#pragma unroll
                    for (int j = 0; j < kBatch; ++j) w[j] = lds128(src + (j0 + j) * kSrcStep);
#pragma unroll
                    for (int j = 0; j < kBatch; ++j) {
                        uint32_t f[8];
                        s8x4_to_f16x4(w[j].x, f[0], f[1]);
                        s8x4_to_f16x4(w[j].y, f[2], f[3]);
                        s8x4_to_f16x4(w[j].z, f[4], f[5]);
                        s8x4_to_f16x4(w[j].w, f[6], f[7]);
                        sts128(dst + dst0 + (j0 + j) * kDstStep, f[0], f[1], f[2], f[3]);
                        sts128(dst + dst1 + (j0 + j) * kDstStep, f[4], f[5], f[6], f[7]);
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&c.bar->full[cs]);
                    mbar_arrive(&c.bar->raw_empty[rs]);
                }
                if (++rs == (uint32_t)C::NRAW) { rs = 0; rph ^= 1u; }
                if (++cs == (uint32_t)C::NSTAGE) { cs = 0; cph ^= 1u; }
            }
        }
    }

    // ---------------------------------------------------------------- MMA issuer
    static __device__ void mma_issuer(const Ctx &c) {
        constexpr uint32_t afmt = (OP == kOpBF16) ? 1u : 0u;  // F16 / BF16 / E4M3
        constexpr uint32_t idesc = idesc_f32acc(afmt, afmt, C::BM, BN);
        uint32_t s = 0, ph = 0, acc = 0, aph = 0;
        for (int t = blockIdx.x; t < c.num_tiles; t += gridDim.x) {
            for (int kb0 = 0; kb0 < c.nkb; kb0 += C::kChunkKBlocks) {
                const int kb1 = min(c.nkb, kb0 + C::kChunkKBlocks);
                if (!mbar_wait(&c.bar->acc_empty[acc], aph ^ 1u, c.w, kSiteMmaAccEmpty)) return;
                tc_fence_after();
                const uint32_t d = c.tmem + acc * BN;
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!mbar_wait(&c.bar->full[s], ph, c.w, kSiteMmaFull)) return;
                    tc_fence_after();
                    const uint32_t sa = smem_u32(c.stage + s * C::kStage);
                    const uint32_t sb = sa + C::kAStage;
#pragma unroll
                    for (int k = 0; k < C::kMmaPerKBlock; ++k) {
                        const uint64_t ad = sdesc_sw128(sa + 32 * k);
                        const uint64_t bd = sdesc_sw128(sb + 32 * k);
                        const uint32_t accum = (kb > kb0 || k > 0) ? 1u : 0u;
                        if (OP == kOpF8) mma_f8(d, ad, bd, idesc, accum);
                        else mma_f16(d, ad, bd, idesc, accum);
                    }
                    mma_commit(&c.bar->empty[s]);
                    if (++s == (uint32_t)C::NSTAGE) { s = 0; ph ^= 1u; }
                }
                mma_commit(&c.bar->acc_full[acc]);
                if (++acc == 2u) { acc = 0; aph ^= 1u; }
            }
        }
    }

    // ---------------------------------------------------------------- epilogue
    // TMEM column (within one accumulator buffer) of this thread's chunk j.
    static __device__ __forceinline__ int chunk_col(int j, int half) {
        if (C::kSwiGLU) {
            constexpr int kHalfChunks = C::kChunks32 / 2;
            return j < kHalfChunks ? half * (BN / 4) + 32 * j
                                   : BN / 2 + half * (BN / 4) + 32 * (j - kHalfChunks);
        }
        return half * (BN / 2) + 32 * j;
    }

    // Finish 32 consecutive output columns n0.. of one row from 32 fp32
    // accumulator values (for SwiGLU: gate values v, up values u).
    static __device__ __forceinline__ void finish32(const GemmArgs &a, int row, bool row_ok,
                                                    int n0, const float (&v)[32],
                                                    const float (&u)[32]) {
        if (!row_ok) return;
        const float sa = (EPI == kEpiScaleBias || EPI == kEpiSwiGLU) ? __ldg(a.sa + row) : 0.0f;
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            const int n = n0 + 8 * g;
            if (n >= a.N) break;  // N % 8 == 0: whole groups in or out
            float y[8];
            if (EPI == kEpiScaleBias || EPI == kEpiSwiGLU) {
                const float4 s0 = __ldg(reinterpret_cast<const float4 *>(a.sb + n));
                const float4 s1 = __ldg(reinterpret_cast<const float4 *>(a.sb + n) + 1);
                const float sb[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
#pragma unroll
                for (int i = 0; i < 8; ++i) y[i] = scale_bias(v[8 * g + i], sa, sb[i], a.bias, n + i);
                if (EPI == kEpiSwiGLU) {
                    const int nu = a.n_half + n;
                    const float4 t0 = __ldg(reinterpret_cast<const float4 *>(a.sb + nu));
                    const float4 t1 = __ldg(reinterpret_cast<const float4 *>(a.sb + nu) + 1);
                    const float su[8] = {t0.x, t0.y, t0.z, t0.w, t1.x, t1.y, t1.z, t1.w};
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        y[i] = silu_mul(y[i], scale_bias(u[8 * g + i], sa, su[i], a.bias, nu + i));
                }
            } else if (EPI == kEpiAddBF16) {
                const uint4 o = *reinterpret_cast<const uint4 *>(
                    static_cast<const uint16_t *>(a.out) + (int64_t)row * a.ldo + n);
                const uint32_t ow[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    y[2 * i] = __fadd_rn(bf16_lo(ow[i]), v[8 * g + 2 * i]);
                    y[2 * i + 1] = __fadd_rn(bf16_hi(ow[i]), v[8 * g + 2 * i + 1]);
                }
            } else {  // kEpiStoreBF16
#pragma unroll
                for (int i = 0; i < 8; ++i) y[i] = v[8 * g + i];
            }
            uint4 pk = make_uint4(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]),
                                  pack_bf16x2(y[4], y[5]), pack_bf16x2(y[6], y[7]));
            *reinterpret_cast<uint4 *>(static_cast<uint16_t *>(a.out) + (int64_t)row * a.ldo + n) = pk;
        }
    }

    static __device__ __forceinline__ void store_s32(const GemmArgs &a, int row, bool row_ok, int n0,
                                                     const int32_t *tot) {
        if (!row_ok) return;
        int32_t *o = static_cast<int32_t *>(a.out) + (int64_t)row * a.ldo;
#pragma unroll
        for (int g = 0; g < 8; ++g) {
            const int n = n0 + 4 * g;
            if (n >= a.N) break;
            *reinterpret_cast<int4 *>(o + n) = make_int4(tot[4 * g], tot[4 * g + 1], tot[4 * g + 2],
                                                         tot[4 * g + 3]);
        }
    }

    static __device__ void epilogue(const Ctx &c, const GemmArgs &a) {
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
        const int e = warp - C::kEpiWarp0, quad = warp & 3, half = e >> 2;
        const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
        uint32_t acc = 0, aph = 0;
        for (int t = blockIdx.x; t < c.num_tiles; t += gridDim.x) {
            int mb, nb;
            tile_coords(c, t, mb, nb);
            const int row = mb * C::BM + quad * 32 + lane;
            const bool row_ok = row < a.M;
            int32_t tot[C::kI8 ? C::kColsPerThread : 1];
            if (C::kI8) {
#pragma unroll
                for (int i = 0; i < C::kColsPerThread; ++i) tot[i] = 0;
            }
            for (int kb0 = 0; kb0 < c.nkb; kb0 += C::kChunkKBlocks) {
                if (!mbar_wait(&c.bar->acc_full[acc], aph, c.w, kSiteEpiAccFull)) return;
                tc_fence_after();
                const uint32_t tbase = c.tmem + acc * BN + lane_off;
                if (C::kI8) {
#pragma unroll
                    for (int j = 0; j < C::kChunks32; ++j) {
                        uint32_t r[32];
                        tmem_ld32(tbase + chunk_col(j, half), r);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 32; ++i) tot[32 * j + i] += __float2int_rn(__uint_as_float(r[i]));
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&c.bar->acc_empty[acc]);
                    if (++acc == 2u) { acc = 0; aph ^= 1u; }
                    if (kb0 + C::kChunkKBlocks < c.nkb) continue;  // more chunks of this tile
                    // the tile's exact int32 accumulators are complete
                    if (EPI == kEpiStoreS32) {
#pragma unroll
                        for (int j = 0; j < C::kChunks32; ++j)
                            store_s32(a, row, row_ok, nb * BN + chunk_col(j, half), tot + 32 * j);
                    } else if (C::kSwiGLU) {
#pragma unroll
                        for (int j = 0; j < C::kChunks32 / 2; ++j) {
                            float v[32], u[32];
#pragma unroll
                            for (int i = 0; i < 32; ++i) {
                                v[i] = __int2float_rn(tot[32 * j + i]);
                                u[i] = __int2float_rn(tot[32 * (j + C::kChunks32 / 2) + i]);
                            }
                            finish32(a, row, row_ok, nb * (BN / 2) + chunk_col(j, half), v, u);
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < C::kChunks32; ++j) {
                            float v[32];
#pragma unroll
                            for (int i = 0; i < 32; ++i) v[i] = __int2float_rn(tot[32 * j + i]);
                            finish32(a, row, row_ok, nb * BN + chunk_col(j, half), v, v);
                        }
                    }
                } else {
                    if (C::kSwiGLU) {
#pragma unroll
                        for (int j = 0; j < C::kChunks32 / 2; ++j) {
                            uint32_t rg[32], ru[32];
                            tmem_ld32(tbase + chunk_col(j, half), rg);
                            tmem_ld32(tbase + chunk_col(j + C::kChunks32 / 2, half), ru);
                            tmem_ld_wait();
                            float v[32], u[32];
#pragma unroll
                            for (int i = 0; i < 32; ++i) {
                                v[i] = __uint_as_float(rg[i]);
                                u[i] = __uint_as_float(ru[i]);
                            }
                            finish32(a, row, row_ok, nb * (BN / 2) + chunk_col(j, half), v, u);
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < C::kChunks32; ++j) {
                            uint32_t r[32];
                            tmem_ld32(tbase + chunk_col(j, half), r);
                            tmem_ld_wait();
                            float v[32];
#pragma unroll
                            for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
                            finish32(a, row, row_ok, nb * BN + chunk_col(j, half), v, v);
                        }
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&c.bar->acc_empty[acc]);
                    if (++acc == 2u) { acc = 0; aph ^= 1u; }
                }
            }
        }
    }
};

template <int OP, int EPI, int BN>
__global__ void __launch_bounds__(Cfg<OP, EPI, BN>::kThreads, 1)
gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
            const GemmArgs args) {
    using C = Cfg<OP, EPI, BN>;
    using G = Gemm<OP, EPI, BN>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t base = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + (((base + 1023u) & ~1023u) - base);
    Barriers *bar = reinterpret_cast<Barriers *>(smem + C::NSTAGE * C::kStage + C::NRAW * C::kRawStage);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::NSTAGE; ++s) {
            mbar_init(&bar->full[s], C::kI8 ? C::kConvWarps : 1);
            mbar_init(&bar->empty[s], 1);
        }
        for (int s = 0; s < C::NRAW; ++s) {
            mbar_init(&bar->raw_full[s], 1);
            mbar_init(&bar->raw_empty[s], C::kConvWarps);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bar->acc_full[s], 1);
            mbar_init(&bar->acc_empty[s], 8);
        }
        mbar_init(&bar->drain, 1);
        bar->abort = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) {
        tmem_alloc(&bar->tmem_slot, C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    typename G::Ctx c;
    c.stage = smem;
    c.raw = smem + C::NSTAGE * C::kStage;
    c.bar = bar;
    c.tmem = bar->tmem_slot;
    c.num_m = (args.M + C::BM - 1) / C::BM;
    c.num_n = (args.N + C::kOutColsPerTile - 1) / C::kOutColsPerTile;
    c.num_tiles = c.num_m * c.num_n;
    c.nkb = C::kI8 ? (args.K + 63) / 64 : (args.K + C::BK - 1) / C::BK;
    c.w.limit_ns = args.wait_limit_ns;
    c.w.abort = &bar->abort;
    c.w.status = args.status;

    uint32_t fills[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    if (warp < C::kEpiWarp0) {
        // INT8: control and converter warps hand registers to the epilogue
        // warps, which hold the int32 totals
        if (C::kI8) asm volatile("setmaxnreg.dec.sync.aligned.u32 64;");
        if (warp == 0) {
            if (lane == 0) {
                G::producer(c, &tmA, &tmB, args, fills);
                G::drain_copies(c, fills, args.status);
            }
        } else if (warp == 1) {
            if (lane == 0) {
                G::mma_issuer(c);
                // wind down: wait until every MMA issued by this thread completed
                mma_commit(&bar->drain);
                mbar_wait_drain(&bar->drain, 0, 200000000ull, args.status);
            }
        } else if (C::kI8) {
            G::converter(c, threadIdx.x - 64);
        }
    } else {
        if (C::kI8) asm volatile("setmaxnreg.inc.sync.aligned.u32 192;");
        G::epilogue(c, args);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(c.tmem, C::kTmemCols);
    }
}

template <int OP, int EPI, int BN>
cudaError_t launch_one(const CUtensorMap &tmA, const CUtensorMap &tmB, const GemmArgs &args,
                       int num_sms, cudaStream_t st) {
    using C = Cfg<OP, EPI, BN>;
    auto kern = gemm_kernel<OP, EPI, BN>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    const int num_m = (args.M + C::BM - 1) / C::BM;
    const int num_n = (args.N + C::kOutColsPerTile - 1) / C::kOutColsPerTile;
    const int tiles = num_m * num_n;
    const int grid = tiles < num_sms ? tiles : num_sms;
    kern<<<grid, C::kThreads, C::kSmemBytes, st>>>(tmA, tmB, args);
    return cudaGetLastError();
}

}  // namespace

int gemm_smem_bytes(int op, int bn) {
    if (op == kOpI8) return Cfg<kOpI8, kEpiScaleBias, 256>::kSmemBytes;
    if (op == kOpF8) return Cfg<kOpF8, kEpiScaleBias, 256>::kSmemBytes;
    if (bn == 64) return Cfg<kOpBF16, kEpiStoreBF16, 64>::kSmemBytes;
    if (bn == 128) return Cfg<kOpBF16, kEpiStoreBF16, 128>::kSmemBytes;
    return Cfg<kOpBF16, kEpiStoreBF16, 256>::kSmemBytes;
}

cudaError_t launch_gemm(int op, int epi, int bn, const CUtensorMap &tmA, const CUtensorMap &tmB,
                        const GemmArgs &args, int num_sms, cudaStream_t st) {
    if (op == kOpI8 && bn == 256) {
        switch (epi) {
            case kEpiScaleBias: return launch_one<kOpI8, kEpiScaleBias, 256>(tmA, tmB, args, num_sms, st);
            case kEpiSwiGLU: return launch_one<kOpI8, kEpiSwiGLU, 256>(tmA, tmB, args, num_sms, st);
            case kEpiStoreS32: return launch_one<kOpI8, kEpiStoreS32, 256>(tmA, tmB, args, num_sms, st);
            default: break;
        }
    } else if (op == kOpF8 && bn == 256) {
        switch (epi) {
            case kEpiScaleBias: return launch_one<kOpF8, kEpiScaleBias, 256>(tmA, tmB, args, num_sms, st);
            case kEpiSwiGLU: return launch_one<kOpF8, kEpiSwiGLU, 256>(tmA, tmB, args, num_sms, st);
            default: break;
        }
    } else if (op == kOpBF16) {
        if (epi == kEpiStoreBF16) {
            if (bn == 64) return launch_one<kOpBF16, kEpiStoreBF16, 64>(tmA, tmB, args, num_sms, st);
            if (bn == 128) return launch_one<kOpBF16, kEpiStoreBF16, 128>(tmA, tmB, args, num_sms, st);
            if (bn == 256) return launch_one<kOpBF16, kEpiStoreBF16, 256>(tmA, tmB, args, num_sms, st);
        } else if (epi == kEpiAddBF16 && bn == 256) {
            return launch_one<kOpBF16, kEpiAddBF16, 256>(tmA, tmB, args, num_sms, st);
        }
    }
    return cudaErrorInvalidValue;
}

}  // namespace clef
