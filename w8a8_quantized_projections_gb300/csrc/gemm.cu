// gemm.cu -- persistent, warp-specialised tcgen05 GEMM for sm_103a with the
// fused epilogues of the W8A8 projection path.
//
// Tiles are 128 output rows per CTA by BN columns, accumulated in TMEM (fp32).
// Operands are K-major ("row . row^T"): A is the activation [M][K], B the
// weight [N][K].  Two tile modes:
//   single  one CTA per 128 x BN tile, two TMEM accumulator buffers so the
//           epilogue of one tile overlaps the mainloop of the next;
//   pair    (BN = 256, M > 128) a cluster of two CTAs shares a 256 x 256 tile
//           through tcgen05 cta_group::2: each CTA stages its own 128 A rows and
//           half of the B rows, the leader CTA issues the MMAs for both, and the
//           tensor cores of the two SMs read each B half once.  This halves the
//           B operand's shared-memory traffic per SM, which is what bounds the
//           single mode (about 128 B per clock per SM covers TMA writes, thread
//           accesses and tensor-core operand reads together).
//
// Schedule: one CTA (or pair) per SM, persistent over tiles slot, slot +
// nslots, ... in M-fastest order, so that concurrently running CTAs share
// weight tiles in L2 (N-fastest for the LoRA launches, whose large operand is
// the activation or y).  INT8 stream-K (a caller-bound workspace, pair mode,
// not SwiGLU): when the last wave of tiles would leave pairs idle, the whole
// waves run as above and the remaining tiles' k-blocks are dealt to the pairs
// in even runs; the pieces of a tile meet as exact int32 partial sums.
//
// Warp roles:
//   warp 0     TMA producer (one elected lane)
//   warp 1     TMEM allocator and MMA issuer (one elected lane; in pair mode the
//              leader's only)
//   INT8 only  converter warps widening int8 codes to fp16 in the 128-byte
//              swizzled K-major layout the tensor core reads
//   8 warps    epilogue (TMEM -> registers -> scales / bias / SwiGLU -> HBM);
//              warp w reads TMEM lanes 32*(w%4)..+31, two warps per lane
//              quadrant split the tile's columns
//
// INT8 route.  tcgen05 has no integer MMA on sm_103a, so INT8 codes are
// multiplied exactly on the fp16 path: every code in [-127, 127] is exact in
// fp16, every product (<= 16129) is exact in fp32, and a sum of at most 1024
// such products stays below 2^24, so every partial sum the tensor core forms
// is an exactly representable integer.  The K loop is therefore cut into
// chunks of at most 1024; each chunk's fp32 accumulator is converted to int32
// by the epilogue warps (exact) and added to int32 totals held in registers.
// The result is the exact int32 accumulator, whatever the summation order or
// split.
//
// Sources: "CLEF Calibrated INT8 ConvRot" model card, Benefits (kernels fuse
// calibrated scales, biases and MLP SwiGLU); "Loading CLEF INT8" usage
// notes (fuse_mlp paired gate/up epilogue; gate/up packed at load);
// "clef-flash-FP8" model card, Quantization table (FP8 W8A8 dynamic);
// TensorFold pull request 1364 (LoRA products on bf16 tensor cores,
// y = bf16(y + bf16(x A^T) B^T)).
#include <algorithm>
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "clef_kernels.h"
#include "clef_ptx.cuh"

namespace clef {

namespace {

template <int OP, int EPI, int BN_, bool PAIR>
struct Cfg {
    static constexpr int BM = 128;                         // A rows per CTA
    static constexpr int BN = BN_;                         // accumulator columns
    static constexpr int kTileRows = PAIR ? 2 * BM : BM;   // output rows per tile
    static constexpr bool kI8 = (OP == kOpI8);
    // Every MMA operand k-block is 128 bytes of K: 64 fp16/bf16 or 128 e4m3.
    static constexpr int kOperandBytes = (OP == kOpF8) ? 1 : 2;
    static constexpr int BK = 128 / kOperandBytes;         // K elements per k-block
    static constexpr int kMmaPerKBlock = 4;                // each MMA consumes 32 bytes of K
    static constexpr int kBRows = PAIR ? BN / 2 : BN;      // B rows staged per CTA
    static constexpr int kAStage = BM * 128;               // 16 KB
    static constexpr int kBStage = kBRows * 128;
    static constexpr int kStage = kAStage + kBStage;
    // Raw int8 k-block (INT8 only): 64 codes = 64 bytes per row, no swizzle.
    static constexpr int kRawA = BM * 64, kRawB = kBRows * 64, kRawStage = kRawA + kRawB;
    static constexpr int kSmemBudget = 232448 - 1024 - 512;  // opt-in max - align slack - barriers
    // INT8: fp16 operand stages (converter -> MMA hand-off) and raw int8
    // stages (TMA lookahead to cover L2/HBM latency).
    // Pair mode: raw stages are half as large; six of them give the TMA its
    // lookahead and four fp16 stages absorb the converters' per-k-block
    // latency (measured against 3 + 8 and 5 + 4: 1502 x 34816 x 5120 in 414
    // against 432 and 426 us).
    // Single CTAs: 4 raw stages, a multiple of their 2 converter groups (see
    // kConvGroups: 5 let a group's raw-stage waits skip a phase).
    static constexpr int NRAW = kI8 ? (PAIR ? 6 : 4) : 0;
    // Epilogue warps: 16 for the FP8 SwiGLU epilogue (exp and an IEEE
    // division per output must keep pace with a k-loop less than half as long
    // as INT8's: 120 -> 102 us on 1502 x 24576 x 4096), 8 otherwise (the
    // INT8 int32 totals take most registers; the scale/bias epilogue is light
    // and more warps only crowd the producer and MMA warps' schedulers).
    // kParts warps share each TMEM lane quadrant, splitting the tile's columns.
    static constexpr int kEpiWarps = (!kI8 && BN_ == 256 && (EPI == kEpiSwiGLU || EPI == kEpiLoraSwiGLU)) ? 16 : 8;
    static constexpr int kParts = kEpiWarps / 4;
    // LoRA gate/up adds then SwiGLU over base g|u tiles read by TMA (bf16
    // operands, the unfused LoRA path)
    static constexpr bool kLoraSwi = (EPI == kEpiLoraSwiGLU);
    // y += acc: a ring of kYBufs y tiles (BM x BN bf16) that TMA loads
    // kYBufs - 1 tiles ahead and stores.  128-wide tiles keep 3, which leaves
    // room for 4 operand stages: the t and B operands come from L2 and their
    // latency bounds this short-K GEMM as much as y's (24,032 x 4096 rank-256
    // expand: 2 y buffers + 5 stages 102.7 us, 4 + 3 103.3 us, 3 + 4 96.5 us;
    // 256-wide pair tiles with 2 + 3: 114.7 us)
    static constexpr int kYTile = BM * BN * 2;
    static constexpr int kYBufs = (EPI == kEpiAddBF16 && BN == 128) ? 3 : 2;
    static constexpr int kEpiStage = (EPI == kEpiAddBF16 || kLoraSwi) ? kYBufs * kYTile : 0;
    static constexpr int NSTAGE_RAWFREE = (kSmemBudget - NRAW * kRawStage - kEpiStage) / kStage;
    static constexpr int NSTAGE = kI8 ? (PAIR ? 4 : 2) : (NSTAGE_RAWFREE > 8 ? 8 : NSTAGE_RAWFREE);
    static constexpr int kChunkKBlocks = kI8 ? 16 : (1 << 30);  // 1024 K per exact chunk
    static constexpr int kConvWarps = kI8 ? 6 : 0;
    static constexpr int kEpiWarp0 = kI8 ? 8 : 4;
    static constexpr int kNumWarps = kEpiWarp0 + kEpiWarps;
    static constexpr int kThreads = kNumWarps * 32;
    static constexpr int kAccBufs = 2;                     // double-buffered accumulator
    static constexpr int kTmemCols = kAccBufs * BN;
    static constexpr int kColsPerThread = BN / kParts;     // columns one epilogue thread owns
    static constexpr int kChunks32 = kColsPerThread / 32;
    static constexpr bool kSwiGLU =   // gate|up tile
        (EPI == kEpiSwiGLU || EPI == kEpiLoraSwiGLU || EPI == kEpiSwiGLULora);
    // INT8 with the LoRA expand fused: after a tile's INT8 k-blocks, the
    // producer loads the tile's t rows and B-factor rows (bf16) by TMA straight
    // into the fp16 operand ring, the converters pass those stages through,
    // and the MMA issuer accumulates t B^T as the tile's last chunk
    static constexpr bool kLoraFused = (EPI == kEpiScaleBiasLora || EPI == kEpiSwiGLULora);
    // Fused LoRA, B-factor rows one LoRA k-block stages per CTA: gate/up
    // k-blocks carry one factor's rows only (gate or up, halved between a
    // pair), each the operand of an N = BN/2 MMA into its half of the
    // accumulator
    static constexpr int kLoraBRows = kSwiGLU ? (PAIR ? BN / 4 : BN / 2) : kBRows;
    // epilogues that apply the row and column scales and the bias
    static constexpr bool kScaled =
        (EPI == kEpiScaleBias || EPI == kEpiSwiGLU || EPI == kEpiScaleBiasLora || EPI == kEpiSwiGLULora);
    // INT8 stream-K is compiled into the pair kernels (exact int32 pieces)
    // but not the SwiGLU one: the gate/up launches of the workloads fill at
    // least 94% of their last wave, and with the split path compiled in the
    // unsplit gate/up kernel ran 1.2% slower (352.7 against 344.5 us)
    //
    // FP8 linear: a launch with K of at least 64 k-blocks (8,192) sums each
    // tile's K as kKParts fixed parts (ceil(nkb / kKParts) k-blocks each, the
    // last the rest), accumulator chunks that the epilogue adds in fp32 in K
    // order.  The cut depends on K alone and the parts are added in the same
    // order whether a tile runs whole or its parts run on several CTA pairs
    // (stream-K over a partly empty last wave, the parts meeting in the
    // workspace), so a row's bits do not depend on M.
    //
    // LoRA x A^T (bf16 store): the same with 4 parts from 96 k-blocks (K =
    // 6,144) on, for the adapters of the 24,032-token layer's o (K = 6,144)
    // and down (K = 17,408) projections, whose 94 row blocks leave a second
    // wave of 18 tiles on 76 pairs: 4 parts divide both k-block counts (96,
    // 272), and 18 x 4 pieces fit in one wave.  Single-CTA tiles (calls of
    // at most 128 rows, narrow ranks) sum the same parts, so a row's bits do
    // not depend on the call's row count.
    static constexpr bool kKSplit =
        (OP == kOpF8 && EPI == kEpiScaleBias) || (OP == kOpBF16 && EPI == kEpiStoreBF16);
    static constexpr int kKSplitMinKBlocks = (OP == kOpF8) ? 64 : 96;
    static constexpr int kKParts = (OP == kOpF8) ? 3 : 4;
    static constexpr bool kStreamK = PAIR && ((kI8 && !kSwiGLU && !kLoraFused) || kKSplit);
    static constexpr int kOutColsPerTile = kSwiGLU ? BN / 2 : BN;
    // full[s]: TMA (native) or the local converter warps (INT8); in pair mode
    // the leader's barrier also counts the peer's forwarded readiness.
    // The converter warps form kConvGroups groups of kGroupWarps; group g
    // widens k-blocks g, g + kConvGroups, ... of the CTA's k-block sequence, so
    // a warp pays its per-k-block waits, fence and arrives once every
    // kConvGroups k-blocks (1, 2, 3 groups: 1502 x 34816 x 5120 in 399, 381,
    // 359 us).  Each of a group's waits on a stage barrier must target the
    // phase just after one it already knows complete, never two ahead (the
    // parity test of an mbarrier wait cannot tell those apart):
    // - fp16 stages: the group's successive k-blocks lie at most NSTAGE
    //   apart.  Their "empty" phases complete in k-block order (the MMAs
    //   release the stages in order), so the wait for a k-block's stage
    //   follows the release its previous k-block waited for, which is at
    //   least the stage's preceding phase;
    // - raw stages: NRAW a multiple of kConvGroups.  Their "full" phases
    //   complete when copies land, in no guaranteed order, so the stage's
    //   preceding phase must be one of the group's own k-blocks (with 5
    //   stages and 2 groups a group's next use of a stage came two phases
    //   after its last one).
    static constexpr int kConvGroups = PAIR ? 3 : 2;   // single CTAs have 2 fp16 stages
    static constexpr int kGroupWarps = kConvWarps / kConvGroups;
    static constexpr int kFullArrivals = kI8 ? kGroupWarps : 1;
    static constexpr int kAccEmptyArrivals = kEpiWarps * (PAIR ? 2 : 1);
    static constexpr int kSmemBytes = NSTAGE * kStage + NRAW * kRawStage + kEpiStage + 1024 + 512;
    static_assert(BN == 64 || BN == 128 || BN == 256, "tile width");
    static_assert(!PAIR || BN == 256, "pair mode uses 256-wide tiles");
    static_assert(kTmemCols >= 32 && kTmemCols <= 512, "TMEM columns");
    static_assert(kSmemBytes <= 232448, "shared memory");
    static_assert(NSTAGE >= 2, "pipeline depth");
    static_assert(!kI8 || (kConvWarps % kConvGroups == 0 && kConvGroups <= NSTAGE && NRAW % kConvGroups == 0),
                  "converter groups");
    // stream-K counters and pieces are laid out for eight epilogue warps of
    // 128 int32 columns each
    static_assert(!kStreamK || (kEpiWarps == 8 && kColsPerThread == 128), "stream-K layout");
    static_assert(!kLoraFused || (kI8 && NSTAGE <= 4), "the fused LoRA expand rides the INT8 fp16 operand ring");
};

struct Barriers {
    uint64_t full[8], empty[8];
    uint64_t raw_full[8], raw_empty[8];
    uint64_t acc_full[2], acc_empty[2];
    uint64_t drain;
    uint64_t never;      // nothing arrives here: the forced-timeout test waits on it
    uint64_t ybar[4];    // y += acc: the y tile in buffer b has landed
    uint64_t ltma[4];    // fused LoRA: the t and B tiles in fp16 operand slot s have landed
    uint64_t epi_done;   // y += acc: every epilogue warp has written the tile's y
    uint32_t tmem_slot;
    int abort;
    // INT8 stream-K (kept here rather than in registers): the count of slots
    // sharing the last tiles' k-blocks (0 = off) and the first of those tiles
    int sk, sk_tail0;
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

// Arrive with an expected transaction count and return the phase token,
// which a later wait names unambiguously (unlike a parity).
__device__ __forceinline__ uint64_t mbar_arrive_expect_tx_token(uint64_t *bar, uint32_t bytes) {
    uint64_t st;
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 %0, [%1], %2;"
                 : "=l"(st) : "r"(smem_u32(bar)), "r"(bytes) : "memory");
    return st;
}

// Time-limited wait for the phase a token was taken in; like
// mbar_wait_drain it ignores the abort flag (used for copies that must land
// before their shared memory may be reused or released).
__device__ __forceinline__ bool mbar_wait_token(uint64_t *bar, uint64_t token, uint64_t limit_ns,
                                                unsigned int *status, unsigned int site) {
    const uint32_t a = smem_u32(bar);
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 0;; ++it) {
        uint32_t ok;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}\n"
            : "=r"(ok) : "r"(a), "l"(token) : "memory");
        if (ok) return true;
        if ((it & 63u) == 63u && globaltimer_ns() - t0 > limit_ns) {
            record_status(status, kStatusTimeout | (site << 8));
            return false;
        }
    }
}

// Arrive `count` times at once.
__device__ __forceinline__ void mbar_arrive_n(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
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

__device__ __forceinline__ float bf16_round(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// silu(g) * u = g / (1 + exp(-g)) * u in fp32, two ways whose bf16 results
// both stay within one ulp of the correctly rounded libm value.
// IEEE: CUDA expf and a correctly rounded division.
__device__ __forceinline__ float silu_mul_ieee(float g, float u) {
    const float d = __fadd_rn(1.0f, expf(-g));
    return __fmul_rn(__fdiv_rn(g, d), u);
}

// Fast: the hardware exp2 and reciprocal approximations (a few fp32 ulps).
// Denominators above 2^126 (g below about -87) are scaled by 2^-64 with the
// numerator, exactly, to keep the fast quotient in its accurate range.
__device__ __forceinline__ float silu_mul_fast(float g, float u) {
    const float d = __fadd_rn(1.0f, __expf(-g));
    const float sc = d > 0x1p126f ? 0x1p-64f : 1.0f;
    return __fmul_rn(__fdividef(g * sc, d * sc), u);
}

// Epilogue value of one accumulator: ((acc * sa) * sb) + bias, each rounded
// (no bias: no add, so a -0 product stays -0).
__device__ __forceinline__ float scale_bias(float acc, float sa, float sb, float bias, bool has_bias) {
    const float y = __fmul_rn(__fmul_rn(acc, sa), sb);
    return has_bias ? __fadd_rn(y, bias) : y;
}

// Column scales and biases of output columns n .. n + 7 (n % 8 == 0; sb and
// the bias 16-byte aligned): two 16-byte loads of sb and one of the bias.
// Every lane of a warp reads the same columns, so each load is one L1
// wavefront -- eight scalar loads per column group were the epilogue's
// largest L1 cost, taken at every tile's end while the next tile's first
// k-blocks were being widened.
__device__ __forceinline__ void load_cols8(const float *sb, const uint16_t *bias, int n, float (&s)[8],
                                           float (&b)[8]) {
    const float4 s0 = __ldg(reinterpret_cast<const float4 *>(sb + n));
    const float4 s1 = __ldg(reinterpret_cast<const float4 *>(sb + n) + 1);
    s[0] = s0.x; s[1] = s0.y; s[2] = s0.z; s[3] = s0.w;
    s[4] = s1.x; s[5] = s1.y; s[6] = s1.z; s[7] = s1.w;
    if (bias) {
        const uint4 w = __ldg(reinterpret_cast<const uint4 *>(bias + n));
        const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            b[2 * i] = bf16_lo(ww[i]);
            b[2 * i + 1] = bf16_hi(ww[i]);
        }
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) b[i] = 0.0f;
    }
}

// Output columns n .. n + 15 of one row (bf16; w: eight packed words in
// column order).  One 32-byte store when every row of the output starts on a
// 32-byte boundary (out_v32) and all 16 columns lie inside N, else 16-byte
// stores of the 8-column groups inside N (N % 8 == 0).  A warp's lanes hold
// 32 different rows, so every store instruction touches 32 lines: the wider
// store halves the instructions and the L1 work of the epilogue's writes.
__device__ __forceinline__ void store_bf16x16(const GemmArgs &a, int row, int n, const uint32_t (&w)[8]) {
    if (n >= a.N) return;
    uint16_t *p = static_cast<uint16_t *>(a.out) + (int64_t)row * a.ldo + n;
    if (a.out_v32 && n + 16 <= a.N) {
        asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
                     :: "l"(p), "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]),
                        "r"(w[7])
                     : "memory");
    } else {
        *reinterpret_cast<uint4 *>(p) = make_uint4(w[0], w[1], w[2], w[3]);
        if (n + 8 < a.N) *reinterpret_cast<uint4 *>(p + 8) = make_uint4(w[4], w[5], w[6], w[7]);
    }
}

// ---------------------------------------------------------------- CTA pairs

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Shared::cluster address of the same shared variable in the pair's leader (rank 0).
__device__ __forceinline__ uint32_t leader_addr(const void *local) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, 0;" : "=r"(r) : "r"(smem_u32(local)));
    return r;
}

__device__ __forceinline__ void arrive_cluster(uint32_t cluster_bar) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar)
                 : "memory");
}

// Relaxed cluster-scope arrive: no release fence.  Used only to forward a
// readiness signal whose data ordering was already established locally (see
// Gemm::forwarder); a release at cluster scope costs about a microsecond.
__device__ __forceinline__ void arrive_cluster_relaxed(uint32_t cluster_bar) {
    asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar)
                 : "memory");
}

__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
                 ::: "memory");
}

__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar_addr, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(bar_addr), "r"(parity)
        : "memory");
    return ok != 0;
}

// Time-limited wait with cluster-scope acquire (barriers that receive arrivals
// from the peer CTA or multicast commits); otherwise as mbar_wait.
__device__ __forceinline__ bool mbar_wait_cl(uint64_t *bar, uint32_t parity, const WaitCtx &w,
                                             unsigned int site) {
    const uint32_t a = smem_u32(bar);
    if (mbar_try_wait_cluster(a, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait_cluster(a, parity)) return true;
        if ((it & 63u) == 0u) {
            if (*w.abort) return false;
            if (globaltimer_ns() - t0 > w.limit_ns) {
                record_status(w.status, kStatusTimeout | (site << 8));
                *w.abort = 1;
                return false;
            }
        }
    }
}

__device__ __forceinline__ void mma2_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}\n"
        ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma2_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                        uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}\n"
        ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive on the barrier at this shared offset in both CTAs of the pair once
// the pair's MMAs issued so far by this thread have completed.
__device__ __forceinline__ void mma2_commit_both(uint64_t *bar) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(smem_u32(bar)), "h"((uint16_t)3) : "memory");
}

__device__ __forceinline__ void mma2_commit_local(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 ::"r"(smem_u32(bar)) : "memory");
}

// TMA tile store from shared memory (bulk-group completion) and its waits.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *m, const void *smem_src, int32_t c0,
                                             int32_t c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];"
        ::"l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(smem_src)), "r"(c0), "r"(c1)
        : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_all() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// TMA tile load into this CTA's shared memory whose completion is counted on
// a barrier that may live in the peer CTA (shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(void *smem_dst, const CUtensorMap *m, int32_t c0,
                                                 int32_t c1, uint32_t cluster_bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];"
        ::"r"(smem_u32(smem_dst)), "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1),
          "r"(cluster_bar)
        : "memory");
}

}  // namespace

namespace {

template <int OP, int EPI, int BN, bool PAIR>
struct Gemm {
    using C = Cfg<OP, EPI, BN, PAIR>;

    struct Ctx {
        uint8_t *stage;      // NSTAGE x (A tile, B tile), 1024-aligned
        uint8_t *raw;        // NRAW x (raw A, raw B) for INT8
        uint8_t *epi;        // kEpiStage bytes of epilogue buffers
        const CUtensorMap *tmC;  // y += acc: the y tensor map; LoRA gate/up: the base g|u map
        const CUtensorMap *tmD;  // LoRA gate/up: the h tensor map; fused LoRA: the B factor
        const CUtensorMap *tmB2; // fused LoRA, SwiGLU: the up factor
        Barriers *bar;
        uint32_t tmem;       // accumulator base (the leader's allocation in pair mode)
        uint32_t rank;       // rank in the CTA pair (0 in single mode)
        int slot, nslots;    // tile-loop start and stride
        int num_m, num_n, num_tiles, nkb;
        int n_fastest;       // tile order: 0 = M fastest, 1 = N fastest
        int band_m;          // M fastest: row blocks per band (1 .. num_m)
        int force_timeout;   // test knob: this CTA's MMA issuer waits on a barrier nothing signals
        int nl;              // fused LoRA: bf16 k-blocks per tile (0 = none)
        int chunk;           // k-blocks per accumulator chunk
        WaitCtx w;
    };

    // M-fastest: the CTAs running at the same time share B (weight) tiles,
    // within bands of band_m row blocks (a band's every column block before
    // the next band), so that the band's A rows are read from DRAM once;
    // N-fastest: they share A row blocks (x A^T, where x is the large operand).
    static __device__ __forceinline__ void tile_coords(const Ctx &c, int t, int &mb, int &nb) {
        if (c.n_fastest) {
            nb = t % c.num_n;
            mb = t / c.num_n;
        } else {
            const int band = t / (c.band_m * c.num_n);
            const int m0 = band * c.band_m;
            const int rows = min(c.band_m, c.num_m - m0);
            const int local = t - band * c.band_m * c.num_n;
            mb = m0 + local % rows;
            nb = local / rows;
        }
    }

    // A CTA's work is a list of segments: a tile and a range of its k-blocks.
    // Classic schedule: whole tiles slot, slot + nslots, ...  Stream-K: the
    // same for the tiles before sk_tail0 (the whole waves), then the k-blocks
    // of the remaining tiles, in (tile, k-block) order, dealt to the first sk
    // slots in even contiguous runs: slot p < sk owns k-block indices [b(p),
    // b(p + 1)) with b(p) = floor(p * (num_tiles - sk_tail0) * nkb / sk).
    // part: -1 for a whole tile, 0 for the slot's first piece of a split
    // tile, 1 for its second (a run is shorter than a tile, so it touches at
    // most two).
    struct Seg {
        int tile, kb0, kb1, part;
    };
    static __device__ __forceinline__ int sk_of(const Ctx &c) { return C::kStreamK ? c.bar->sk : 0; }
    static __device__ __forceinline__ int sk_tail0(const Ctx &c) { return C::kStreamK ? c.bar->sk_tail0 : 0; }
    // (32-bit arithmetic: the launcher splits only when slots x remaining
    // k-blocks stays below 2^32)
    static __device__ __forceinline__ int sk_bound(const Ctx &c, int p) {
        return (int)((uint32_t)p * (uint32_t)((c.num_tiles - sk_tail0(c)) * c.nkb) / (uint32_t)sk_of(c));
    }
    static __device__ __forceinline__ int sk_owner(const Ctx &c, int v) {
        int p = (int)((uint32_t)v * (uint32_t)sk_of(c) / (uint32_t)((c.num_tiles - sk_tail0(c)) * c.nkb));
        while (p + 1 < sk_of(c) && sk_bound(c, p + 1) <= v) ++p;
        while (p > 0 && sk_bound(c, p) > v) --p;
        return p;
    }
    // The slot's segments: `whole` whole tiles, then (stream-K) the pieces
    // of its run, `total` in all.  Loops run i = 0 .. total - 1 over seg_at.
    struct Segs {
        int whole, total;
    };
    static __device__ __forceinline__ Segs seg_plan(const Ctx &c) {
        const int whole_end = sk_of(c) ? sk_tail0(c) : c.num_tiles;
        Segs p;
        p.whole = c.slot < whole_end ? (whole_end - 1 - c.slot) / c.nslots + 1 : 0;
        p.total = p.whole;
        if (sk_of(c) && c.slot < sk_of(c)) {
            const int v0 = sk_bound(c, c.slot), v1 = sk_bound(c, c.slot + 1);
            if (v1 > v0) p.total += (v1 - 1) / c.nkb - v0 / c.nkb + 1;
        }
        return p;
    }
    static __device__ __forceinline__ Seg seg_at(const Ctx &c, const Segs &p, int i) {
        Seg sg;
        if (i < p.whole) {
            sg.tile = c.slot + i * c.nslots;
            sg.kb0 = 0;
            sg.kb1 = c.nkb;
            sg.part = -1;
            return sg;
        }
        const int v0 = sk_bound(c, c.slot), v1 = sk_bound(c, c.slot + 1);
        const int rel0 = v0 / c.nkb;
        if (i == p.whole) {
            sg.tile = sk_tail0(c) + rel0;
            sg.kb0 = v0 - rel0 * c.nkb;
            sg.kb1 = min(c.nkb, sg.kb0 + (v1 - v0));
            sg.part = (sg.kb0 == 0 && sg.kb1 == c.nkb) ? -1 : 0;
        } else {
            sg.tile = sk_tail0(c) + rel0 + 1;
            sg.kb0 = 0;
            sg.kb1 = v1 - (rel0 + 1) * c.nkb;
            sg.part = 1;
        }
        return sg;
    }

    // Waits on barriers that receive arrivals from the peer CTA or from the
    // pair's multicast commits use cluster-scope acquire.
    static __device__ __forceinline__ bool wait_pair(uint64_t *bar, uint32_t parity, const Ctx &c,
                                                     unsigned int site) {
        return PAIR ? mbar_wait_cl(bar, parity, c.w, site) : mbar_wait(bar, parity, c.w, site);
    }

    // Row of the weight operand that this CTA's B stage starts with.
    static __device__ __forceinline__ int b_row(const Ctx &c, const GemmArgs &a, int nb, int half) {
        if (C::kLoraSwi) return nb * (BN / 2);   // each half from its own tensor map
        if (C::kSwiGLU) return (half ? a.n_half : 0) + nb * (BN / 2);
        return nb * BN + (int)c.rank * C::kBRows;
    }

    // Fused LoRA: the LoRA k-blocks that follow a segment's k-blocks (a whole
    // tile's; the fused kernels never split tiles).
    static __device__ __forceinline__ int lora_kblocks(const Ctx &c, const Seg &sg) {
        return (C::kLoraFused && sg.part < 0) ? c.nl : 0;
    }

    // Fused LoRA: first column of t read by the tiles of column block nb (the
    // segment of the adapter whose output columns the tile covers).
    static __device__ __forceinline__ int lora_tcol(const GemmArgs &a, int nb) {
        const int n0 = nb * C::kOutColsPerTile;
        int tcol = a.lora_seg_tcol[0];
#pragma unroll
        for (int k = 1; k < kLoraMaxSegs; ++k)
            if (k < a.lora_nseg && n0 >= a.lora_seg_end[k - 1]) tcol = a.lora_seg_tcol[k];
        return tcol;
    }

    // ---------------------------------------------------------------- producer
    static __device__ void producer(const Ctx &c, const CUtensorMap *tmA, const CUtensorMap *tmB0,
                                    const CUtensorMap *tmB2, const GemmArgs &a, uint32_t (&fills)[8]) {
        // B operand of the gate (half 0) and up (half 1) rows: LoRA gate/up
        // reads the up factor from its own map, shifted along K
        auto bmap = [&](int h) { return (C::kLoraSwi && h) ? tmB2 : tmB0; };
        auto bk = [&](int h, int k0) { return (C::kLoraSwi && h) ? k0 - a.k_shift : k0; };
        // two stacked factors (b2_row0 > 0): B rows from b2_row0 on are rows
        // row - b2_row0 of the second map (no stage straddles b2_row0)
        auto bsplit = [&](const CUtensorMap *&m, int row) {
            if (!C::kSwiGLU && a.b2_row0 > 0 && row >= a.b2_row0) {
                m = tmB2;
                return row - a.b2_row0;
            }
            return row;
        };
        const CUtensorMap *tmB = tmB0;
        static_assert(C::NRAW <= 8 && C::NSTAGE <= 8, "fill bookkeeping");
        uint32_t s = 0, ph = 0;
        const int nstage = C::kI8 ? C::NRAW : C::NSTAGE;
        const Segs sp = seg_plan(c);
        for (int si = 0; si < sp.total; ++si) {
            const Seg sg = seg_at(c, sp, si);
            int mb, nb;
            tile_coords(c, sg.tile, mb, nb);
            const int row_a = mb * C::kTileRows + (int)c.rank * C::BM;
            const int kb_end = sg.kb1 + lora_kblocks(c, sg);
            for (int kb = sg.kb0; kb < kb_end; ++kb) {
                if (C::kLoraFused && kb >= sg.kb1) {
                    // a LoRA k-block: its t and B tiles go straight into the fp16
                    // operand slot, copied by the converter group that owns the
                    // k-block (it alone knows when the slot is free); the raw slot
                    // is passed on empty, to keep the two rings in step
                    if (!mbar_wait(&c.bar->raw_empty[s], ph ^ 1u, c.w, kSiteTmaEmpty)) return;
                    mbar_arrive(&c.bar->raw_full[s]);
                } else if (C::kI8) {
                    if (!mbar_wait(&c.bar->raw_empty[s], ph ^ 1u, c.w, kSiteTmaEmpty)) return;
                    uint64_t *full = &c.bar->raw_full[s];
                    uint8_t *ra = c.raw + s * C::kRawStage;
                    uint8_t *rb = ra + C::kRawA;
                    const int k0 = kb * 64;
                    mbar_arrive_expect_tx(full, C::kRawStage);
                    tma_load_2d(ra, tmA, k0, row_a, full);
                    if (C::kSwiGLU && !PAIR) {
                        tma_load_2d(rb, tmB, k0, b_row(c, a, nb, 0), full);
                        tma_load_2d(rb + (BN / 2) * 64, tmB, k0, b_row(c, a, nb, 1), full);
                    } else {
                        tma_load_2d(rb, tmB, k0, b_row(c, a, nb, (int)c.rank), full);
                    }
                } else {
                    if (!wait_pair(&c.bar->empty[s], ph ^ 1u, c, kSiteTmaEmpty)) return;
                    uint8_t *sa = c.stage + s * C::kStage;
                    uint8_t *sb = sa + C::kAStage;
                    const int k0 = kb * C::BK;
                    if (PAIR) {
                        // both CTAs' copies complete on the leader's barrier
                        const uint32_t lfull = leader_addr(&c.bar->full[s]);
                        if (c.rank == 0) mbar_arrive_expect_tx(&c.bar->full[s], 2 * C::kStage);
                        tma_load_2d_pair(sa, tmA, k0, row_a, lfull);
                        const CUtensorMap *mb_ = bmap((int)c.rank);
                        const int br = bsplit(mb_, b_row(c, a, nb, (int)c.rank));
                        tma_load_2d_pair(sb, mb_, bk((int)c.rank, k0), br, lfull);
                    } else {
                        uint64_t *full = &c.bar->full[s];
                        mbar_arrive_expect_tx(full, C::kStage);
                        tma_load_2d(sa, tmA, k0, row_a, full);
                        if (C::kSwiGLU) {
                            tma_load_2d(sb, bmap(0), bk(0, k0), b_row(c, a, nb, 0), full);
                            tma_load_2d(sb + (BN / 2) * 128, bmap(1), bk(1, k0), b_row(c, a, nb, 1), full);
                        } else {
                            const CUtensorMap *mb_ = tmB;
                            const int br = bsplit(mb_, b_row(c, a, nb, 0));
                            tma_load_2d(sb, mb_, k0, br, full);
                        }
                    }
                }
                fills[s] = ph | 2u;  // bit 1: stage filled at least once; bit 0: parity
                if (++s == (uint32_t)nstage) { s = 0; ph ^= 1u; }
            }
        }
    }

    // Before the CTA exits: wait (time-limited) until every copy issued into
    // each stage has landed, so no TMA write targets a finished CTA.  In pair
    // mode the native copies of both CTAs complete on the leader's barriers,
    // so the leader waits for them (the pair then meets at a cluster barrier).
    static __device__ void drain_copies(const Ctx &c, const uint32_t (&fills)[8], unsigned int *st) {
        if (PAIR && !C::kI8 && c.rank != 0) return;
        const int nstage = C::kI8 ? C::NRAW : C::NSTAGE;
        for (int s = 0; s < nstage; ++s) {
            if (!(fills[s] & 2u)) continue;
            uint64_t *full = C::kI8 ? &c.bar->raw_full[s] : &c.bar->full[s];
            mbar_wait_drain(full, fills[s] & 1u, 200000000ull, st);
        }
    }

    // Fused LoRA, one converter lane, once fp16 operand slot cs is free: copy
    // the LoRA k-block kin of this CTA's tile number ktile into it (the tile's
    // t rows and B-factor rows, bf16, 64 of K, already in the MMA's swizzled
    // layout) by TMA, wait for the bytes to land, then arrive for the whole
    // converter group on the slot's "full" barrier and release raw slot rs.
    // Returns false if the copy did not land in time.
    static __device__ bool lora_copy(const Ctx &c, const GemmArgs &a, uint32_t cs, uint32_t rs, int ktile,
                                     int kin) {
        int mb, nb;
        tile_coords(c, c.slot + ktile * c.nslots, mb, nb);
        const int row_a = mb * C::kTileRows + (int)c.rank * C::BM;
        uint8_t *sa = c.stage + cs * C::kStage;
        uint8_t *sb = sa + C::kAStage;
        const int k0 = 64 * (kin - c.nkb);
        uint64_t *lb = &c.bar->ltma[cs];
        const uint64_t tok = mbar_arrive_expect_tx_token(lb, C::kAStage + C::kLoraBRows * 128);
        tma_load_2d(sa, c.tmC, lora_tcol(a, nb) + k0, row_a, lb);
        if (C::kSwiGLU) {
            // t's first r_pad columns (the gate adapter's) meet the gate
            // factor's rows, the rest the up factor's; a pair splits the
            // tile's BN/2 rows of either factor by halves
            const int rp = c.nl * 32;
            const bool up = k0 >= rp;
            const int brow = nb * (BN / 2) + (PAIR ? (int)c.rank * C::kLoraBRows : 0);
            tma_load_2d(sb, up ? c.tmB2 : c.tmD, up ? k0 - rp : k0, brow, lb);
        } else {
            tma_load_2d(sb, c.tmD, k0, b_row(c, a, nb, (int)c.rank), lb);
        }
        // the copy must land before anyone may read or release the slot,
        // also when another role has given up (hence no abort check)
        if (!mbar_wait_token(lb, tok, 200000000ull, c.w.status, kSiteConvEmpty)) {
            *c.w.abort = 1;
            return false;
        }
        mbar_arrive_n(&c.bar->full[cs], C::kGroupWarps);
        mbar_arrive_n(&c.bar->raw_empty[rs], C::kGroupWarps);
        return true;
    }

    // ---------------------------------------------------------------- converters
    // Each converter thread owns the same 16-byte raw pieces in every k-block:
    // piece = ctid & 3 of rows (ctid >> 2) + S j (A rows 0..127, then B rows),
    // where S = threads / 4 is a multiple of 8, so the 128-byte swizzle phase
    // (row & 7) of a thread's rows is constant and all shared addresses are a
    // per-thread base plus compile-time offsets.
    static __device__ void converter(const Ctx &c, const GemmArgs &a, int ctid_all) {
        constexpr int kThr = (C::kI8 ? C::kGroupWarps : 2) * 32;  // native ops never call this
        constexpr int kG = C::kI8 ? C::kConvGroups : 1;
        constexpr int kRows = C::BM + C::kBRows;
        constexpr int kPer = (kRows * 4 + kThr - 1) / kThr;     // the last task may be partial
        static_assert(!C::kI8 || (kThr / 4) % 8 == 0, "constant swizzle phase");
        constexpr uint32_t kSrcStep = (kThr / 4) * 64, kDstStep = (kThr / 4) * 128;
        const int group = ctid_all / kThr, ctid = ctid_all - group * kThr;
        const int row0 = ctid >> 2, piece = ctid & 3, phase = row0 & 7;
        const uint32_t src0 = (uint32_t)(row0 * 64 + piece * 16);
        const uint32_t dst0 = (uint32_t)(row0 * 128 + (((2 * piece) ^ phase) << 4));
        const uint32_t dst1 = (uint32_t)(row0 * 128 + (((2 * piece + 1) ^ phase) << 4));
        const uint32_t raw_base = smem_u32(c.raw), stage_base = smem_u32(c.stage);
        const int lane = threadIdx.x & 31;
        // this CTA's k-blocks in order, over all its segments: its whole tiles,
        // then (stream-K) its run of the remaining tiles' k-blocks
        const int whole_end = sk_of(c) ? sk_tail0(c) : c.num_tiles;
        // k-blocks per whole tile (fused LoRA: the tile's INT8 k-blocks, then its
        // bf16 LoRA k-blocks, which the producer has already placed by TMA)
        const int per = c.nkb + (C::kLoraFused ? c.nl : 0);
        int total = (c.slot < whole_end ? (whole_end - 1 - c.slot) / c.nslots + 1 : 0) * per;
        if (sk_of(c) && c.slot < sk_of(c)) total += sk_bound(c, c.slot + 1) - sk_bound(c, c.slot);
        uint32_t rs = (uint32_t)group, rph = 0, cs = (uint32_t)group, cph = 0;
        int kin = group;   // fused LoRA: the k-block's index within its tile
        int ktile = 0;     // and its tile's index in this CTA's tile sequence
        while (C::kLoraFused && kin >= per) { kin -= per; ++ktile; }
        for (int kidx = group; kidx < total; kidx += kG) {
            if (!mbar_wait(&c.bar->raw_full[rs], rph, c.w, kSiteConvRaw)) return;
            if (C::kLoraFused && kin >= c.nkb) {
                // a LoRA k-block: every warp of the group waits for the slot to be
                // free, as for an INT8 k-block (each warp's successive waits on the
                // ring's "empty" barriers must stay at most NSTAGE k-blocks apart,
                // or a parity wait could pass a phase two behind); then one lane
                // copies the tile's t rows and B-factor rows (bf16, 64 of K,
                // already in the MMA's swizzled layout) into it by TMA, waits for
                // them to land, and arrives for the whole group
                if (!wait_pair(&c.bar->empty[cs], cph ^ 1u, c, kSiteConvEmpty)) return;
                bool ok = true;
                if (ctid == 0) ok = lora_copy(c, a, cs, rs, ktile, kin);
                __syncwarp();
                if (!__shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0)) return;
                rs += kG;
                if (rs >= (uint32_t)C::NRAW) { rs -= C::NRAW; rph ^= 1u; }
                cs += kG;
                if (cs >= (uint32_t)C::NSTAGE) { cs -= C::NSTAGE; cph ^= 1u; }
                kin += kG;
                while (kin >= per) { kin -= per; ++ktile; }
                continue;
            }
            if (!wait_pair(&c.bar->empty[cs], cph ^ 1u, c, kSiteConvEmpty)) return;
            const uint32_t src = raw_base + rs * C::kRawStage + src0;
            const uint32_t dst = stage_base + cs * C::kStage;
            constexpr int kBatch = kPer >= 4 ? 4 : kPer;  // loads in flight per thread
#pragma unroll
            for (int j0 = 0; j0 < kPer; j0 += kBatch) {
                uint4 w[kBatch];
#pragma unroll
                for (int j = 0; j < kBatch; ++j)
                    if (j0 + j < kPer && row0 + (kThr / 4) * (j0 + j) < kRows)
                        w[j] = lds128(src + (j0 + j) * kSrcStep);
#pragma unroll
                for (int j = 0; j < kBatch; ++j) {
                    if (j0 + j >= kPer || row0 + (kThr / 4) * (j0 + j) >= kRows) continue;
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
            // the group's next k-block is kG ahead in both rings (kG <= ring sizes)
            rs += kG;
            if (rs >= (uint32_t)C::NRAW) { rs -= C::NRAW; rph ^= 1u; }
            cs += kG;
            if (cs >= (uint32_t)C::NSTAGE) { cs -= C::NSTAGE; cph ^= 1u; }
            if (C::kLoraFused) {
                kin += kG;
                while (kin >= per) { kin -= per; ++ktile; }
            }
        }
    }

    // Pair mode, INT8, peer CTA: once this CTA's converters have filled an
    // operand stage, tell the leader with one cluster-scope arrive (the
    // converters themselves only arrive on the local barrier).  The stage's
    // data is this CTA's own shared memory, already written and fenced to the
    // async proxy by the converters before their local arrive, which this
    // thread has observed; the leader's tensor-core reads of it are issued only
    // after this arrive lands, so a relaxed arrive suffices.
    static __device__ void forwarder(const Ctx &c) {
        uint32_t s = 0, ph = 0;
        const Segs sp = seg_plan(c);
        for (int si = 0; si < sp.total; ++si) {
            const Seg sg = seg_at(c, sp, si);
            const int kb_end = sg.kb1 + lora_kblocks(c, sg);
            for (int kb = sg.kb0; kb < kb_end; ++kb) {
                if (!mbar_wait(&c.bar->full[s], ph, c.w, kSiteMmaFull)) return;
                arrive_cluster_relaxed(leader_addr(&c.bar->full[s]));
                if (++s == (uint32_t)C::NSTAGE) { s = 0; ph ^= 1u; }
            }
        }
    }

    // ---------------------------------------------------------------- MMA issuer
    static __device__ void mma_issuer(const Ctx &c) {
        constexpr uint32_t afmt = (OP == kOpBF16) ? 1u : 0u;  // F16 / BF16 / E4M3
        constexpr uint32_t idesc = idesc_f32acc(afmt, afmt, C::kTileRows, BN);
        uint32_t s = 0, ph = 0, acc = 0, aph = 0;
        if (c.force_timeout) {
            mbar_wait(&c.bar->never, 0, c.w, kSiteMmaFull);  // runs out; sets the abort flag
            return;
        }
        const Segs sp = seg_plan(c);
        for (int si = 0; si < sp.total; ++si) {
            const Seg sg = seg_at(c, sp, si);
            for (int kb0 = sg.kb0; kb0 < sg.kb1; kb0 += c.chunk) {
                const int kb1 = min(sg.kb1, kb0 + c.chunk);
                if (!wait_pair(&c.bar->acc_empty[acc], aph ^ 1u, c, kSiteMmaAccEmpty)) return;
                tc_fence_after();
                const uint32_t d = c.tmem + acc * BN;
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!wait_pair(&c.bar->full[s], ph, c, kSiteMmaFull)) return;
                    tc_fence_after();
                    const uint32_t sa = smem_u32(c.stage + s * C::kStage);
                    const uint32_t sb = sa + C::kAStage;
#pragma unroll
                    for (int k = 0; k < C::kMmaPerKBlock; ++k) {
                        const uint64_t ad = sdesc_sw128(sa + 32 * k);
                        const uint64_t bd = sdesc_sw128(sb + 32 * k);
                        const uint32_t accum = (kb > kb0 || k > 0) ? 1u : 0u;
                        if (PAIR) {
                            if (OP == kOpF8) mma2_f8(d, ad, bd, idesc, accum);
                            else mma2_f16(d, ad, bd, idesc, accum);
                        } else {
                            if (OP == kOpF8) mma_f8(d, ad, bd, idesc, accum);
                            else mma_f16(d, ad, bd, idesc, accum);
                        }
                    }
                    if (PAIR) mma2_commit_both(&c.bar->empty[s]);
                    else mma_commit(&c.bar->empty[s]);
                    if (++s == (uint32_t)C::NSTAGE) { s = 0; ph ^= 1u; }
                }
                if (PAIR) mma2_commit_both(&c.bar->acc_full[acc]);
                else mma_commit(&c.bar->acc_full[acc]);
                if (++acc == (uint32_t)C::kAccBufs) { acc = 0; aph ^= 1u; }
            }
            const int nl = lora_kblocks(c, sg);
            if (C::kLoraFused && nl > 0) {
                // the tile's LoRA chunk: t B^T with bf16 operands into a fresh
                // accumulator, which the epilogue adds to the rounded base values.
                // Gate/up: the first nl/2 k-blocks sum the gate adapter into the
                // gate half of the columns, the rest the up adapter into the up half
                constexpr uint32_t idesc_l = idesc_f32acc(1u, 1u, C::kTileRows, C::kSwiGLU ? BN / 2 : BN);
                if (!wait_pair(&c.bar->acc_empty[acc], aph ^ 1u, c, kSiteMmaAccEmpty)) return;
                tc_fence_after();
                for (int j = 0; j < nl; ++j) {
                    const bool up = C::kSwiGLU && 2 * j >= nl;
                    const int j0 = up ? nl / 2 : 0;   // the half's first k-block
                    const uint32_t d = c.tmem + acc * BN + (up ? BN / 2 : 0);
                    if (!wait_pair(&c.bar->full[s], ph, c, kSiteMmaFull)) return;
                    tc_fence_after();
                    const uint32_t sa = smem_u32(c.stage + s * C::kStage);
                    const uint32_t sb = sa + C::kAStage;
#pragma unroll
                    for (int k = 0; k < C::kMmaPerKBlock; ++k) {
                        const uint64_t ad = sdesc_sw128(sa + 32 * k);
                        const uint64_t bd = sdesc_sw128(sb + 32 * k);
                        const uint32_t accum = (j > j0 || k > 0) ? 1u : 0u;
                        if (PAIR) mma2_f16(d, ad, bd, idesc_l, accum);
                        else mma_f16(d, ad, bd, idesc_l, accum);
                    }
                    if (PAIR) mma2_commit_both(&c.bar->empty[s]);
                    else mma_commit(&c.bar->empty[s]);
                    if (++s == (uint32_t)C::NSTAGE) { s = 0; ph ^= 1u; }
                }
                if (PAIR) mma2_commit_both(&c.bar->acc_full[acc]);
                else mma_commit(&c.bar->acc_full[acc]);
                if (++acc == (uint32_t)C::kAccBufs) { acc = 0; aph ^= 1u; }
            }
        }
    }

    // ---------------------------------------------------------------- epilogue
    // TMEM column (within one accumulator buffer) of this thread's chunk j.
    static __device__ __forceinline__ int chunk_col(int j, int half) {
        if (C::kSwiGLU) {
            constexpr int kHalfChunks = C::kChunks32 / 2;
            return j < kHalfChunks ? half * (BN / 2 / C::kParts) + 32 * j
                                   : BN / 2 + half * (BN / 2 / C::kParts) + 32 * (j - kHalfChunks);
        }
        return half * (BN / C::kParts) + 32 * j;
    }

    // The fused SwiGLU's silu: the fast form for INT8 (399 against 410 us on
    // the 1502-token gate/up shape), the IEEE form for FP8, where the fast one
    // measured slower (103 against 100 us).
    static __device__ __forceinline__ float silu(float g, float u) {
        if constexpr (OP == kOpI8) return silu_mul_fast(g, u);
        else return silu_mul_ieee(g, u);
    }

    // Finish 32 consecutive output columns n0.. of one row from 32 fp32
    // accumulator values (for SwiGLU: gate values v, up values u).
    static __device__ __forceinline__ void finish32(const GemmArgs &a, int row, bool row_ok,
                                                    int n0, const float (&v)[32],
                                                    const float (&u)[32]) {
        if (!row_ok) return;
        const float sa = C::kScaled ? __ldg(a.sa + row) : 0.0f;
        const bool hb = a.bias != nullptr;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint32_t w[8];
#pragma unroll
            for (int g2 = 0; g2 < 2; ++g2) {
                const int g = 2 * h + g2, n = n0 + 8 * g;
                float y[8];
                if (n >= a.N) {   // N % 8 == 0: whole groups in or out
#pragma unroll
                    for (int i = 0; i < 8; ++i) y[i] = 0.0f;
                } else if (C::kScaled) {
                    float sb[8], bb[8];
                    load_cols8(a.sb, a.bias, n, sb, bb);
#pragma unroll
                    for (int i = 0; i < 8; ++i) y[i] = scale_bias(v[8 * g + i], sa, sb[i], bb[i], hb);
                    if (EPI == kEpiSwiGLU || EPI == kEpiSwiGLULora) {
                        load_cols8(a.sb, a.bias, a.n_half + n, sb, bb);
#pragma unroll
                        for (int i = 0; i < 8; ++i) y[i] = silu(y[i], scale_bias(u[8 * g + i], sa, sb[i], bb[i], hb));
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
#pragma unroll
                for (int i = 0; i < 4; ++i) w[4 * g2 + i] = pack_bf16x2(y[2 * i], y[2 * i + 1]);
            }
            store_bf16x16(a, row, n0 + 16 * h, w);
        }
    }

    // Fused LoRA, scale/bias: 16 columns n0.. of one row from the exact int32
    // totals and the fp32 LoRA sums: y = bf16(bf16(base) + lora) with base the
    // scale/bias value, the same rounded operations as the INT8 linear
    // followed by the LoRA add's expand.
    static __device__ __forceinline__ void finish16_lora(const GemmArgs &a, int row, int n0, const int32_t *tot,
                                                         const uint32_t (&lv)[16]) {
        const float sa = __ldg(a.sa + row);
        const bool hb = a.bias != nullptr;
        uint32_t w[8];
#pragma unroll
        for (int g = 0; g < 2; ++g) {
            const int n = n0 + 8 * g;
            float y[8];
            if (n < a.N) {   // N % 8 == 0: whole groups in or out
                float sb[8], bb[8];
                load_cols8(a.sb, a.bias, n, sb, bb);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float base = bf16_round(scale_bias(__int2float_rn(tot[8 * g + i]), sa, sb[i], bb[i], hb));
                    y[i] = __fadd_rn(base, __uint_as_float(lv[8 * g + i]));
                }
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) y[i] = 0.0f;
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) w[4 * g + i] = pack_bf16x2(y[2 * i], y[2 * i + 1]);
        }
        store_bf16x16(a, row, n0, w);
    }

    // Fused LoRA, SwiGLU: 16 gate columns n0.. from the gate and up totals and
    // their LoRA sums: g = bf16(bf16(base_g) + lora_g), u likewise, h =
    // bf16(silu(g) * u) -- the rounded operations of the packed INT8 linear,
    // the gate/up LoRA adds and the unfused SwiGLU.
    static __device__ __forceinline__ void finish16_swiglu_lora(const GemmArgs &a, int row, int n0,
                                                                const int32_t *tg, const int32_t *tu,
                                                                const uint32_t (&lg)[16],
                                                                const uint32_t (&lu)[16]) {
        const float sa = __ldg(a.sa + row);
        const bool hb = a.bias != nullptr;
        uint32_t w[8];
#pragma unroll
        for (int g = 0; g < 2; ++g) {
            const int n = n0 + 8 * g;
            float h[8];
            if (n < a.N) {
                float sg[8], bg[8], su[8], bu[8];
                load_cols8(a.sb, a.bias, n, sg, bg);
                load_cols8(a.sb, a.bias, a.n_half + n, su, bu);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float gb = bf16_round(scale_bias(__int2float_rn(tg[8 * g + i]), sa, sg[i], bg[i], hb));
                    const float ub = bf16_round(scale_bias(__int2float_rn(tu[8 * g + i]), sa, su[i], bu[i], hb));
                    const float gv = bf16_round(__fadd_rn(gb, __uint_as_float(lg[8 * g + i])));
                    const float uv = bf16_round(__fadd_rn(ub, __uint_as_float(lu[8 * g + i])));
                    h[i] = silu_mul_fast(gv, uv);
                }
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) h[i] = 0.0f;
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) w[4 * g + i] = pack_bf16x2(h[2 * i], h[2 * i + 1]);
        }
        store_bf16x16(a, row, n0, w);
    }

    // Fused LoRA: finish this thread's row from its int32 totals and the LoRA
    // accumulator at tbase, 16 columns at a time (the accumulator is released
    // once its last columns are in registers).
    static __device__ __forceinline__ void finish_row_lora(const Ctx &c, const GemmArgs &a, int row, bool row_ok,
                                                           int nb, int half, const int32_t *tot, uint32_t tbase,
                                                           uint32_t acc, int lane) {
        if constexpr (C::kSwiGLU) {
            constexpr int kH = C::kChunks32 / 2;   // 32-column chunks of gate (then as many of up)
#pragma unroll
            for (int q = 0; q < 2 * kH; ++q) {
                const int j = q >> 1, o = 16 * (q & 1);
                uint32_t lg[16], lu[16];
                tmem_ld16(tbase + chunk_col(j, half) + o, lg);
                tmem_ld16(tbase + chunk_col(j + kH, half) + o, lu);
                tmem_ld_wait();
                if (q == 2 * kH - 1) release_acc(c, acc, lane);
                if (row_ok)
                    finish16_swiglu_lora(a, row, nb * (BN / 2) + chunk_col(j, half) + o, tot + 32 * j + o,
                                         tot + 32 * (j + kH) + o, lg, lu);
            }
        } else {
#pragma unroll
            for (int q = 0; q < 2 * C::kChunks32; ++q) {
                const int j = q >> 1, o = 16 * (q & 1);
                uint32_t lv[16];
                tmem_ld16(tbase + chunk_col(j, half) + o, lv);
                tmem_ld_wait();
                if (q == 2 * C::kChunks32 - 1) release_acc(c, acc, lane);
                if (row_ok) finish16_lora(a, row, nb * BN + chunk_col(j, half) + o, tot + 32 * j + o, lv);
            }
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

    // Finish this thread's row from its kColsPerThread accumulator values
    // (fp32 bits, or exact int32 totals for INT8).
    template <class T>
    static __device__ __forceinline__ void finish_row(const GemmArgs &a, int row, bool row_ok, int nb,
                                                      int half, const T *acc) {
        auto val = [](T x) -> float {
            if constexpr (sizeof(T) == 4 && T(-1) < T(0)) return __int2float_rn((int32_t)x);
            else return __uint_as_float((uint32_t)x);
        };
        if (EPI == kEpiStoreS32) {
            if constexpr (C::kI8) {
#pragma unroll
                for (int j = 0; j < C::kChunks32; ++j)
                    store_s32(a, row, row_ok, nb * BN + chunk_col(j, half),
                              reinterpret_cast<const int32_t *>(acc) + 32 * j);
            }
        } else if (C::kSwiGLU) {
#pragma unroll
            for (int j = 0; j < C::kChunks32 / 2; ++j) {
                float v[32], u[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    v[i] = val(acc[32 * j + i]);
                    u[i] = val(acc[32 * (j + C::kChunks32 / 2) + i]);
                }
                finish32(a, row, row_ok, nb * (BN / 2) + chunk_col(j, half), v, u);
            }
        } else {
#pragma unroll
            for (int j = 0; j < C::kChunks32; ++j) {
                float v[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = val(acc[32 * j + i]);
                finish32(a, row, row_ok, nb * BN + chunk_col(j, half), v, v);
            }
        }
    }

    // y += acc through TMA.  The CTA's y tile (its BM rows of the tile, BN
    // columns) moves as BN / 64 boxes of 64 columns x BM rows with the 128-byte
    // swizzle: box k of buffer b at epi + b * kYTile + k * BM * 128, row r's
    // 16-byte unit u at r * 128 + ((u ^ (r & 7)) << 4).  Boxes wholly past the
    // tensor's rows or columns are neither loaded nor stored.
    static __device__ __forceinline__ int y_row0(const Ctx &c, int t) {
        int mb, nb;
        tile_coords(c, t, mb, nb);
        return mb * C::kTileRows + (int)c.rank * C::BM;
    }

    static __device__ void y_tile_load(const Ctx &c, const GemmArgs &a, int t, int b) {
        int mb, nb;
        tile_coords(c, t, mb, nb);
        const int r0 = y_row0(c, t), c0 = nb * BN;
        uint64_t *bar = &c.bar->ybar[b];
        int boxes = 0;
        if (r0 < a.M)
            for (int k = 0; k < BN / 64; ++k) boxes += (c0 + 64 * k < a.N) ? 1 : 0;
        if (boxes == 0) {
            mbar_arrive(bar);
            return;
        }
        mbar_arrive_expect_tx(bar, (uint32_t)(boxes * C::BM * 128));
        uint8_t *dst = c.epi + b * C::kYTile;
        for (int k = 0; k < BN / 64; ++k)
            if (c0 + 64 * k < a.N) tma_load_2d(dst + k * C::BM * 128, c.tmC, c0 + 64 * k, r0, bar);
    }

    static __device__ void y_tile_store(const Ctx &c, const GemmArgs &a, int t, int b) {
        int mb, nb;
        tile_coords(c, t, mb, nb);
        const int r0 = y_row0(c, t), c0 = nb * BN;
        if (r0 < a.M) {
            const uint8_t *src = c.epi + b * C::kYTile;
            for (int k = 0; k < BN / 64; ++k)
                if (c0 + 64 * k < a.N) tma_store_2d(c.tmC, src + k * C::BM * 128, c0 + 64 * k, r0);
        }
        bulk_commit();
    }

    // This thread's row (TMEM lane) rl of the tile: y[rl][cols of chunk j] +=
    // acc chunk v, in place in buffer b.
    static __device__ __forceinline__ void add_chunk_smem(const Ctx &c, int b, int rl, int half, int j,
                                                          const uint32_t (&v)[32]) {
        const int col = chunk_col(j, half);          // 32-aligned column within the tile
        const uint32_t box = smem_u32(c.epi) + (uint32_t)(b * C::kYTile) +
                             (uint32_t)((col >> 6) * C::BM * 128) + (uint32_t)rl * 128u;
        const int u0 = (col & 63) >> 3;              // first 16-byte unit of the chunk (0 or 4)
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint32_t addr = box + ((uint32_t)((u0 + q) ^ (rl & 7)) << 4);
            const uint4 w = lds128(addr);
            const uint32_t ow[4] = {w.x, w.y, w.z, w.w};
            float y[8];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                y[2 * k] = __fadd_rn(bf16_lo(ow[k]), __uint_as_float(v[8 * q + 2 * k]));
                y[2 * k + 1] = __fadd_rn(bf16_hi(ow[k]), __uint_as_float(v[8 * q + 2 * k + 1]));
            }
            sts128(addr, pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]), pack_bf16x2(y[4], y[5]),
                   pack_bf16x2(y[6], y[7]));
        }
    }

    // LoRA gate/up + SwiGLU through TMA.  Buffer b holds the tile's base gate
    // columns (boxes 0, 1: g|u columns nb * 128 .. + 127) and up columns (boxes
    // 2, 3: the same columns + n_half), laid out as the y tiles of y += acc; h
    // is written over the gate boxes and stored from there.
    static __device__ void gu_tile_load(const Ctx &c, const GemmArgs &a, int t, int b) {
        int mb, nb;
        tile_coords(c, t, mb, nb);
        const int r0 = y_row0(c, t), g0 = nb * (BN / 2);
        uint64_t *bar = &c.bar->ybar[b];
        int boxes = 0;
        if (r0 < a.M)
            for (int k = 0; k < 2; ++k) boxes += (g0 + 64 * k < a.N) ? 2 : 0;
        if (boxes == 0) {
            mbar_arrive(bar);
            return;
        }
        mbar_arrive_expect_tx(bar, (uint32_t)(boxes * C::BM * 128));
        uint8_t *dst = c.epi + b * C::kYTile;
        for (int k = 0; k < 2; ++k) {
            if (g0 + 64 * k >= a.N) continue;
            tma_load_2d(dst + k * C::BM * 128, c.tmC, g0 + 64 * k, r0, bar);
            tma_load_2d(dst + (2 + k) * C::BM * 128, c.tmC, a.n_half + g0 + 64 * k, r0, bar);
        }
    }

    static __device__ void h_tile_store(const Ctx &c, const GemmArgs &a, int t, int b) {
        int mb, nb;
        tile_coords(c, t, mb, nb);
        const int r0 = y_row0(c, t), g0 = nb * (BN / 2);
        if (r0 < a.M) {
            const uint8_t *src = c.epi + b * C::kYTile;
            for (int k = 0; k < 2; ++k)
                if (g0 + 64 * k < a.N) tma_store_2d(c.tmD, src + k * C::BM * 128, g0 + 64 * k, r0);
        }
        bulk_commit();
    }

    // This thread's row rl: g = bf16(yg + acc_g), u = bf16(yu + acc_u),
    // h = bf16(silu(g) * u) for the 32 gate columns of part p (and the matching
    // up columns), in place of the gate values in buffer b.  The same rounded
    // operations as the LoRA add followed by the unfused SwiGLU kernel.
    static __device__ __forceinline__ void lora_swiglu_smem(const Ctx &c, int b, int rl, int p,
                                                            const uint32_t (&vg)[32],
                                                            const uint32_t (&vu)[32]) {
        const int col = 32 * p;                      // gate column within the tile's 128
        const uint32_t base = smem_u32(c.epi) + (uint32_t)(b * C::kYTile) + (uint32_t)rl * 128u;
        const uint32_t gbox = base + (uint32_t)((col >> 6) * C::BM * 128);
        const uint32_t ubox = gbox + (uint32_t)(2 * C::BM * 128);
        const int u0 = (col & 63) >> 3;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint32_t off = (uint32_t)((u0 + q) ^ (rl & 7)) << 4;
            const uint4 gw4 = lds128(gbox + off), uw4 = lds128(ubox + off);
            const uint32_t gw[4] = {gw4.x, gw4.y, gw4.z, gw4.w}, uw[4] = {uw4.x, uw4.y, uw4.z, uw4.w};
            float h[8];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float g_lo = bf16_round(__fadd_rn(bf16_lo(gw[k]), __uint_as_float(vg[8 * q + 2 * k])));
                const float g_hi = bf16_round(__fadd_rn(bf16_hi(gw[k]), __uint_as_float(vg[8 * q + 2 * k + 1])));
                const float u_lo = bf16_round(__fadd_rn(bf16_lo(uw[k]), __uint_as_float(vu[8 * q + 2 * k])));
                const float u_hi = bf16_round(__fadd_rn(bf16_hi(uw[k]), __uint_as_float(vu[8 * q + 2 * k + 1])));
                h[2 * k] = silu_mul_fast(g_lo, u_lo);
                h[2 * k + 1] = silu_mul_fast(g_hi, u_hi);
            }
            sts128(gbox + off, pack_bf16x2(h[0], h[1]), pack_bf16x2(h[2], h[3]), pack_bf16x2(h[4], h[5]),
                   pack_bf16x2(h[6], h[7]));
        }
    }

    static __device__ __forceinline__ void release_acc(const Ctx &c, uint32_t acc, int lane) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
            if (PAIR) arrive_cluster(leader_addr(&c.bar->acc_empty[acc]));
            else mbar_arrive(&c.bar->acc_empty[acc]);
        }
    }

    // Stream-K: a piece of a tile.  Each epilogue warp owns the int32 sums of
    // 32 rows x kColsPerThread columns: it stores them in its block of the
    // workspace, and the warp that arrives last on the block's counter adds
    // the other pieces' blocks to its own sums and finishes the rows.  The
    // sums are exact integers, so the result is the same whatever the split.
    // Returns whether this warp finishes the rows.
    static __device__ __forceinline__ int sk_block(const Ctx &c, int q, int tile, int e) {
        const int first = sk_bound(c, q) >= (tile - sk_tail0(c)) * c.nkb ? 0 : 1;
        return ((q * 2 + first) * 2 + (int)c.rank) * C::kEpiWarps + e;
    }
    // (T = int32_t: exact integer sums, in any order; T = uint32_t: the fp32
    // bit patterns of an FP8 tile's K parts, added in K order)
    template <class T>
    static __device__ bool sk_combine(const Ctx &c, const GemmArgs &a, const Seg &sg, int e, int lane,
                                      T (&tot)[C::kColsPerThread]) {
        constexpr int kV = C::kColsPerThread / 4;   // int4 per lane per block
        static_assert(32 * kV * 16 == 16384, "workspace block");
        {
            int4 *mine = a.sk_ws + (int64_t)sk_block(c, c.slot, sg.tile, e) * (32 * kV) + lane;
#pragma unroll
            for (int j = 0; j < kV; ++j)
                mine[j * 32] = make_int4((int)tot[4 * j], (int)tot[4 * j + 1], (int)tot[4 * j + 2],
                                         (int)tot[4 * j + 3]);
        }
        __threadfence();
        __syncwarp();
        const int v_first = (sg.tile - sk_tail0(c)) * c.nkb;
        const int q0 = sk_owner(c, v_first), q1 = sk_owner(c, v_first + c.nkb - 1);
        int *cnt = a.sk_cnt + (sg.tile * 2 + (int)c.rank) * 8 + e;
        int old = 0;
        if (lane == 0) old = atomicAdd(cnt, 1);
        old = __shfl_sync(0xFFFFFFFFu, old, 0);
        if (old != q1 - q0) return false;
        __threadfence();
        if constexpr (!(sizeof(T) == 4 && T(-1) < T(0))) {
            // fp32 parts: summed in K order from the workspace, this piece's
            // own included, as a whole tile sums its chunks
            {
                const int4 *o = a.sk_ws + (int64_t)sk_block(c, q0, sg.tile, e) * (32 * kV) + lane;
#pragma unroll
                for (int j = 0; j < kV; ++j) {
                    const int4 v = __ldcg(o + j * 32);
                    tot[4 * j] = (T)v.x;
                    tot[4 * j + 1] = (T)v.y;
                    tot[4 * j + 2] = (T)v.z;
                    tot[4 * j + 3] = (T)v.w;
                }
            }
#pragma unroll 1
            for (int q = q0 + 1; q <= q1; ++q) {
                const int4 *o = a.sk_ws + (int64_t)sk_block(c, q, sg.tile, e) * (32 * kV) + lane;
#pragma unroll
                for (int j = 0; j < kV; ++j) {
                    const int4 v = __ldcg(o + j * 32);
                    const int vs[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        tot[4 * j + i] =
                            __float_as_uint(__fadd_rn(__uint_as_float(tot[4 * j + i]), __int_as_float(vs[i])));
                }
            }
            if (lane == 0) atomicExch(cnt, 0);   // zero again for the next launch
            return true;
        }
#pragma unroll 1
        for (int q = q0; q <= q1; ++q) {
            if (q == c.slot) continue;
            const int4 *o = a.sk_ws + (int64_t)sk_block(c, q, sg.tile, e) * (32 * kV) + lane;
#pragma unroll
            for (int j = 0; j < kV; ++j) {
                const int4 v = __ldcg(o + j * 32);
                tot[4 * j] += v.x;
                tot[4 * j + 1] += v.y;
                tot[4 * j + 2] += v.z;
                tot[4 * j + 3] += v.w;
            }
        }
        if (lane == 0) atomicExch(cnt, 0);   // zero again for the next launch
        return true;
    }

    static __device__ void epilogue(const Ctx &c, const GemmArgs &a) {
        int yiter = 0, yloads = 0;
        epilogue_tiles(c, a, yiter, yloads);
        if constexpr (EPI == kEpiAddBF16 || C::kLoraSwi) {
            const int e = (int)(threadIdx.x >> 5) - C::kEpiWarp0, lane = threadIdx.x & 31;
            if (e == 0 && lane == 0) {
                // every TMA store has finished before the CTA's shared memory goes
                // away, and a y load still in flight (after an abort) has landed
                bulk_wait_all();
                for (int k = yiter; k < yloads; ++k)
                    mbar_wait_drain(&c.bar->ybar[k % C::kYBufs], (uint32_t)(k / C::kYBufs) & 1u, 200000000ull,
                                    a.status);
            }
        }
    }

    // yiter: y tiles finished; yloads: y tile loads issued (y += acc only).
    static __device__ void epilogue_tiles(const Ctx &c, const GemmArgs &a, int &yiter, int &yloads) {
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
        const int e = warp - C::kEpiWarp0, quad = warp & 3, half = e >> 2;
        const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
        uint32_t acc = 0, aph = 0;
        const Segs sp = seg_plan(c);
        for (int si = 0; si < sp.total; ++si) {
            const Seg sg = seg_at(c, sp, si);
            const int t = sg.tile;
            int mb, nb;
            tile_coords(c, t, mb, nb);
            const int row = mb * C::kTileRows + (int)c.rank * C::BM + quad * 32 + lane;
            const bool row_ok = row < a.M;
            if constexpr (C::kI8) {
                int32_t tot[C::kColsPerThread];
#pragma unroll
                for (int i = 0; i < C::kColsPerThread; ++i) tot[i] = 0;
                for (int kb0 = sg.kb0; kb0 < sg.kb1; kb0 += c.chunk) {
                    if (!wait_pair(&c.bar->acc_full[acc], aph, c, kSiteEpiAccFull)) return;
                    tc_fence_after();
                    const uint32_t tbase = c.tmem + acc * BN + lane_off;
#pragma unroll
                    for (int j = 0; j < C::kChunks32; ++j) {
                        uint32_t r[32];
                        tmem_ld32(tbase + chunk_col(j, half), r);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 32; ++i) tot[32 * j + i] += __float2int_rn(__uint_as_float(r[i]));
                    }
                    release_acc(c, acc, lane);
                    if (++acc == (uint32_t)C::kAccBufs) { acc = 0; aph ^= 1u; }
                }
                // the tile's exact int32 accumulators are complete (stream-K:
                // once the last piece to arrive has added the others)
                if constexpr (C::kLoraFused) {
                    if (lora_kblocks(c, sg) > 0) {
                        if (!wait_pair(&c.bar->acc_full[acc], aph, c, kSiteEpiAccFull)) return;
                        tc_fence_after();
                        finish_row_lora(c, a, row, row_ok, nb, half, tot, c.tmem + acc * BN + lane_off, acc, lane);
                        if (++acc == (uint32_t)C::kAccBufs) { acc = 0; aph ^= 1u; }
                    } else {
                        finish_row(a, row, row_ok, nb, half, tot);
                    }
                } else if (sg.part < 0 || sk_combine(c, a, sg, e, lane, tot)) {
                    finish_row(a, row, row_ok, nb, half, tot);
                }
            } else if constexpr (C::kLoraSwi) {
                // base g|u tiles by TMA through the ring (kYBufs - 1 tiles ahead),
                // h computed in place over the gate columns, stored by TMA after a
                // bounded epilogue rendezvous
                const int b = yiter % C::kYBufs;
                if (e == 0 && lane == 0) {
                    // the ring: at the CTA's first tile, load its first kYBufs - 1
                    // tiles; then, each tile, load the one kYBufs - 1 ahead into the
                    // buffer whose last tenant (tile yiter - 1) has had its store read out
                    if (yiter == 0)
                        for (int i = 0; i < C::kYBufs - 1 && t + i * c.nslots < c.num_tiles; ++i) {
                            gu_tile_load(c, a, t + i * c.nslots, i);
                            ++yloads;
                        }
                    const int tn = t + (C::kYBufs - 1) * c.nslots;
                    if (tn < c.num_tiles) {
                        bulk_wait_read_all();
                        gu_tile_load(c, a, tn, (yiter + C::kYBufs - 1) % C::kYBufs);
                        ++yloads;
                    }
                }
                if (!wait_pair(&c.bar->acc_full[acc], aph, c, kSiteEpiAccFull)) return;
                tc_fence_after();
                if (!mbar_wait(&c.bar->ybar[b], (uint32_t)(yiter / C::kYBufs) & 1u, c.w, kSiteEpiAccFull)) return;
                const uint32_t tbase = c.tmem + acc * BN + lane_off;
                uint32_t vg[32], vu[32];
                tmem_ld32(tbase + chunk_col(0, half), vg);
                tmem_ld32(tbase + chunk_col(1, half), vu);
                tmem_ld_wait();
                release_acc(c, acc, lane);
                if (++acc == (uint32_t)C::kAccBufs) { acc = 0; aph ^= 1u; }
                lora_swiglu_smem(c, b, quad * 32 + lane, half, vg, vu);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&c.bar->epi_done);
                if (e == 0 && lane == 0) {
                    if (!mbar_wait(&c.bar->epi_done, (uint32_t)yiter & 1u, c.w, kSiteEpiAccFull)) return;
                    h_tile_store(c, a, t, b);
                }
                ++yiter;
            } else if constexpr (EPI == kEpiAddBF16) {
                // y += acc: the tile's y arrives by TMA through the ring (loaded
                // kYBufs - 1 tiles ahead), each thread adds its accumulator row in
                // place, and the tile leaves by TMA once every epilogue thread is done
                const int b = yiter % C::kYBufs;
                if (e == 0 && lane == 0) {
                    // the ring: at the CTA's first tile, load its first kYBufs - 1
                    // tiles; then, each tile, load the one kYBufs - 1 ahead into the
                    // buffer whose last tenant (tile yiter - 1) has had its store read out
                    if (yiter == 0)
                        for (int i = 0; i < C::kYBufs - 1 && t + i * c.nslots < c.num_tiles; ++i) {
                            y_tile_load(c, a, t + i * c.nslots, i);
                            ++yloads;
                        }
                    const int tn = t + (C::kYBufs - 1) * c.nslots;
                    if (tn < c.num_tiles) {
                        bulk_wait_read_all();
                        y_tile_load(c, a, tn, (yiter + C::kYBufs - 1) % C::kYBufs);
                        ++yloads;
                    }
                }
                if (!wait_pair(&c.bar->acc_full[acc], aph, c, kSiteEpiAccFull)) return;
                tc_fence_after();
                if (!mbar_wait(&c.bar->ybar[b], (uint32_t)(yiter / C::kYBufs) & 1u, c.w, kSiteEpiAccFull)) return;
                const uint32_t tbase = c.tmem + acc * BN + lane_off;
#pragma unroll
                for (int j = 0; j < C::kChunks32; ++j) {
                    uint32_t v[32];
                    tmem_ld32(tbase + chunk_col(j, half), v);
                    tmem_ld_wait();
                    if (j == C::kChunks32 - 1) {
                        release_acc(c, acc, lane);
                        if (++acc == (uint32_t)C::kAccBufs) { acc = 0; aph ^= 1u; }
                    }
                    add_chunk_smem(c, b, quad * 32 + lane, half, j, v);
                }
                fence_proxy_async_smem();   // the tile's smem writes, before the TMA store reads them
                __syncwarp();
                if (lane == 0) mbar_arrive(&c.bar->epi_done);
                if (e == 0 && lane == 0) {
                    if (!mbar_wait(&c.bar->epi_done, (uint32_t)yiter & 1u, c.w, kSiteEpiAccFull)) return;
                    y_tile_store(c, a, t, b);
                }
                ++yiter;
            } else if constexpr (C::kKSplit) {
                // FP8 linear: the tile's (or the stream-K piece's) accumulator
                // chunks, the first as it is, the later K parts added in fp32 in
                // K order; a split tile's parts meet in the workspace, where the
                // piece arriving last sums them all in K order
                uint32_t v[C::kColsPerThread];
                for (int kb0 = sg.kb0; kb0 < sg.kb1; kb0 += c.chunk) {
                    if (!wait_pair(&c.bar->acc_full[acc], aph, c, kSiteEpiAccFull)) return;
                    tc_fence_after();
                    const uint32_t tbase = c.tmem + acc * BN + lane_off;
                    if (kb0 == sg.kb0) {
#pragma unroll
                        for (int j = 0; j < C::kChunks32; ++j)
                            tmem_ld32(tbase + chunk_col(j, half), *reinterpret_cast<uint32_t(*)[32]>(v + 32 * j));
                        tmem_ld_wait();
                    } else {
#pragma unroll
                        for (int j = 0; j < C::kChunks32; ++j) {
                            uint32_t r[32];
                            tmem_ld32(tbase + chunk_col(j, half), r);
                            tmem_ld_wait();
#pragma unroll
                            for (int i = 0; i < 32; ++i)
                                v[32 * j + i] = __float_as_uint(
                                    __fadd_rn(__uint_as_float(v[32 * j + i]), __uint_as_float(r[i])));
                        }
                    }
                    release_acc(c, acc, lane);
                    if (++acc == (uint32_t)C::kAccBufs) { acc = 0; aph ^= 1u; }
                }
                bool whole = sg.part < 0;   // always, where tiles are never split
                if constexpr (C::kStreamK) {
                    if (!whole) whole = sk_combine(c, a, sg, e, lane, v);
                }
                if (whole) finish_row(a, row, row_ok, nb, half, v);
            } else {
                if (!wait_pair(&c.bar->acc_full[acc], aph, c, kSiteEpiAccFull)) return;
                tc_fence_after();
                const uint32_t tbase = c.tmem + acc * BN + lane_off;
                uint32_t v[C::kColsPerThread];
#pragma unroll
                for (int j = 0; j < C::kChunks32; ++j)
                    tmem_ld32(tbase + chunk_col(j, half), *reinterpret_cast<uint32_t(*)[32]>(v + 32 * j));
                tmem_ld_wait();
                release_acc(c, acc, lane);  // the MMA may refill the buffer while this row is finished
                if (++acc == (uint32_t)C::kAccBufs) { acc = 0; aph ^= 1u; }
                finish_row(a, row, row_ok, nb, half, v);
            }
        }
    }
};

template <int OP, int EPI, int BN, bool PAIR>
__global__ void __launch_bounds__(Cfg<OP, EPI, BN, PAIR>::kThreads, 1)
gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
            const __grid_constant__ CUtensorMap tmB2, const __grid_constant__ CUtensorMap tmC,
            const __grid_constant__ CUtensorMap tmD,
            const GemmArgs args) {
    using C = Cfg<OP, EPI, BN, PAIR>;
    using G = Gemm<OP, EPI, BN, PAIR>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t base = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + (((base + 1023u) & ~1023u) - base);
    Barriers *bar = reinterpret_cast<Barriers *>(smem + C::NSTAGE * C::kStage + C::NRAW * C::kRawStage +
                                                 C::kEpiStage);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = PAIR ? cluster_rank() : 0u;

    if (threadIdx.x == 0) {
        const int full_arrivals = C::kFullArrivals + ((PAIR && C::kI8 && rank == 0) ? 1 : 0);
        for (int s = 0; s < C::NSTAGE; ++s) {
            mbar_init(&bar->full[s], full_arrivals);
            mbar_init(&bar->empty[s], 1);
        }
        for (int s = 0; s < C::NRAW; ++s) {
            mbar_init(&bar->raw_full[s], 1);
            mbar_init(&bar->raw_empty[s], C::kGroupWarps);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bar->acc_full[s], 1);
            mbar_init(&bar->acc_empty[s], C::kAccEmptyArrivals);
        }
        mbar_init(&bar->drain, 1);
        for (int i = 0; i < C::kYBufs; ++i) mbar_init(&bar->ybar[i], 1);
        if (C::kLoraFused)
            for (int i = 0; i < C::NSTAGE; ++i) mbar_init(&bar->ltma[i], 1);
        mbar_init(&bar->epi_done, C::kEpiWarps);
        mbar_init(&bar->never, 1);
        bar->abort = 0;
        bar->sk = C::kStreamK ? args.sk : 0;
        bar->sk_tail0 = args.sk_tail0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        if (C::kLoraSwi || (C::kLoraFused && C::kSwiGLU)) tma_prefetch_desc(&tmB2);
        if (EPI == kEpiAddBF16 || C::kLoraSwi || C::kLoraFused) tma_prefetch_desc(&tmC);
        if (C::kLoraSwi || C::kLoraFused) tma_prefetch_desc(&tmD);
    }
    if (warp == 1) {
        if (PAIR) {
            // both CTAs of the pair issue the allocation; it pairs up across the
            // two CTAs and returns the same columns in each
            asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;"
                         ::"r"(smem_u32(&bar->tmem_slot)), "r"(C::kTmemCols) : "memory");
            asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
        } else {
            tmem_alloc(&bar->tmem_slot, C::kTmemCols);
            tmem_relinquish();
        }
    }
    tc_fence_before();
    __syncthreads();
    if (PAIR) cluster_sync();  // both CTAs' barriers and TMEM are set up
    tc_fence_after();
    // the set-up above touches no global memory; everything after may read
    // what the stream's previous kernels wrote
    pdl_wait();

    typename G::Ctx c;
    c.stage = smem;
    c.raw = smem + C::NSTAGE * C::kStage;
    c.epi = smem + C::NSTAGE * C::kStage + C::NRAW * C::kRawStage;   // 1024-aligned
    c.tmC = &tmC;
    c.tmD = &tmD;
    c.tmB2 = &tmB2;
    c.bar = bar;
    const uint32_t own_tmem = bar->tmem_slot;
    if (PAIR) {
        uint32_t lt;
        asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(lt) : "r"(leader_addr(&bar->tmem_slot)));
        c.tmem = lt;
    } else {
        c.tmem = own_tmem;
    }
    if (args.dbg && threadIdx.x == 0) {
        args.dbg[2 * blockIdx.x] = (int)own_tmem;
        args.dbg[2 * blockIdx.x + 1] = (int)c.tmem;
    }
    c.rank = rank;
    c.slot = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
    c.nslots = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;
    c.num_m = (args.M + C::kTileRows - 1) / C::kTileRows;
    c.num_n = (args.N + C::kOutColsPerTile - 1) / C::kOutColsPerTile;
    c.num_tiles = c.num_m * c.num_n;
    c.nkb = C::kI8 ? (args.K + 63) / 64 : (args.K + C::BK - 1) / C::BK;
    c.n_fastest = args.n_fastest;
    c.band_m = (args.band_m > 0 && args.band_m < c.num_m) ? args.band_m : c.num_m;

    c.force_timeout = args.force_timeout == 1 || (args.force_timeout >= 2 && args.force_timeout - 2 == c.slot);
    c.nl = C::kLoraFused ? args.lora_nkb : 0;
    c.chunk = C::kI8 ? C::kChunkKBlocks
                     : ((C::kKSplit && c.nkb >= C::kKSplitMinKBlocks) ? (c.nkb + C::kKParts - 1) / C::kKParts
                                                                       : (1 << 30));
    c.w.limit_ns = args.wait_limit_ns;
    c.w.abort = &bar->abort;
    c.w.status = args.status;

    uint32_t fills[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    const bool issues_mma = !PAIR || rank == 0;
    // FP8 SwiGLU (16 epilogue warps; 20 launched at 96 registers): the control
    // warpgroup (TMA producer, MMA issuer) hands registers to the epilogue
    // warps, 4 x 32 x 56 + 16 x 32 x 104 = 60,416 of 61,440 (removes the
    // epilogue's spill; the 1502 x 24576 x 4096 call 104.0 -> 102.4 us)
    constexpr bool kF8Split = OP == kOpF8 && C::kEpiWarps == 16 && C::kEpiWarp0 == 4;
    // FP8 linear and LoRA x A^T (8 epilogue warps; 12 launched at 168
    // registers), whose epilogue holds a tile row's running sum of the K parts
    // while it reads the next part: FP8 4 x 32 x 56 + 8 x 32 x 224 = 64,512
    // of 64,512; bf16 4 x 32 x 80 + 8 x 32 x 208 = 63,488 (its TMA producer,
    // which also serves stacked B factors, spilled at 56 and 64)
    constexpr bool kKSplitRegs = C::kKSplit && C::kEpiWarps == 8 && C::kEpiWarp0 == 4;
    if (warp < C::kEpiWarp0) {
        // INT8: control and converter warps hand registers to the epilogue
        // warps, which hold the int32 totals
        if (C::kI8) asm volatile("setmaxnreg.dec.sync.aligned.u32 64;");
        if (kF8Split || (kKSplitRegs && OP == kOpF8)) asm volatile("setmaxnreg.dec.sync.aligned.u32 56;");
        if (kKSplitRegs && OP == kOpBF16) asm volatile("setmaxnreg.dec.sync.aligned.u32 80;");
        if (warp == 0) {
            if (lane == 0) {
                G::producer(c, &tmA, &tmB, &tmB2, args, fills);
                G::drain_copies(c, fills, args.status);
            }
        } else if (warp == 1) {
            if (lane == 0 && issues_mma) {
                G::mma_issuer(c);
                // wind down: wait until every MMA issued by this thread completed
                if (PAIR) mma2_commit_local(&bar->drain);
                else mma_commit(&bar->drain);
                mbar_wait_drain(&bar->drain, 0, 200000000ull, args.status);
            } else if (lane == 0 && PAIR && C::kI8) {
                G::forwarder(c);
            }
        } else if (C::kI8 && warp < 2 + C::kConvWarps) {
            G::converter(c, args, threadIdx.x - 64);
        }
    } else {
        if (C::kI8) asm volatile("setmaxnreg.inc.sync.aligned.u32 192;");
        if (kF8Split) asm volatile("setmaxnreg.inc.sync.aligned.u32 104;");
        if (kKSplitRegs && OP == kOpF8) asm volatile("setmaxnreg.inc.sync.aligned.u32 224;");
        if (kKSplitRegs && OP == kOpBF16) asm volatile("setmaxnreg.inc.sync.aligned.u32 208;");
        G::epilogue(c, args);
    }
    // this thread's role is done: the stream's next kernel may be scheduled
    // (signalling at the start instead measured slower on the long INT8
    // GEMMs' steps)
    pdl_launch_dependents();
    tc_fence_before();
    __syncthreads();
    if (PAIR) {
        if (bar->abort) {  // let copies still signalling the other CTA land first
            const uint64_t t0 = globaltimer_ns();
            while (globaltimer_ns() - t0 < 2000000ull) {
            }
        }
        cluster_sync();
    }
    if (warp == 1) {
        tc_fence_after();
        if (PAIR)
            asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(own_tmem),
                         "r"(C::kTmemCols) : "memory");
        else
            tmem_dealloc(own_tmem, C::kTmemCols);
    }
}

// Row blocks per band of the M-fastest tile order: as many as keep the band's
// A rows (the activations) within 24 MB of L2, so that they are read from DRAM
// once while the weight tiles stream past; bands of even size.  Without bands
// a launch whose activations exceed L2 re-reads them for every column block
// (24,032 x 34,816 x 5,120 INT8: 17.8 GB of DRAM reads).  The 24,032-token
// layer step with bands of 16 / 24 / 40 / 64 / 96 MB: 11.83 / 11.84 / 11.87 /
// 11.97 / 12.01 ms (12.59 unbanded).
inline int band_rows(int num_m, int tile_rows, int64_t K, int a_bytes) {
    const int64_t per = (int64_t)tile_rows * K * a_bytes;
    int64_t band = ((int64_t)24 << 20) / (per > 0 ? per : 1);
    if (band < 1) band = 1;
    if (band >= num_m) return num_m;
    const int64_t nbands = (num_m + band - 1) / band;
    return (int)((num_m + nbands - 1) / nbands);
}

// Every row of the output starts on a 32-byte boundary (bf16 outputs): the
// epilogue may store 16 columns of a row at once.
inline int out_rows_v32(const GemmArgs &a) {
    return ((reinterpret_cast<uintptr_t>(a.out) & 31u) == 0 && a.ldo % 16 == 0) ? 1 : 0;
}

// k-blocks per tile of a launch (INT8: 64 of K; bf16: 64; FP8: 128)
inline int64_t nkb_of_op(int op, int64_t K) { return op == kOpF8 ? (K + 127) / 128 : (K + 63) / 64; }

// Programmatic dependent launch for a GEMM whose CTAs (pairs) each run at
// most 128 k-blocks: there the previous kernel's tail and this one's launch
// and set-up are a visible share of the time (the 1,502-token FP8 layer step
// 272 -> 260 us, the 298-token linear 34 -> 31 us), while the long INT8
// GEMMs measured slower with it (the 24,032-token layer step +0.7%).
inline bool short_launch(int tiles, int64_t nkb, int ctas) {
    return ctas > 0 && (int64_t)tiles * nkb <= 128 * (int64_t)ctas;
}

template <int OP, int EPI, int BN, bool PAIR>
int launch_one(const Operand &A, const Operand &B, const GemmArgs &args, int num_sms,
               cudaStream_t st, const Operand *B2 = nullptr) {
    using C = Cfg<OP, EPI, BN, PAIR>;
    const CUtensorMapDataType dt =
        (OP == kOpBF16) ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
    // INT8: raw 64-byte rows, no swizzle (converters re-lay them out);
    // native: 128-byte rows in the 128-byte swizzle the MMA descriptors expect.
    const uint32_t box_k = C::kI8 ? 64u : (uint32_t)C::BK;
    const CUtensorMapSwizzle sw = C::kI8 ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B;
    CUtensorMap ta, tb;
    int rc = internal_make_tmap(&ta, dt, A.base, A.inner, A.rows, A.pitch, box_k, C::BM, sw);
    if (rc) return rc;
    rc = internal_make_tmap(&tb, dt, B.base, B.inner, B.rows, B.pitch, box_k,
                            C::kSwiGLU ? BN / 2 : C::kBRows, sw);
    if (rc) return rc;
    CUtensorMap tb2 = tb, tc = tb, td = tb;
    if (EPI == kEpiAddBF16) {   // y tiles: 64-column boxes of BM rows, 128-byte swizzle
        rc = internal_make_tmap(&tc, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, args.out, (uint64_t)args.N,
                                (uint64_t)args.M, (uint64_t)args.ldo * 2, 64, C::BM,
                                CU_TENSOR_MAP_SWIZZLE_128B);
        if (rc) return rc;
    }
    if (C::kLoraSwi) {          // base g|u tiles in, h tiles out, the same boxes
        rc = internal_make_tmap(&tc, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, args.aux, 2 * (uint64_t)args.n_half,
                                (uint64_t)args.M, (uint64_t)args.ld_aux * 2, 64, C::BM,
                                CU_TENSOR_MAP_SWIZZLE_128B);
        if (rc) return rc;
        rc = internal_make_tmap(&td, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, args.out, (uint64_t)args.N,
                                (uint64_t)args.M, (uint64_t)args.ldo * 2, 64, C::BM,
                                CU_TENSOR_MAP_SWIZZLE_128B);
        if (rc) return rc;
    }
    if (C::kLoraFused) {   // t rows (A of the LoRA chunk) and the B factor(s), bf16, 64 of K per box
        rc = internal_make_tmap(&tc, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, args.lora_t, (uint64_t)args.lora_ldt,
                                (uint64_t)args.M, (uint64_t)args.lora_ldt * 2, 64, C::BM,
                                CU_TENSOR_MAP_SWIZZLE_128B);
        if (rc) return rc;
        const uint32_t brows = C::kLoraBRows;
        rc = internal_make_tmap(&td, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, args.lora_b, (uint64_t)args.lora_r,
                                (uint64_t)args.N, (uint64_t)args.lora_r * 2, 64, brows,
                                CU_TENSOR_MAP_SWIZZLE_128B);
        if (rc) return rc;
        if (C::kSwiGLU) {   // the up factor
            rc = internal_make_tmap(&tb2, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, args.lora_b2, (uint64_t)args.lora_r,
                                    (uint64_t)args.N, (uint64_t)args.lora_r * 2, 64, brows,
                                    CU_TENSOR_MAP_SWIZZLE_128B);
            if (rc) return rc;
        }
    }
    if (C::kLoraSwi) {
        if (!B2) return internal_cuda_error(cudaErrorInvalidValue, "LoRA gate/up needs the up factor");
        rc = internal_make_tmap(&tb2, dt, B2->base, B2->inner, B2->rows, B2->pitch, box_k, BN / 2, sw);
        if (rc) return rc;
    } else if (args.b2_row0 > 0) {   // a second factor stacked below the first
        if (!B2 || C::kSwiGLU || args.b2_row0 % C::kBRows != 0)
            return internal_cuda_error(cudaErrorInvalidValue, "stacked B operands");
        rc = internal_make_tmap(&tb2, dt, B2->base, B2->inner, B2->rows, B2->pitch, box_k, C::kBRows, sw);
        if (rc) return rc;
    }
    auto kern = gemm_kernel<OP, EPI, BN, PAIR>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return internal_cuda_error(e, "gemm smem attribute");
    const int num_m = (args.M + C::kTileRows - 1) / C::kTileRows;
    const int num_n = (args.N + C::kOutColsPerTile - 1) / C::kOutColsPerTile;
    const int tiles = num_m * num_n;
    if (PAIR) {
        // persistent pairs: no more than can be resident at once
        static int max_pairs = -1;
        if (max_pairs < 0) {
            cudaLaunchConfig_t cfg = {};
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = 2;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.blockDim = dim3(C::kThreads, 1, 1);
            cfg.dynamicSmemBytes = C::kSmemBytes;
            cfg.stream = st;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            // on the whole device, whatever SM budget the first call had
            int dev = 0, all_sms = num_sms;
            if (cudaGetDevice(&dev) == cudaSuccess)
                cudaDeviceGetAttribute(&all_sms, cudaDevAttrMultiProcessorCount, dev);
            cfg.gridDim = dim3(2 * (all_sms / 2), 1, 1);
            int n = 0;
            e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
            max_pairs = (e == cudaSuccess && n > 0) ? n : all_sms / 2;
        }
        // the pairs this launch may use: the SM budget leaves the rest free
        const int cap = std::min(max_pairs, num_sms / 2);
        int pairs = tiles < cap ? tiles : cap;
        GemmArgs la = args;
        la.out_v32 = out_rows_v32(args);
        la.sk = 0;
        la.sk_tail0 = 0;
        la.band_m = band_rows(num_m, C::kTileRows, args.K, OP == kOpBF16 ? 2 : 1);
        const int nkb_k = (args.K + C::BK - 1) / C::BK;
        if (C::kStreamK && C::kKSplit && args.sk_ws && args.sk_cnt) {
            // FP8 linear with K parts: when the tiles left after the whole
            // waves fit kKParts times in the pairs, each runs as its parts (its
            // own accumulator chunks, cut by K alone) on kKParts pairs, so the
            // last wave takes a part's time: pair p < kKParts R runs part
            // p % kKParts of tail tile p / kKParts.
            const int tail0 = (tiles / cap) * cap;
            const int rest = tiles - tail0;
            if (nkb_k >= C::kKSplitMinKBlocks && nkb_k % C::kKParts == 0 && rest > 0 &&
                C::kKParts * rest <= cap && tiles <= kSkMaxTiles &&
                args.sk_ws_bytes >= (int64_t)cap * kSkBytesPerPair) {
                la.sk = C::kKParts * rest;
                la.sk_tail0 = tail0;
                pairs = tail0 > 0 ? cap : la.sk;
            }
        } else if (C::kStreamK && args.sk_ws && args.sk_cnt) {
            // Stream-K where the last wave of whole tiles would leave more
            // than 8% of the pairs' time idle (the GEMM time follows the count
            // of waves: 1502 x 5120 x 17408 and 1502 x 6400 x 17408 both take
            // 206 us unsplit).  The whole waves stay whole tiles (running pairs
            // then share weight tiles in L2, as unsplit); the R tiles left are
            // dealt as k-block runs of at least 16 k-blocks to up to every
            // pair, and the workspace must hold every pair's two pieces.  A
            // launch of less than one wave stays unsplit (300 x 6144 x 5120:
            // 53.5 us unsplit, 55.6 us with every tile split; 298 x 2048 x 2048
            // 28.4 against 31.2 us) unless it keeps under an eighth of the
            // pairs busy (200 x 2048 x 8192, 8 tiles: 59.4 -> 45.2 us; 130 x
            // 1024 x 4096, 4 tiles: 39.4 -> 35.1 us).
            const int nkb = (args.K + 63) / 64;
            const int64_t waves = (tiles + cap - 1) / cap;
            const double fill = (double)tiles / (double)(waves * cap);
            const int tail0 = tiles >= cap ? (tiles / cap) * cap : 0;
            const int64_t rest = (int64_t)(tiles - tail0) * nkb;
            // runs of at least 16 k-blocks, or 8 when a launch of under an
            // eighth of a wave is split (small M, long K)
            const int minrun = tail0 > 0 ? C::kChunkKBlocks : 8;
            const int p2 = (int)std::min<int64_t>(cap, rest / minrun);
            // (the device splits runs with 32-bit products of a slot index and
            // the remaining k-block count)
            const bool fits32 = rest * (int64_t)cap < ((int64_t)1 << 32);
            if (fill < 0.92 && (tail0 > 0 || 8 * tiles <= cap) && p2 > tiles - tail0 &&
                tiles <= kSkMaxTiles && fits32 &&
                args.sk_ws_bytes >= (int64_t)cap * kSkBytesPerPair) {
                la.sk = p2;
                la.sk_tail0 = tail0;
                pairs = tail0 > 0 ? cap : p2;
            }
        }
        e = launch_kernel(kern, dim3(2 * pairs), dim3(C::kThreads), C::kSmemBytes, st, 2,
                          short_launch(tiles, nkb_of_op(OP, args.K) + (C::kLoraFused ? args.lora_nkb : 0), pairs), ta, tb, tb2, tc, td, la);
    } else {
        const int grid = tiles < num_sms ? tiles : num_sms;
        GemmArgs la = args;
        la.out_v32 = out_rows_v32(args);
        la.band_m = band_rows(num_m, C::kTileRows, args.K, OP == kOpBF16 ? 2 : 1);
        e = launch_kernel(kern, dim3(grid), dim3(C::kThreads), C::kSmemBytes, st, 1,
                          short_launch(tiles, nkb_of_op(OP, args.K) + (C::kLoraFused ? args.lora_nkb : 0), grid), ta, tb, tb2, tc, td, la);
    }
    if (e != cudaSuccess) return internal_cuda_error(e, "gemm launch");
    return 0;
}

}  // namespace

bool gemm_uses_pair(int bn, int M, int num_sms) { return bn == 256 && M > 128 && num_sms >= 2; }

int lora_shrink_width(int64_t M, int64_t N, int num_sms, int64_t split) {
    // Wide CTA-pair tiles whenever they apply, although narrower tiles fill
    // the last wave better: on 24,032 x 5120 -> 256, 256-wide pair tiles took
    // 91 us against 94 us for 128-wide and 130 us for 64-wide single tiles,
    // which stage the same x rows in two or four SMs and read more operand
    // bytes per product.  Small ranks keep tiles no wider than the rank.
    if (N > 128 && gemm_uses_pair(256, (int)M, num_sms) && (split == 0 || split % 128 == 0)) return 256;
    int bn = N <= 64 ? 64 : (N <= 128 ? 128 : 256);
    while (split > 0 && bn > 64 && split % bn != 0) bn /= 2;   // no tile straddles the split
    return bn;
}

int launch_gemm(int op, int epi, int bn, const Operand &A, const Operand &B, const GemmArgs &args,
                int num_sms, cudaStream_t st, const Operand *B2) {
    const bool pair = gemm_uses_pair(bn, args.M, num_sms);
#define CLEF_GEMM(OPV, EPIV, BNV)                                                        \
    return pair ? launch_one<OPV, EPIV, BNV, true>(A, B, args, num_sms, st)              \
                : launch_one<OPV, EPIV, BNV, false>(A, B, args, num_sms, st)
    if (op == kOpI8 && bn == 256) {
        if (epi == kEpiScaleBias) CLEF_GEMM(kOpI8, kEpiScaleBias, 256);
        if (epi == kEpiSwiGLU) CLEF_GEMM(kOpI8, kEpiSwiGLU, 256);
        if (epi == kEpiStoreS32) CLEF_GEMM(kOpI8, kEpiStoreS32, 256);
        if (epi == kEpiScaleBiasLora) CLEF_GEMM(kOpI8, kEpiScaleBiasLora, 256);
        if (epi == kEpiSwiGLULora) CLEF_GEMM(kOpI8, kEpiSwiGLULora, 256);
    } else if (op == kOpF8 && bn == 256) {
        if (epi == kEpiScaleBias) CLEF_GEMM(kOpF8, kEpiScaleBias, 256);
        if (epi == kEpiSwiGLU) CLEF_GEMM(kOpF8, kEpiSwiGLU, 256);
    } else if (op == kOpBF16) {
        if (epi == kEpiStoreBF16) {
            if (bn == 64) return launch_one<kOpBF16, kEpiStoreBF16, 64, false>(A, B, args, num_sms, st, B2);
            if (bn == 128) return launch_one<kOpBF16, kEpiStoreBF16, 128, false>(A, B, args, num_sms, st, B2);
            if (bn == 256)
                return pair ? launch_one<kOpBF16, kEpiStoreBF16, 256, true>(A, B, args, num_sms, st, B2)
                            : launch_one<kOpBF16, kEpiStoreBF16, 256, false>(A, B, args, num_sms, st, B2);
        } else if (epi == kEpiAddBF16 && bn == 256) {
            CLEF_GEMM(kOpBF16, kEpiAddBF16, 256);
        } else if (epi == kEpiAddBF16 && bn == 128) {
            return launch_one<kOpBF16, kEpiAddBF16, 128, false>(A, B, args, num_sms, st);
        } else if (epi == kEpiLoraSwiGLU && bn == 256) {
            const bool pr = gemm_uses_pair(bn, args.M, num_sms);
            return pr ? launch_one<kOpBF16, kEpiLoraSwiGLU, 256, true>(A, B, args, num_sms, st, B2)
                      : launch_one<kOpBF16, kEpiLoraSwiGLU, 256, false>(A, B, args, num_sms, st, B2);
        }
    }
#undef CLEF_GEMM
    return internal_cuda_error(cudaErrorInvalidValue, "no GEMM instantiation for this operand/epilogue/width");
}

}  // namespace clef
