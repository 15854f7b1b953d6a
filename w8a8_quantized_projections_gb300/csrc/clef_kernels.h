// clef_kernels.h -- internal launchers shared by the C-ABI layer (abi.cu)
// and the kernel translation units.  Not part of the public ABI.
#pragma once

#include <cstdint>
#include <utility>
#include <cuda.h>
#include <cuda_runtime.h>

namespace clef {

// The library's programmatic-dependent-launch switch (clef_set_pdl).
bool internal_pdl();

// Launch a kernel of the library: cluster_x > 1 launches clusters of that
// many CTAs; with pdl and the library's PDL switch on, the launch carries the
// programmatic stream-serialization attribute, so the kernel's CTAs may be
// scheduled (and run their set-up) while the stream's previous kernel
// finishes.  Every kernel of the library therefore signals its dependents once
// its own work is done (pdl_launch_dependents) and waits for the grids it
// depends on (pdl_wait) before its first access to global memory.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                          int cluster_x, bool pdl, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    unsigned n = 0;
    if (cluster_x > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = (unsigned)cluster_x;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    if (pdl && internal_pdl()) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

enum ActMode : int { kActInt8H128 = 0, kActFp8 = 1, kActFp8H128 = 2 };

// What the quantizer launch needs from the device set-up.  staging: 0 =
// always the one-CTA-per-row kernel; 1 = the persistent TMA-staged kernel for
// calls of at least 8 rows per SM whose row length suits it; 2 = the staged
// kernel wherever the row length suits it.
struct QuantEnv {
    int num_sms;
    unsigned int *status;
    uint64_t wait_limit_ns;
    int staging;
    // static scale (static_r > 0): codes use r = static_r = fp32(1 / static_s)
    // for every row and every row's scale is static_s; 0: per-token amax
    float static_r = 0.0f, static_s = 0.0f;
};

cudaError_t launch_quant_act(int mode, const uint16_t *x, int64_t M, int64_t K, int64_t ldx,
                             uint8_t *q, float *scale, const QuantEnv &env, cudaStream_t st);

// Operand kinds of the tensor-core GEMM.
enum GemmOp : int {
    kOpI8 = 0,    // int8 codes in HBM, widened to fp16 on chip, exact chunked accumulation
    kOpF8 = 1,    // e4m3 codes, kind::f8f6f4
    kOpBF16 = 2,  // bf16 operands, kind::f16
};

// Epilogues.
enum GemmEpi : int {
    kEpiScaleBias = 0,  // y = bf16((acc * sa[m]) * sb[n] + bias[n])
    kEpiSwiGLU = 1,     // h = bf16(silu(g) * u), g/u from the two halves of the tile
    kEpiStoreBF16 = 2,  // t = bf16(acc)
    kEpiAddBF16 = 3,    // y = bf16(float(y) + acc), y read and written
    kEpiStoreS32 = 4,   // acc as int32 (INT8 operands only)
    kEpiLoraSwiGLU = 5, // gate/up LoRA adds then SwiGLU: g = bf16(yg + acc_g),
                        // u = bf16(yu + acc_u), h = bf16(silu(g) * u); yg|yu read
                        // from aux, h written to out (bf16 operands only)
    // INT8 GEMMs with the runtime LoRA expand fused (a last bf16 accumulator
    // chunk per tile, lora = t B^T over the padded rank):
    kEpiScaleBiasLora = 6,  // y = bf16(bf16((acc * sa) * sb + bias) + lora)
    kEpiSwiGLULora = 7,     // g = bf16(bf16(epilogue(gate)) + lora_g), u likewise,
                            // h = bf16(silu(g) * u)
};

// Column segments of a fused LoRA expand: output columns below seg_end[i]
// (and at or above seg_end[i - 1]) read t's columns seg_tcol[i] ..
// seg_tcol[i] + r_pad - 1 (adapters of a packed projection group).
constexpr int kLoraMaxSegs = 4;

struct GemmArgs {
    int M, N, K;             // output rows, output columns (h columns for SwiGLU), depth
    int n_half;              // SwiGLU: row offset of the up half inside the packed B operand
    const float *sa;         // per-row scale [M]
    const float *sb;         // per-column scale (packed order for SwiGLU)
    const uint16_t *bias;    // bf16, may be null
    void *out;               // bf16 or int32 output
    int64_t ldo;             // output row pitch (elements)
    int out_v32;             // bf16 output whose every row starts on a 32-byte
                             // boundary (the launcher sets it)
    unsigned int *status;    // device status word
    uint64_t wait_limit_ns;
    int *dbg;                // optional: per CTA, its own TMEM base and the one it uses
    int force_timeout;       // test knob: 1 = every CTA's MMA issuer waits on a barrier
                             // nothing signals; n >= 2: only the CTA (pair) of tile-loop slot n - 2
    // kEpiLoraSwiGLU: the base gate|up values (bf16 [M][2 * n_half], pitch
    // ld_aux elements), and the K offset of the up half's factor: up rows of
    // the B operand come from the second tensor map at K coordinate k - k_shift
    const void *aux;
    int64_t ld_aux;
    int k_shift;
    // tile order: 0 = M fastest (running CTAs share weight tiles), 1 = N
    // fastest (running CTAs share activation row blocks: LoRA x A^T)
    int n_fastest;
    // M fastest: tiles are ordered in bands of band_m row blocks, all of a
    // band's column blocks before the next band, so that a band's A rows stay
    // in L2 while the weights stream past (0 = one band; the launcher sets it)
    int band_m;
    // kEpiStoreBF16 with two stacked B factors: rows from b2_row0 on come from
    // the second operand (its row b2_row0 less); 0 = one B operand
    int b2_row0;
    // INT8 stream-K (sk > 0): tiles from sk_tail0 on are dealt to the first
    // sk CTA pairs as even runs of k-blocks; pieces of a tile meet in the
    // workspace: sk_cnt holds kSkMaxTiles x 2 x 8 arrival counters (zero
    // between launches), sk_ws the int32 partial sums.  sk_ws_bytes: the
    // partial region's size.  The launcher sets sk and sk_tail0.
    int sk;
    int sk_tail0;
    int *sk_cnt;
    int4 *sk_ws;
    int64_t sk_ws_bytes;
    // fused LoRA expand (kEpiScaleBiasLora, kEpiSwiGLULora): lora_t is t (bf16
    // [M][lora_ldt]), lora_b the B factor (bf16 [N][lora_r]; for SwiGLU the
    // gate factor, the up factor being lora_b2, and t holds t_gate in columns
    // 0 .. r_pad - 1 and t_up after); lora_nkb: bf16 k-blocks of 64 per tile
    // (r_pad / 64, twice that for SwiGLU)
    const void *lora_t;
    int64_t lora_ldt;
    const void *lora_b;
    const void *lora_b2;
    int lora_r;
    int lora_nkb;
    int lora_nseg;
    int lora_seg_end[kLoraMaxSegs];
    int lora_seg_tcol[kLoraMaxSegs];
};

// Stream-K workspace: counters for up to kSkMaxTiles tiles, then per CTA pair
// two pieces x two CTAs x eight epilogue warps x 16 KB of int32 sums.
constexpr int kSkMaxTiles = 4096;
constexpr int64_t kSkCounterBytes = (int64_t)kSkMaxTiles * 2 * 8 * 4;
constexpr int64_t kSkBytesPerPair = 2 * 2 * 8 * 16384;

// A row-major 2-D operand: rows of `inner` elements, `pitch` bytes apart.
struct Operand {
    const void *base;
    uint64_t inner, rows, pitch;
};

// A: [M][K] activation rows, B: [rows][K] weight rows.  Builds the TMA maps for
// the chosen tile mode and launches on st.  bn selects the tile width (256 for
// the W8A8 GEMMs; 64/128/256 for the LoRA rank).  Returns a clef_status code.
int launch_gemm(int op, int epi, int bn, const Operand &A, const Operand &B, const GemmArgs &args,
                int num_sms, cudaStream_t st, const Operand *B2 = nullptr);

// Whether a launch with this width and row count uses CTA pairs.
bool gemm_uses_pair(int bn, int M, int num_sms);

// Tile width (64, 128 or 256) for t = x A^T with N = the padded rank (256
// uses CTA pairs when M > 128).  split > 0: the column where a second
// stacked factor starts, which no tile may straddle.
int lora_shrink_width(int64_t M, int64_t N, int num_sms, int64_t split);

cudaError_t launch_swiglu_bf16(const uint16_t *y_gu, int64_t M, int64_t N, int64_t ldg,
                               uint16_t *h, int64_t ldh, cudaStream_t st);

// Services of abi.cu for other translation units: per-device checks and
// set-up (SM count, status-word address), TMA tensor maps, and the calling
// thread's last-error text.
int internal_device(int *num_sms, unsigned int **status);
// clef_lora_add's two launches (arguments already checked) with t at the
// given dense [M][round_up(r, 64)] scratch: the same tile widths, wait limit
// and test knob as the public call.
int internal_lora_add(const void *x, int64_t ldx, const void *A, const void *B, int64_t M, int64_t K,
                      int64_t N, int64_t r, void *t, void *y, int64_t ldy, cudaStream_t st);
int internal_make_tmap(CUtensorMap *m, CUtensorMapDataType dt, const void *base, uint64_t inner,
                       uint64_t rows, uint64_t pitch_bytes, uint32_t box_inner, uint32_t box_rows,
                       CUtensorMapSwizzle sw);
// rank-dimensional tensor map: dims[0] innermost, strides[i] = byte pitch of
// dimension i + 1, box[i] elements per copy; zero fill outside the tensor.
int internal_make_tmap_nd(CUtensorMap *m, CUtensorMapDataType dt, int rank, const void *base,
                          const uint64_t *dims, const uint64_t *strides, const uint32_t *box,
                          CUtensorMapSwizzle sw);
void internal_set_error(const char *msg);
int internal_cuda_error(cudaError_t e, const char *what);  // records the text, returns CLEF_ERR_CUDA

}  // namespace clef
