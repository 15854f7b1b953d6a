/*
 * clef.h -- C ABI of the GB300 (sm_103a) W8A8 quantized projection library.
 *
 * The library computes the quantized decoder linear projections of a
 * Clef-style single-pass decision backbone: a per-token activation
 * quantizer (block-128 Walsh-Hadamard rotation, absmax scale, symmetric INT8
 * codes; FP8-e4m3 dynamic variant), W8A8 GEMMs whose epilogues fuse the
 * row x column scales, the bias and, for packed gate/up weights, the SwiGLU
 * product, and the runtime LoRA add.  Every step runs in hand-written CUDA
 * kernels on the caller's stream.
 *
 * Conventions shared by every entry point:
 *  - Pointers are DEVICE pointers to memory the caller owns (clef_copy_sm
 *    also takes page-locked host memory); the library never allocates, frees
 *    or synchronises inside these calls.
 *  - Matrices are row-major.  x/activations are [M][K]; weights are [N][K]
 *    (output-channel major, the Linear convention), so the GEMMs contract
 *    both operands along their contiguous K axis.
 *  - bf16 tensors hold IEEE bfloat16 bit patterns (uint16_t storage); e4m3
 *    tensors hold OCP FP8 E4M3 codes (finite variant, max 448).
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls
 *    launch asynchronously and return; results are ready when the stream is.
 *  - Return value: CLEF_OK, or an error code from argument checks made on
 *    the host before anything is launched (nothing is launched on error),
 *    or CLEF_ERR_CUDA when a launch fails.  Device-side waits that exceed
 *    their time limit record CLEF_ERR_TIMEOUT in a library-owned status word
 *    read by clef_poll_status(); the kernels never trap.
 *  - M = 0 is a valid empty call: it returns CLEF_OK without a launch (its
 *    row-indexed pointers may then be null, as those of empty tensors are).
 *  - Inputs are assumed finite; NaN/Inf inputs give unspecified codes.
 *  - Alignment: every tensor base and every row pitch must be a multiple of
 *    16 bytes (TMA and vector-access rule); the checks below state it per
 *    call as the element counts that satisfy it.
 *
 * Sources (web pages; cited by title and section):
 *  [INT8]  "CLEF Calibrated INT8 ConvRot" model card: Benefits (kernels fuse
 *          calibrated scales, biases and MLP SwiGLU) and the note under the
 *          latency table (a CUDA ConvRot activation quantizer feeds integer
 *          GEMMs).
 *  [USAGE] "Loading CLEF INT8" usage notes: fuse_mlp (paired gate/up epilogue
 *          fusion) and gate/up weights packed during loading.
 *  [FP8]   "clef-flash-FP8" model card, Quantization table and the note below
 *          the recipe (FP8 weights per channel, FP8 activations per token,
 *          dynamic; weight scales computed from the weights).
 *  [LORA]  TensorFold pull request 1364, first bullet of the description:
 *          y = bf16(y + bf16(x A^T) B^T), fp32 sums, bf16 add; A (rank, k),
 *          B (n, rank); ranks zero-padded to whole 64-groups; a row's bits
 *          independent of row count and chunking.
 */
#ifndef CLEF_H
#define CLEF_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum clef_status {
    CLEF_OK = 0,
    CLEF_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, bad size or stride */
    CLEF_ERR_UNSUPPORTED = 2,   /* device is not sm_103, or a mode not built */
    CLEF_ERR_CUDA = 3,          /* a CUDA runtime call or launch failed */
    CLEF_ERR_TIMEOUT = 4        /* a device-side wait exceeded its limit */
} clef_status;

typedef enum clef_act_mode {
    CLEF_ACT_INT8_H128 = 0,     /* rotate 128-blocks, s = amax/127, int8 codes */
    CLEF_ACT_FP8_E4M3 = 1,      /* no rotation, s = amax/448, e4m3 codes */
    CLEF_ACT_FP8_E4M3_H128 = 2  /* rotate 128-blocks, then the FP8 codes */
} clef_act_mode;

/*
 * clef_quant_act -- per-token activation quantizer [INT8: latency-table
 * note, "ConvRot activation quantizer"; FP8: Quantization table,
 * "Activations FP8, per-token, dynamic"].  Also the weight quantizer: run on
 * W's N rows it gives the per-output-channel codes and scales.
 *
 * For each row m of x (bf16 [M][K], row pitch ldx elements):
 *   v = x[m] widened to fp32; for the H128 modes each contiguous 128-block of
 *   v is rotated by the orthonormal Walsh-Hadamard butterfly (strides 1, 2,
 *   4, ..., 64, (a+b, a-b) in fp32, then one multiply by fp32(1/sqrt(128)));
 *   amax = max |v|;
 *   INT8:  scale[m] = amax/127, q = clamp(rne(v * (127/amax)), -127, 127);
 *   FP8:   scale[m] = amax/448, q = e4m3_rn_satfinite(v * (448/amax));
 *   an all-zero row gives scale 0 and codes 0.
 * q: int8 or e4m3 [M][K], dense (row pitch K); scale: fp32 [M].
 * Requirements: K > 0, K % 128 == 0 for H128 modes else K % 32 == 0,
 *   K <= 65536, ldx >= K, ldx % 8 == 0; x and q 16-byte aligned, scale 4-byte.
 */
int clef_quant_act(const void *x, int64_t M, int64_t K, int64_t ldx, int mode,
                   void *q, float *scale, void *stream);

/*
 * clef_quant_act_static -- the quantizer with one static scale s for the
 * whole tensor (a calibrated scale [INT8: "calibrated scales" of the
 * Benefits list]) in place of the per-token amax:
 *   v as in clef_quant_act; r = fp32(1 / s);
 *   INT8:  q = clamp(rne(fp32(v * r)), -127, 127)
 *   FP8:   q = e4m3_rn_satfinite(fp32(v * r))   (saturates at +-448)
 *   scale[m] = s for every row, so the GEMM entry points apply unchanged.
 * s must be positive and finite; other arguments and requirements as for
 * clef_quant_act.
 */
int clef_quant_act_static(const void *x, int64_t M, int64_t K, int64_t ldx, int mode,
                          float s, void *q, float *scale, void *stream);

/*
 * clef_w8a8_linear -- W8A8 INT8 linear with the fused scale/bias epilogue
 * [INT8: Benefits, "fuse calibrated scales, biases"].
 *   acc[m][n] = sum_k qx[m][k] * qw[n][k]        (exact int32)
 *   y[m][n]   = bf16(((float)acc * sx[m]) * sw[n] + bias[n])
 * qx: int8 [M][K] dense; sx: fp32 [M]; qw: int8 [N][K] dense; sw: fp32 [N];
 * bias: bf16 [N] or NULL; y: bf16 [M][N], row pitch ldy elements.
 * Requirements: K % 16 == 0, N % 8 == 0, ldy >= N, ldy % 8 == 0; qx, qw,
 * sw, bias and y 16-byte aligned, sx 4-byte.  The
 * library receives bare pointers and cannot check buffer lengths: sx must
 * hold M values and sw and bias N (the packed gate/up calls: 2N), else the
 * kernels read past their ends.
 */
int clef_w8a8_linear(const int8_t *qx, const float *sx, const int8_t *qw, const float *sw,
                     const void *bias, int64_t M, int64_t N, int64_t K,
                     void *y, int64_t ldy, void *stream);

/*
 * clef_w8a8_gateup_swiglu -- INT8 gate/up projection with the paired SwiGLU
 * epilogue [USAGE: fuse_mlp; gate/up packed during loading; INT8: Benefits,
 * "MLP SwiGLU"].  qw_gu: int8 [2N][K] with the gate rows 0..N-1 followed by
 * the up rows N..2N-1; sw_gu, bias_gu: [2N] in the same order (bias may be
 * NULL).  With g, u the unrounded fp32 epilogue values of rows n and N+n:
 *   h[m][n] = bf16(g / (1 + exp(-g)) * u)
 * evaluated in fp32 with the hardware exp2 and reciprocal approximations
 * (the bf16 result is within one ulp of the correctly rounded value).
 * h: bf16 [M][N], row pitch ldh.  Requirements as clef_w8a8_linear.
 */
int clef_w8a8_gateup_swiglu(const int8_t *qx, const float *sx, const int8_t *qw_gu,
                            const float *sw_gu, const void *bias_gu,
                            int64_t M, int64_t N, int64_t K,
                            void *h, int64_t ldh, void *stream);

/*
 * clef_fp8_linear -- FP8 e4m3 W8A8 dynamic linear [FP8: Quantization table,
 * "Weights FP8, per-channel; Activations FP8, per-token, dynamic"].
 *   acc = sum_k qx[m][k] * qw[n][k] in fp32 (tensor-core accumulation order;
 *         for K >= 8192, K is cut into three fixed parts of ceil(ceil(K/128)
 *         / 3) * 128 elements (the last the rest), each summed apart, the
 *         three added in K order, for every M, so that a row's bits never
 *         depend on the call's row count or on a split)
 *   y[m][n] = bf16(((float)acc * sx[m]) * sw[n] + bias[n])
 * qx: e4m3 [M][K]; qw: e4m3 [N][K]; other arguments as clef_w8a8_linear.
 */
int clef_fp8_linear(const void *qx, const float *sx, const void *qw, const float *sw,
                    const void *bias, int64_t M, int64_t N, int64_t K,
                    void *y, int64_t ldy, void *stream);

/*
 * clef_fp8_gateup_swiglu -- the FP8 counterpart of clef_w8a8_gateup_swiglu
 * (the paired SwiGLU epilogue of [USAGE] over the FP8 scheme of [FP8]); its
 * silu uses CUDA expf and a correctly rounded division.
 */
int clef_fp8_gateup_swiglu(const void *qx, const float *sx, const void *qw_gu,
                           const float *sw_gu, const void *bias_gu,
                           int64_t M, int64_t N, int64_t K,
                           void *h, int64_t ldh, void *stream);

/*
 * clef_lora_add -- runtime LoRA add [LORA: y = bf16(y + bf16(x A^T) B^T),
 * fp32 sums and a bf16 add, rank zero-padded to a 64-group].
 *   t[m][j] = bf16(sum_k x[m][k] * A[j][k])  for j < r, 0 for r <= j < r_pad
 *   y[m][n] = bf16((float)y[m][n] + sum_j t[m][j] * B[n][j])   (in place)
 * with r_pad = r rounded up to a multiple of 64.
 * x: bf16 [M][K], row pitch ldx (the unquantized, unrotated input of the
 * projection); A: bf16 [r][K] dense; B: bf16 [N][r] dense;
 * t_scratch: bf16 [M][r_pad] dense, caller-owned scratch that receives t;
 * y: bf16 [M][N], row pitch ldy, read and written.
 * Requirements: K % 8 == 0, r % 8 == 0, 0 < r <= 1024, N % 8 == 0,
 *   ldx >= K, ldx % 8 == 0, ldy >= N, ldy % 8 == 0.
 */
int clef_lora_add(const void *x, int64_t ldx, const void *A, const void *B,
                  int64_t M, int64_t K, int64_t N, int64_t r,
                  void *t_scratch, void *y, int64_t ldy, void *stream);

/*
 * clef_w8a8_linear_lora -- the INT8 linear with the runtime LoRA expand
 * fused into the same GEMM [LORA; INT8: Benefits].  t = bf16(x A^T) comes
 * from a clef_lora_shrink call made before (t's columns past r must be
 * finite); each output tile accumulates t B^T as a last bf16 tensor-core
 * chunk, and its epilogue adds it to the rounded base value, so y is never
 * written and read back between the two:
 *   y[m][n] = bf16(bf16(((float)acc * sx[m]) * sw[n] + bias[n])
 *                  + sum_{j<r} t[m][tcol(n) + j] * B[n][j])
 * -- the same bytes as clef_w8a8_linear followed by clef_lora_expand_add from
 * t + tcol(n).  B: bf16 [N][r] dense (for packed projections, the adapters'
 * B factors stacked in output-column order; zero rows for columns without
 * an adapter).  nseg (0..4) column segments map output columns to t columns:
 * columns below seg_end[i] (and at or above seg_end[i-1]) read t columns
 * seg_tcol[i] .. seg_tcol[i] + r_pad - 1 (r_pad = r rounded up to 64);
 * nseg = 0 means one segment at t column 0.  seg_end increasing, every end
 * but the last a multiple of 256, the last equal to N; seg_tcol multiples of
 * 8 with seg_tcol + r_pad <= ldt.  t: bf16, row pitch ldt (multiple of 8).
 * Other arguments and requirements as clef_w8a8_linear; 0 < r <= 1024,
 * r % 8 == 0.  This call never splits tiles across SMs (no stream-K
 * workspace is used).
 */
int clef_w8a8_linear_lora(const int8_t *qx, const float *sx, const int8_t *qw, const float *sw,
                          const void *bias, int64_t M, int64_t N, int64_t K, const void *t, int64_t ldt,
                          const void *B, int64_t r, int nseg, const int64_t *seg_end,
                          const int64_t *seg_tcol, void *y, int64_t ldy, void *stream);

/*
 * clef_w8a8_gateup_swiglu_lora -- the INT8 gate/up SwiGLU call with the gate
 * and up LoRA adds fused [LORA; USAGE: fuse_mlp]: with t_gu = [x A_gate^T |
 * x A_up^T] from one clef_lora_shrink over the stacked A factors (each padded
 * with zero rows to r_pad),
 *   g = bf16(bf16(gate epilogue value) + sum_j t_gu[m][j] * B_gate[n][j])
 *   u = bf16(bf16(up epilogue value) + sum_j t_gu[m][r_pad + j] * B_up[n][j])
 *   h[m][n] = bf16(silu(g) * u)    (silu as in clef_swiglu_bf16)
 * -- the same bytes as clef_w8a8_linear on the packed weight (bf16 [M][2N])
 * followed by clef_lora_gateup_swiglu, without g and u ever reaching memory.
 * t_gu: bf16 [M][>= 2 r_pad] at pitch ldt (t_gate in columns 0 .. r_pad - 1,
 * t_up in r_pad .. 2 r_pad - 1; columns past r in each must be finite);
 * B_gate, B_up: bf16 [N][r] dense.  Other arguments and requirements as
 * clef_w8a8_gateup_swiglu; 0 < r <= 1024, r % 8 == 0, ldt % 8 == 0.
 */
int clef_w8a8_gateup_swiglu_lora(const int8_t *qx, const float *sx, const int8_t *qw_gu, const float *sw_gu,
                                 const void *bias_gu, int64_t M, int64_t N, int64_t K, const void *t_gu,
                                 int64_t ldt, const void *B_gate, const void *B_up, int64_t r, void *h,
                                 int64_t ldh, void *stream);

/*
 * clef_lora_shrink / clef_lora_expand_add -- the two stages of clef_lora_add
 * as separate calls [LORA], for adapters that share an input: with their A
 * factors stacked (each zero-padded to a multiple of 64 rows) one shrink
 * call reads x once for all of them, and each adapter's expand call reads its
 * own column block of t (t + offset, the shared pitch ldt).  clef_lora_add is
 * exactly clef_lora_shrink into t_scratch (ldt = r_pad) followed by
 * clef_lora_expand_add from it.
 * clef_lora_shrink: t[m][j] = bf16(sum_k x[m][k] * A[j][k]) for j < r_pad
 *   (rows j >= r of A read as zeros, so those columns of t are 0).  The fp32
 *   sum runs in the tensor core's order; for K >= 6144 it is taken as four
 *   fixed parts of ceil(K / 256) x 64 elements (the last the rest), added in
 *   K order, whatever M is, so a row's bits never depend on the call's row
 *   count.  With a workspace bound to the stream (clef_bind_workspace), the
 *   parts of a partly empty last wave of tiles run on several SMs.
 *   x: bf16 [M][K], pitch ldx; A: bf16 [r][K] dense; t: bf16 [M][r_pad],
 *   pitch ldt (only columns 0 .. r_pad - 1 written).
 * clef_lora_expand_add: y[m][n] = bf16((float)y[m][n] + sum_{j<r} t[m][j] * B[n][j])
 *   in place.  t: bf16, columns 0 .. r_pad - 1 read (pitch ldt; columns
 *   r .. r_pad - 1 are multiplied by zeros); B: bf16 [N][r] dense; y: bf16
 *   [M][N], pitch ldy.
 * Requirements: K % 8 == 0, N % 8 == 0, r % 8 == 0, 0 < r <= 4096,
 *   ldx >= K, ldt >= r_pad, ldy >= N, all pitches multiples of 8, every
 *   pointer (t + offset included) 16-byte aligned.
 */
int clef_lora_shrink(const void *x, int64_t ldx, const void *A, int64_t M, int64_t K, int64_t r,
                     void *t, int64_t ldt, void *stream);
int clef_lora_expand_add(const void *t, int64_t ldt, const void *B, int64_t M, int64_t N, int64_t r,
                         void *y, int64_t ldy, void *stream);

/*
 * clef_lora_gateup_swiglu -- runtime LoRA on the gate and up projections
 * [LORA], followed by the MLP product [USAGE], in one pass over the base
 * gate/up values: with t_g = bf16(x A_gate^T) and t_u = bf16(x A_up^T) as in
 * clef_lora_add,
 *   g[m][n] = bf16((float)y_gu[m][n]     + sum_j t_g[m][j] * B_gate[n][j])
 *   u[m][n] = bf16((float)y_gu[m][N + n] + sum_j t_u[m][j] * B_up[n][j])
 *   h[m][n] = bf16(silu(g) * u)   (fp32, silu(g) = g / (1 + exp(-g)) as in
 *                                  clef_swiglu_bf16)
 * -- the same rounded operations as two clef_lora_add calls on the halves of
 * y_gu followed by clef_swiglu_bf16, without writing g and u back.
 * x: bf16 [M][K], row pitch ldx; A_gate, A_up: bf16 [r][K] dense; B_gate,
 * B_up: bf16 [N][r] dense; t_scratch: bf16 [M][2 r_pad] dense scratch
 * (r_pad = r rounded up to 64; receives t_g then t_u); y_gu: bf16 [M][2N]
 * base gate values then up values (the output of clef_w8a8_linear on the
 * packed weight), row pitch ld_gu, read only; h: bf16 [M][N], row pitch ldh.
 * Requirements: K % 8 == 0, r % 8 == 0, 0 < r <= 1024, N % 8 == 0,
 *   ldx >= K, ld_gu >= 2N, ldh >= N, all pitches multiples of 8.
 */
int clef_lora_gateup_swiglu(const void *x, int64_t ldx, const void *A_gate, const void *B_gate,
                            const void *A_up, const void *B_up, int64_t M, int64_t K, int64_t N,
                            int64_t r, void *t_scratch, const void *y_gu, int64_t ld_gu,
                            void *h, int64_t ldh, void *stream);

/*
 * clef_swiglu_bf16 -- the unfused MLP reading (fuse_mlp off in [USAGE]):
 * y_gu holds bf16 gate values in columns 0..N-1 and up values in N..2N-1
 * (row pitch ldg); h[m][n] = bf16(silu(float(g)) * float(u)), silu(g) =
 * g / (1 + exp(-g)) in fp32 with the hardware exp2 and reciprocal
 * approximations (within one bf16 ulp of the correctly rounded value).
 * Requirements: N % 8 == 0, ldg >= 2N, ldg % 8 == 0, ldh >= N, ldh % 8 == 0.
 */
int clef_swiglu_bf16(const void *y_gu, int64_t M, int64_t N, int64_t ldg,
                     void *h, int64_t ldh, void *stream);

/*
 * clef_w8a8_gemm_s32 -- the INT8 GEMM with its raw accumulator as output
 * (acc[m][n] = sum_k qx[m][k] * qw[n][k], exact int32, row pitch ldc),
 * through the same kernel and mainloop as clef_w8a8_linear.  It exists so
 * that the integer accumulators can be compared bit for bit.
 * Requirements: K % 16 == 0, N % 8 == 0, ldc >= N, ldc % 8 == 0.
 */
int clef_w8a8_gemm_s32(const int8_t *qx, const int8_t *qw, int64_t M, int64_t N, int64_t K,
                       int32_t *acc, int64_t ldc, void *stream);

/*
 * clef_lora_add_noalloc -- the same LoRA add as clef_lora_add, without the
 * t_scratch argument, for callers that cannot allocate device memory: a host
 * whose runtime owns a fixed device-memory budget and forbids allocations
 * outside it, a plugin living inside another framework's allocator, or code
 * that must not pay the device-wide synchronisation cudaMalloc/cudaFree can
 * imply.  The pages have no counterpart of this call; it is a library
 * convenience.
 * t lives in a library-owned static device array of 4,194,304 bf16 elements
 * (8 MiB, held by every GPU that loads the library until exit):
 * M * round_up(r, 64) beyond that returns CLEF_ERR_INVALID_ARG.  The call
 * allocates nothing.  Its first call on a device looks up the array's device
 * address (cudaGetSymbolAddress) with that device current; make that first
 * call before any stream capture.  All calls share the array and it keeps the
 * previous call's contents (nothing needs clearing: each call rewrites every
 * element it reads), so calls whose kernels may overlap on the GPU race and
 * must be serialised.  It runs the same launches as clef_lora_add (tile
 * widths, the clef_set_wait_limit_ns limit and the clef_test_force_timeout
 * knob included), so its output bytes equal clef_lora_add's.  Other
 * arguments and requirements as clef_lora_add.
 */
int clef_lora_add_noalloc(const void *x, int64_t ldx, const void *A, const void *B,
                          int64_t M, int64_t K, int64_t N, int64_t r,
                          void *y, int64_t ldy, void *stream);

/*
 * clef_gemm_workspace_bytes / clef_bind_workspace -- optional scratch that
 * lets the INT8 GEMMs (clef_w8a8_linear, clef_w8a8_gemm_s32; M > 128) split
 * tiles across SMs when the last wave of whole 256 x 256 tiles would leave
 * more than 8% of the CTA pairs idle ("stream-K": the whole waves run as
 * whole tiles, the remaining tiles' K is dealt to all pairs in even runs of
 * at least 16 k-blocks of 64 (1,024 K elements; 8 k-blocks, 512 elements,
 * for a launch of under one wave), and the pieces of a tile meet as exact
 * int32 partial sums,
 * so the bytes of every output equal those of an unsplit launch).  The GEMM
 * time follows the number of tile waves (1502 x 5120 x 17408 and 1502 x 6400
 * x 17408 take the same time unsplit), so a shape with a partly empty last
 * wave gains up to the idle fraction.  A launch of less than one wave is
 * split only when its tiles would keep under an eighth of the pairs busy
 * (small M, long K); the gate/up SwiGLU calls never split.  clef_fp8_linear
 * with K >= 8192 sums every tile's K as three fixed parts whatever M is (see
 * there); with a workspace bound, the tiles of a last wave that fits three
 * times in the pairs run as their parts on three pairs each, the same bytes
 * as unsplit.  Other FP8 calls never split.  The LoRA x A^T of
 * clef_lora_shrink, clef_lora_add and clef_lora_gateup_swiglu does the same
 * with four parts for K >= 6144 (see clef_lora_shrink).
 * clef_gemm_workspace_bytes: the size needed on the current device (about
 * 38 MB on a 152-SM GB300), written to *bytes.
 * clef_bind_workspace: binds a caller-owned device buffer of that size to
 * `stream` on the current device (ws = NULL unbinds); INT8 and FP8 linear
 * calls on that stream may then use it, calls on unbound streams never split.  The buffer
 * must be zero-filled when bound; every launch leaves its counter block
 * zeroed again (after a CLEF_ERR_TIMEOUT, refill the buffer with zeros before
 * further use).  Launches that use one buffer must not run concurrently: bind
 * a separate buffer to each stream whose work may overlap.  Binding is host
 * bookkeeping (no stream operation), so it may be done while the stream is
 * being captured into a graph; the graph then keeps the buffer's address.
 * Requirements: ws 16-byte aligned and bytes >= the counter block (the
 * workspace is used for splitting only when bytes >= the size returned);
 * at most 256 bindings.
 */
int clef_gemm_workspace_bytes(int64_t *bytes);
int clef_bind_workspace(void *stream, void *ws, int64_t bytes);

/*
 * clef_mma_peak -- dense tensor-core rate of this device for one instruction
 * route, measured by the library's own microbenchmark (the denominators of
 * the GEMMs' roofline fractions; not part of the projection path):
 *   kind 0: tcgen05.mma kind::f16 with bf16 operands and an fp32 accumulator
 *           (the route of the INT8 GEMMs, whose int8 codes are multiplied
 *           exactly as fp16, and of the LoRA products);
 *   kind 1: tcgen05.mma kind::f8f6f4 with e4m3 operands (the FP8 GEMMs);
 *   kind 2: mma.sync m16n8k32 s8 x s8 -> s32 (the legacy integer route).
 * The tcgen05 kinds run one CTA pair per two SMs issuing 256 x 256 MMAs back
 * to back from shared memory into two TMEM accumulators (no copies); kind 2
 * runs register-operand MMA chains in every warp.  One warm-up launch, then
 * `iters` iterations (4 MMAs of 256 x 256 x 64 (bf16) or x 128 (e4m3) per
 * iteration; 8 m16n8k32 MMAs per warp for kind 2) timed with CUDA events on
 * a private stream; *tflops = 2 x multiply-adds / seconds / 1e12.
 * Synchronises; not for use during stream capture.
 * Requirements: kind in 0..2, 0 < iters <= 2^24.
 */
int clef_mma_peak(int kind, int64_t iters, double *tflops);

/*
 * clef_poll_status -- synchronises the device, then returns and clears the
 * device-side status word (CLEF_OK if no kernel recorded an error).
 */
int clef_poll_status(void);

/*
 * clef_set_wait_limit_ns -- time limit of every device-side wait in kernels
 * launched afterwards (default 1e9 ns).  A wait that exceeds it records
 * CLEF_ERR_TIMEOUT and its kernel winds down and returns.  Test knob.
 */
void clef_set_wait_limit_ns(uint64_t ns);

/*
 * clef_test_force_timeout -- test knob for the device-side failure path.
 * on = 1: the W8A8/FP8/LoRA GEMM kernels launched afterwards make their MMA
 * issuer wait on a barrier that nothing signals; the wait runs out after the
 * clef_set_wait_limit_ns limit, CLEF_ERR_TIMEOUT is recorded in the status
 * word and the kernel winds down (their outputs are then undefined).
 * on = n >= 2: only the CTA (or CTA pair) working through tile-loop slot
 * n - 2 does so, while the others finish their tiles (a stream-K launch then
 * leaves the counters of the tiles that slot shared nonzero: the case
 * clef_bind_workspace's refill rule is for).  0 (default) or negative: off.
 */
void clef_test_force_timeout(int on);

/*
 * clef_set_quant_staging -- which quantizer kernel clef_quant_act launches
 * afterwards.  Two kernels compute the same codes and scales bit for bit: a
 * persistent one that stages rows in shared memory through TMA (for row
 * lengths that are a multiple of 64 and at most 32768) and a one-CTA-per-row
 * one (every row length).  mode 1 (default): the staged kernel for calls of
 * at least 8 rows per SM, where it streams faster; mode 2: the staged kernel
 * wherever the row length allows; mode 0: always the per-row kernel.  Other
 * values are clamped to this range.  The switch exists so that each kernel
 * can be tested and timed.
 */
void clef_set_quant_staging(int mode);

/*
 * clef_set_pdl -- programmatic dependent launch for the kernels the library
 * launches afterwards.  on != 0 (default): each launch carries CUDA's
 * programmatic stream-serialization attribute, so that a kernel's CTAs may be
 * scheduled, and run their set-up (barriers, tensor-memory allocation,
 * descriptor prefetch), while the stream's previous kernel finishes; every
 * kernel waits for the kernels it follows to complete, with their writes
 * visible, before it reads or writes global memory, so results are the same
 * bytes either way.  on == 0: plain stream order.  The switch exists so that
 * both can be tested and timed.
 */
void clef_set_pdl(int on);

/*
 * clef_set_sm_budget -- how many SMs the library's compute launches issued
 * afterwards may fill (GEMMs, LoRA launches, quantizers): sms, rounded down
 * to an even count, or every SM of the device for sms == 0 or sms at least
 * the device's count.  Results are the same bytes under any budget (the
 * tile order and every split follow the shapes, not the SM count; only the
 * number of persistent CTAs changes).  A persistent GEMM CTA takes a whole
 * SM, so work on another stream (clef_copy_sm streaming the next step's
 * inputs) gets SMs only if the budget leaves some free.  Process-wide, like
 * clef_set_pdl; launches captured into a CUDA graph keep the budget that was
 * in force when they were captured.  Stream-K tails (clef_bind_workspace)
 * are dealt over the CTA pairs the budget allows.  Returns
 * CLEF_ERR_INVALID_ARG (budget unchanged) for a negative sms or sms == 1.
 */
int clef_set_sm_budget(int sms);

/*
 * clef_copy_sm -- copy bytes bytes from src to dst with loads and stores
 * issued by ctas CTAs (one per SM; clusters of two where ctas is even)
 * instead of a copy engine.  src and dst are any addresses the device can
 * access: device memory, or page-locked host memory (cudaHostAlloc or
 * cudaHostRegister), read and written through its device mapping.  Pageable
 * host memory returns CLEF_ERR_INVALID_ARG (nothing launched) unless the
 * device reads pageable memory directly (cudaDevAttrPageableMemoryAccess).
 * Copy-engine transfers from page-locked host memory were measured to stall
 * for 20-180 ms, on some GB300 machines about every half second and on others
 * rarely; SM loads over the same link ran at the same rate without stalls on
 * every box tried.  With a budget (clef_set_sm_budget) of the device's SMs
 * less ctas, the copy runs beside the compute launches of another stream.
 * Requirements: dst and src 16-byte aligned, bytes >= 0 and a multiple of
 * 16, 1 <= ctas <= 64, the two ranges disjoint.  Ordered on stream like any
 * kernel; bytes == 0 returns CLEF_OK without a launch.
 */
int clef_copy_sm(void *dst, const void *src, int64_t bytes, int ctas, void *stream);

/* Human-readable name of a status code (static string). */
const char *clef_status_string(int status);

/* Text of the most recent argument or CUDA error seen by this thread's calls
 * (empty if none); valid until the thread's next failing call. */
const char *clef_last_error(void);

/* ABI version of this library (major * 100 + minor). */
int clef_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* CLEF_H */
