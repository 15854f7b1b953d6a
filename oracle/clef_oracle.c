/*
 * clef_oracle.c -- plain, slow CPU oracle for the W8A8 projection path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this file; only the tests, the smoke check and the benchmark's CPU
 * baseline do.  It shares no code, header, table or constant generator with
 * the CUDA path.
 *
 * Every function is the plain definition of one step, written out in the
 * order the method states it, single-threaded, with no blocking or fusion.
 * Build: gcc -O2 -std=c11 -ffp-contract=off (no FMA contraction, IEEE fp32
 * arithmetic rounded to nearest-even after every operation).
 *
 * Sources (web pages, cited by title and section):
 *  - "CLEF Calibrated INT8 ConvRot" model card (terminusresearch/
 *    cloudflare-clef-int8-convrot): Benefits list (CuTeDSL kernels fuse
 *    calibrated scales, biases and MLP SwiGLU) and the note under the latency
 *    table (both INT8 paths quantise activations with a CUDA ConvRot
 *    quantizer before an integer GEMM).
 *  - "Loading CLEF INT8" usage notes: fuse_mlp (paired gate/up epilogue
 *    fusion), gate/up weights packed during loading.
 *  - "clef-flash-FP8" model card, Quantization table: FP8_DYNAMIC, weights
 *    FP8 per channel, activations FP8 per token, dynamic; weight scales are
 *    computed directly from the weights.
 *  - TensorFold pull request 1364 (runtime Clef adapter), first bullet:
 *    y = bf16(y + bf16(x A^T) B^T) with fp32 sums and a bf16 add; A is a
 *    (rank, k) projection and B an (n, rank) one; a rank below a whole
 *    64-group is zero-padded with exact zeros.
 *
 * Readings where the pages are silent (each also stated where it is used):
 *  - ConvRot is named but never defined: it is read as the orthonormal
 *    Sylvester Walsh-Hadamard transform on each contiguous 128-block of a
 *    row, stages of stride 1, 2, 4, ..., 64 with (a+b, a-b) in fp32, then one
 *    fp32 multiply by c = fp32(1/sqrt(128)).
 *  - Per-token scale s = amax/127 (fp32 division); codes use the reciprocal
 *    r = 127/amax (one fp32 division per row) and round-half-even of v*r,
 *    clamped to [-127, 127].  An all-zero row gets s = 0 and codes 0.
 *  - FP8: s = amax/448, r = 448/amax, codes = e4m3 (finite variant, max 448)
 *    round-to-nearest-even with saturation to +-448; the sign of a value that
 *    rounds to zero is kept (negative zero is code 0x80).  Inputs on this
 *    path are finite; an infinity saturates and a NaN gives the NaN code 0x7F.
 *  - Epilogue: y = bf16(((float)acc * s[m]) * sw[n] + bias[n]).
 *  - SwiGLU: g and u are epilogue values before rounding, h = bf16(g / (1 +
 *    expf(-g)) * u); packed weights hold the gate rows first, then the up rows.
 *  - FP8 GEMM sums the exact products; with e4m3 operands and K <= 2^14 the
 *    fp64 running sum is exact (products span 2^-18 .. 2^17.6, sums stay
 *    below 2^32), so acc = fp32(exact sum).
 *  - LoRA: t = bf16(sum_k x*A) and y = bf16(float(y) + fp32(sum_j t*B)); the
 *    sums are taken in fp64 (the fp32 sums the pages name have an unstated
 *    order), which the tests absorb with a derived accumulation bound.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_OK 0
#define ORC_ERR_ARG 1
#define ORC_ERR_OVERFLOW 2
#define ORC_ERR_NOMEM 3

/* ------------------------------------------------------------------ */
/* bf16 storage                                                        */
/* ------------------------------------------------------------------ */

/* bf16 is the top half of an IEEE binary32; widening is exact. */
static float bf16_to_f32(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round a binary32 to bf16, nearest-even.  Inputs are finite in this path. */
static uint16_t f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7F800000u) == 0x7F800000u)          /* inf / nan: keep class */
        return (uint16_t)((u >> 16) | ((u & 0x007FFFFFu) ? 0x40u : 0u));
    uint32_t keep = u >> 16, rest = u & 0xFFFFu;
    if (rest > 0x8000u || (rest == 0x8000u && (keep & 1u)))
        keep += 1u;                                 /* carries into exponent */
    return (uint16_t)keep;
}

/* Round an fp64 value to bf16 in one step, nearest-even (|d| in normal range). */
static uint16_t f64_to_bf16(double d)
{
    if (d == 0.0)
        return signbit(d) ? 0x8000u : 0u;
    int e;
    double f = frexp(fabs(d), &e);          /* |d| = f * 2^e, f in [0.5, 1) */
    double m = ldexp(f, 8);                 /* [128, 256): 8 significant bits */
    double fl = floor(m), fr = m - fl;
    if (fr > 0.5 || (fr == 0.5 && fmod(fl, 2.0) != 0.0))
        fl += 1.0;
    float v = (float)ldexp(fl, e - 8);      /* exact: fl has <= 9 bits */
    if (d < 0)
        v = -v;
    uint32_t u;
    memcpy(&u, &v, sizeof u);
    return (uint16_t)(u >> 16);             /* exact: low half is zero */
}

uint16_t orc_f32_to_bf16(float f) { return f32_to_bf16(f); }
float orc_bf16_to_f32(uint16_t h) { return bf16_to_f32(h); }
uint16_t orc_f64_to_bf16(double d) { return f64_to_bf16(d); }

/* Round half to even to an integer value (|t| < 2^23 here). */
static float rne_int(float t)
{
    float fl = floorf(t);
    float fr = t - fl;                      /* exact for |t| < 2^23 */
    if (fr > 0.5f)
        return fl + 1.0f;
    if (fr < 0.5f)
        return fl;
    return (fmodf(fl, 2.0f) == 0.0f) ? fl : fl + 1.0f;
}

/* ------------------------------------------------------------------ */
/* Block-128 Walsh-Hadamard rotation (the reading of "ConvRot")        */
/* ------------------------------------------------------------------ */

/* Normalisation c = fp32(1/sqrt(128)); its bits are 0x3DB504F3. */
static float wht_c(void) { return (float)(1.0 / sqrt(128.0)); }

/* One 128-block in place: butterfly stages h = 1, 2, 4, ..., 64; at each
 * stage every index i with (i & h) == 0 pairs with i + h and becomes
 * (v[i] + v[i+h], v[i] - v[i+h]) in fp32; then every entry is multiplied
 * by c once.  The stage order is fixed because fp32 rounding depends on it. */
void orc_wht128_f32(float *v)
{
    for (int h = 1; h < 128; h <<= 1)
        for (int i = 0; i < 128; i++)
            if ((i & h) == 0) {
                float a = v[i], b = v[i + h];
                v[i] = a + b;
                v[i + h] = a - b;
            }
    const float c = wht_c();
    for (int i = 0; i < 128; i++)
        v[i] = v[i] * c;
}

/* The same transform in fp64 with the exact normalisation 1/sqrt(128);
 * used only by the tests' orthogonality and invariance checks. */
void orc_wht128_f64(double *v)
{
    for (int h = 1; h < 128; h <<= 1)
        for (int i = 0; i < 128; i++)
            if ((i & h) == 0) {
                double a = v[i], b = v[i + h];
                v[i] = a + b;
                v[i + h] = a - b;
            }
    const double c = 1.0 / sqrt(128.0);
    for (int i = 0; i < 128; i++)
        v[i] = v[i] * c;
}

/* Rotate every 128-block of each bf16 row of x[M][K] (row stride ldx) into
 * fp32 out[M][K] (dense).  K must be a multiple of 128. */
int orc_rotate_rows_f32(const uint16_t *x, int64_t M, int64_t K, int64_t ldx, float *out)
{
    if (M < 0 || K <= 0 || K % 128 != 0 || ldx < K)
        return ORC_ERR_ARG;
    for (int64_t m = 0; m < M; m++) {
        float *v = out + m * K;
        for (int64_t k = 0; k < K; k++)
            v[k] = bf16_to_f32(x[m * ldx + k]);
        for (int64_t b = 0; b < K; b += 128)
            orc_wht128_f32(v + b);
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------ */
/* Per-token symmetric INT8 codes of rotated rows                      */
/* ------------------------------------------------------------------ */

/* Quantise one row of fp32 values v[K] to INT8: amax = max |v| (exact);
 * s = amax / 127; r = 127 / amax; q = clamp(rne(v * r), -127, 127).
 * An all-zero row gives s = 0 and all codes 0. */
static void quant_row_int8(const float *v, int64_t K, int8_t *q, float *s)
{
    float amax = 0.0f;
    for (int64_t k = 0; k < K; k++)
        amax = fmaxf(amax, fabsf(v[k]));
    if (amax == 0.0f) {
        *s = 0.0f;
        memset(q, 0, (size_t)K);
        return;
    }
    *s = amax / 127.0f;
    const float r = 127.0f / amax;
    for (int64_t k = 0; k < K; k++) {
        float t = rne_int(v[k] * r);
        if (t > 127.0f) t = 127.0f;
        if (t < -127.0f) t = -127.0f;
        q[k] = (int8_t)t;
    }
}

/* Activation (or weight-row) quantiser, INT8 with block-128 rotation.
 * x: bf16 [M][K], row stride ldx elements.  q: int8 [M][K] dense.  s: [M]. */
int orc_quant_int8_h128(const uint16_t *x, int64_t M, int64_t K, int64_t ldx,
                        int8_t *q, float *s)
{
    if (M < 0 || K <= 0 || K % 128 != 0 || ldx < K)
        return ORC_ERR_ARG;
    float *v = (float *)malloc((size_t)K * sizeof(float));
    if (!v)
        return ORC_ERR_NOMEM;
    for (int64_t m = 0; m < M; m++) {
        orc_rotate_rows_f32(x + m * ldx, 1, K, ldx, v);
        quant_row_int8(v, K, q + m * K, s + m);
    }
    free(v);
    return ORC_OK;
}

/* ------------------------------------------------------------------ */
/* FP8 e4m3 (finite variant: no infinities, S.1111.111 is NaN)        */
/* ------------------------------------------------------------------ */

/* Value of an e4m3 code: exponent bias 7; e = 0 is subnormal m/8 * 2^-6. */
double orc_e4m3_decode(uint8_t c)
{
    int sgn = c >> 7, e = (c >> 3) & 15, m = c & 7;
    if (e == 15 && m == 7)
        return NAN;
    double mag = (e == 0) ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, e - 7);
    return sgn ? -mag : mag;
}

/* Nearest e4m3 code to an fp32 value, ties to even mantissa, magnitudes
 * beyond 448 (infinities included) saturate to 448 with their sign; NaN gives
 * the NaN code. */
uint8_t orc_e4m3_encode(float f)
{
    if (isnan(f))
        return 0x7F;                              /* the format's NaN, 0 1111 111 */
    uint8_t sgn = signbit(f) ? 0x80 : 0x00;
    double a = fabs((double)f);
    if (a >= 448.0)
        return sgn | 0x7E;                        /* e = 15, m = 6: 448 */
    if (a < ldexp(1.0, -6)) {                     /* subnormal spacing 2^-9 */
        double t = ldexp(a, 9), fl = floor(t), fr = t - fl;
        if (fr > 0.5 || (fr == 0.5 && fmod(fl, 2.0) != 0.0))
            fl += 1.0;                            /* fl == 8 is 2^-6 = code 8 */
        return sgn | (uint8_t)fl;
    }
    int e;
    frexp(a, &e);                                 /* a = f * 2^e, f in [0.5,1) */
    int E = e - 1;                                /* a in [2^E, 2^(E+1)) */
    double t = (ldexp(a, -E) - 1.0) * 8.0;        /* mantissa in [0, 8), exact */
    double fl = floor(t), fr = t - fl;
    if (fr > 0.5 || (fr == 0.5 && fmod(fl, 2.0) != 0.0))
        fl += 1.0;
    int m = (int)fl;
    if (m == 8) {
        m = 0;
        E += 1;
    }
    int be = E + 7;                               /* 1 .. 15 */
    if (be > 15 || (be == 15 && m == 7))
        return sgn | 0x7E;                        /* rounded past 448 */
    return sgn | (uint8_t)((be << 3) | m);
}

static void quant_row_fp8(const float *v, int64_t K, uint8_t *q, float *s)
{
    float amax = 0.0f;
    for (int64_t k = 0; k < K; k++)
        amax = fmaxf(amax, fabsf(v[k]));
    if (amax == 0.0f) {
        *s = 0.0f;
        memset(q, 0, (size_t)K);
        return;
    }
    *s = amax / 448.0f;
    const float r = 448.0f / amax;
    for (int64_t k = 0; k < K; k++)
        q[k] = orc_e4m3_encode(v[k] * r);
}

/* Dynamic per-token FP8 quantiser; rotate != 0 applies the block-128
 * rotation first (then K must be a multiple of 128). */
int orc_quant_fp8(const uint16_t *x, int64_t M, int64_t K, int64_t ldx, int rotate,
                  uint8_t *q, float *s)
{
    if (M < 0 || K <= 0 || ldx < K || (rotate && K % 128 != 0))
        return ORC_ERR_ARG;
    float *v = (float *)malloc((size_t)K * sizeof(float));
    if (!v)
        return ORC_ERR_NOMEM;
    for (int64_t m = 0; m < M; m++) {
        if (rotate)
            orc_rotate_rows_f32(x + m * ldx, 1, K, ldx, v);
        else
            for (int64_t k = 0; k < K; k++)
                v[k] = bf16_to_f32(x[m * ldx + k]);
        quant_row_fp8(v, K, q + m * K, s + m);
    }
    free(v);
    return ORC_OK;
}

/* Static-scale quantiser: one caller-given scale s > 0 for the whole tensor
 * (a calibrated scale, in place of the per-token amax of the dynamic modes).
 * r = fp32(1 / s); v is the rotated row (mode 0: INT8 with block-128
 * rotation; mode 2: FP8 with rotation) or the row itself (mode 1: FP8);
 * INT8 codes q = clamp(rne(fp32(v * r)), -127, 127), FP8 codes
 * e4m3(fp32(v * r)) with saturation to +-448; every row's scale is s. */
int orc_quant_static(const uint16_t *x, int64_t M, int64_t K, int64_t ldx, int mode, float s,
                     void *q, float *sout)
{
    if (M < 0 || K <= 0 || ldx < K || mode < 0 || mode > 2 || !(s > 0.0f) || isinf(s))
        return ORC_ERR_ARG;
    const int rotate = (mode != 1);
    if (rotate && K % 128 != 0)
        return ORC_ERR_ARG;
    float *v = (float *)malloc((size_t)K * sizeof(float));
    if (!v)
        return ORC_ERR_NOMEM;
    const float r = 1.0f / s;
    for (int64_t m = 0; m < M; m++) {
        if (rotate)
            orc_rotate_rows_f32(x + m * ldx, 1, K, ldx, v);
        else
            for (int64_t k = 0; k < K; k++)
                v[k] = bf16_to_f32(x[m * ldx + k]);
        for (int64_t k = 0; k < K; k++) {
            const float t = v[k] * r;
            if (mode == 0) {
                float c = rne_int(t);
                if (c > 127.0f) c = 127.0f;
                if (c < -127.0f) c = -127.0f;
                ((int8_t *)q)[m * K + k] = (int8_t)c;
            } else {
                ((uint8_t *)q)[m * K + k] = orc_e4m3_encode(t);
            }
        }
        sout[m] = s;
    }
    free(v);
    return ORC_OK;
}

/* ------------------------------------------------------------------ */
/* INT8 GEMM and its fused epilogues                                   */
/* ------------------------------------------------------------------ */

/* acc[m][n] = sum_k qx[m][k] * qw[n][k], exact (int64 running sum, then
 * checked to fit int32).  qx: int8 [M][K], qw: int8 [N][K] (output-channel
 * major, the Linear convention), acc: int32 [M][N]. */
int orc_int8_gemm_acc(const int8_t *qx, const int8_t *qw, int64_t M, int64_t N, int64_t K,
                      int32_t *acc)
{
    if (M < 0 || N < 0 || K <= 0)
        return ORC_ERR_ARG;
    for (int64_t m = 0; m < M; m++)
        for (int64_t n = 0; n < N; n++) {
            int64_t a = 0;
            for (int64_t k = 0; k < K; k++)
                a += (int64_t)qx[m * K + k] * (int64_t)qw[n * K + k];
            if (a > INT32_MAX || a < INT32_MIN)
                return ORC_ERR_OVERFLOW;
            acc[m * N + n] = (int32_t)a;
        }
    return ORC_OK;
}

/* Epilogue value before rounding: ((float)acc * s_m) * sw_n + bias_n, each
 * operation rounded in fp32 (conversion of acc is nearest-even). */
static float epilogue_f32(int32_t acc, float s_m, float sw_n, const uint16_t *bias, int64_t n)
{
    float y = ((float)acc * s_m) * sw_n;
    if (bias)
        y = y + bf16_to_f32(bias[n]);
    return y;
}

/* W8A8 INT8 linear: y[m][n] = bf16(epilogue(acc[m][n])).  y has row stride ldy.
 * bias may be NULL. */
int orc_int8_linear(const int8_t *qx, const float *sx, const int8_t *qw, const float *sw,
                    const uint16_t *bias, int64_t M, int64_t N, int64_t K,
                    uint16_t *y, int64_t ldy)
{
    if (ldy < N)
        return ORC_ERR_ARG;
    int32_t *acc = (int32_t *)malloc((size_t)(N > 0 ? N : 1) * sizeof(int32_t));
    if (!acc)
        return ORC_ERR_NOMEM;
    for (int64_t m = 0; m < M; m++) {
        int rc = orc_int8_gemm_acc(qx + m * K, qw, 1, N, K, acc);
        if (rc) {
            free(acc);
            return rc;
        }
        for (int64_t n = 0; n < N; n++)
            y[m * ldy + n] = f32_to_bf16(epilogue_f32(acc[n], sx[m], sw[n], bias, n));
    }
    free(acc);
    return ORC_OK;
}

/* silu(g) * u in fp32: g / (1 + expf(-g)), then times u. */
static float swiglu_f32(float g, float u)
{
    float e = expf(-g);
    float d = 1.0f + e;
    float sg = g / d;
    return sg * u;
}

float orc_swiglu_f32(float g, float u) { return swiglu_f32(g, u); }

/* Gate/up with the paired SwiGLU epilogue.  qw_gu: int8 [2N][K], gate rows
 * 0..N-1 then up rows N..2N-1; sw_gu and bias_gu: [2N] (bias may be NULL).
 * h[m][n] = bf16(silu(g) * u) with g, u the unrounded epilogue values. */
int orc_int8_gateup_swiglu(const int8_t *qx, const float *sx, const int8_t *qw_gu,
                           const float *sw_gu, const uint16_t *bias_gu,
                           int64_t M, int64_t N, int64_t K, uint16_t *h, int64_t ldh)
{
    if (ldh < N)
        return ORC_ERR_ARG;
    int32_t *acc = (int32_t *)malloc((size_t)(N > 0 ? 2 * N : 1) * sizeof(int32_t));
    if (!acc)
        return ORC_ERR_NOMEM;
    for (int64_t m = 0; m < M; m++) {
        int rc = orc_int8_gemm_acc(qx + m * K, qw_gu, 1, 2 * N, K, acc);
        if (rc) {
            free(acc);
            return rc;
        }
        for (int64_t n = 0; n < N; n++) {
            float g = epilogue_f32(acc[n], sx[m], sw_gu[n], bias_gu, n);
            float u = epilogue_f32(acc[N + n], sx[m], sw_gu[N + n], bias_gu, N + n);
            h[m * ldh + n] = f32_to_bf16(swiglu_f32(g, u));
        }
    }
    free(acc);
    return ORC_OK;
}

/* Unfused reading (fuse_mlp off): gate and up already rounded to bf16 and
 * stored side by side in y_gu[M][2N] (row stride ldg);
 * h = bf16(silu(float(g)) * float(u)). */
int orc_swiglu_bf16(const uint16_t *y_gu, int64_t M, int64_t N, int64_t ldg,
                    uint16_t *h, int64_t ldh)
{
    if (M < 0 || N < 0 || ldg < 2 * N || ldh < N)
        return ORC_ERR_ARG;
    for (int64_t m = 0; m < M; m++)
        for (int64_t n = 0; n < N; n++) {
            float g = bf16_to_f32(y_gu[m * ldg + n]);
            float u = bf16_to_f32(y_gu[m * ldg + N + n]);
            h[m * ldh + n] = f32_to_bf16(swiglu_f32(g, u));
        }
    return ORC_OK;
}

/* ------------------------------------------------------------------ */
/* FP8 (e4m3) W8A8 linear                                              */
/* ------------------------------------------------------------------ */

/* acc = fp32(sum_k dec(qx[m][k]) * dec(qw[n][k])), sum exact in fp64 (see
 * header); epilogue as the INT8 path.  qx: e4m3 [M][K], qw: e4m3 [N][K]. */
int orc_fp8_linear(const uint8_t *qx, const float *sx, const uint8_t *qw, const float *sw,
                   const uint16_t *bias, int64_t M, int64_t N, int64_t K,
                   uint16_t *y, int64_t ldy)
{
    if (M < 0 || N < 0 || K <= 0 || K > 16384 || ldy < N)
        return ORC_ERR_ARG;
    for (int64_t m = 0; m < M; m++)
        for (int64_t n = 0; n < N; n++) {
            double a = 0.0;
            for (int64_t k = 0; k < K; k++)
                a += orc_e4m3_decode(qx[m * K + k]) * orc_e4m3_decode(qw[n * K + k]);
            float acc = (float)a;
            float v = (acc * sx[m]) * sw[n];
            if (bias)
                v = v + bf16_to_f32(bias[n]);
            y[m * ldy + n] = f32_to_bf16(v);
        }
    return ORC_OK;
}

/* ------------------------------------------------------------------ */
/* Runtime LoRA add                                                     */
/* ------------------------------------------------------------------ */

/* Stage 1: t[m][j] = bf16(sum_k x[m][k] * A[j][k]) for j < r, and exact zeros
 * for r <= j < r_pad.  x: bf16 [M][K] (row stride ldx), A: bf16 [r][K],
 * t: bf16 [M][r_pad] dense. */
int orc_lora_t(const uint16_t *x, int64_t ldx, const uint16_t *A, int64_t M, int64_t K,
               int64_t r, int64_t r_pad, uint16_t *t)
{
    if (M < 0 || K <= 0 || r <= 0 || r_pad < r || ldx < K)
        return ORC_ERR_ARG;
    for (int64_t m = 0; m < M; m++)
        for (int64_t j = 0; j < r_pad; j++) {
            if (j >= r) {
                t[m * r_pad + j] = 0;
                continue;
            }
            double a = 0.0;
            for (int64_t k = 0; k < K; k++)
                a += (double)bf16_to_f32(x[m * ldx + k]) * (double)bf16_to_f32(A[j * K + k]);
            t[m * r_pad + j] = f64_to_bf16(a);
        }
    return ORC_OK;
}

/* Stage 2: y[m][n] = bf16(float(y[m][n]) + fp32(sum_j t[m][j] * B[n][j])), in
 * place.  t: bf16 [M][r_pad], B: bf16 [N][r] (columns j >= r read as zero),
 * y: bf16 [M][N] with row stride ldy. */
int orc_lora_y(const uint16_t *t, const uint16_t *B, int64_t M, int64_t N, int64_t r,
               int64_t r_pad, uint16_t *y, int64_t ldy)
{
    if (M < 0 || N < 0 || r <= 0 || r_pad < r || ldy < N)
        return ORC_ERR_ARG;
    for (int64_t m = 0; m < M; m++)
        for (int64_t n = 0; n < N; n++) {
            double a = 0.0;
            for (int64_t j = 0; j < r_pad; j++) {
                double b = (j < r) ? (double)bf16_to_f32(B[n * r + j]) : 0.0;
                a += (double)bf16_to_f32(t[m * r_pad + j]) * b;
            }
            float z = (float)a;
            y[m * ldy + n] = f32_to_bf16(bf16_to_f32(y[m * ldy + n]) + z);
        }
    return ORC_OK;
}

/* FP8 gate/up with the paired SwiGLU epilogue (packing as the INT8 call):
 * g, u = fp32 epilogue values of rows n and N+n of qw_gu [2N][K];
 * h = bf16(silu(g) * u). */
int orc_fp8_gateup_swiglu(const uint8_t *qx, const float *sx, const uint8_t *qw_gu,
                          const float *sw_gu, const uint16_t *bias_gu,
                          int64_t M, int64_t N, int64_t K, uint16_t *h, int64_t ldh)
{
    if (M < 0 || N < 0 || K <= 0 || K > 16384 || ldh < N)
        return ORC_ERR_ARG;
    for (int64_t m = 0; m < M; m++)
        for (int64_t n = 0; n < N; n++) {
            float gu[2];
            for (int half = 0; half < 2; half++) {
                int64_t row = n + half * N;
                double a = 0.0;
                for (int64_t k = 0; k < K; k++)
                    a += orc_e4m3_decode(qx[m * K + k]) * orc_e4m3_decode(qw_gu[row * K + k]);
                float v = ((float)a * sx[m]) * sw_gu[row];
                if (bias_gu)
                    v = v + bf16_to_f32(bias_gu[row]);
                gu[half] = v;
            }
            h[m * ldh + n] = f32_to_bf16(swiglu_f32(gu[0], gu[1]));
        }
    return ORC_OK;
}
