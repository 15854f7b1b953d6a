// abi.cu -- the extern "C" boundary declared in include/clef.h: host-side
// argument checks (nothing is launched on a bad argument), TMA tensor maps
// for each operand, dispatch to the kernels on the caller's stream, and the
// library-owned device status word that time-limited device waits report to.
#include <atomic>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/clef.h"
#include "clef_kernels.h"

namespace clef {

__device__ unsigned int g_status = 0u;

namespace {

constexpr int kMaxDevices = 64;

struct DeviceState {
    bool ready = false;
    bool supported = false;
    int index = 0;
    int num_sms = 0;
    unsigned int *status = nullptr;  // device address of g_status on this device
};

DeviceState g_dev[kMaxDevices];
std::mutex g_mu;

// Caller-owned stream-K workspaces bound to (device, stream); guarded by g_mu.
struct WsBinding {
    int dev;
    void *stream;
    void *ptr;
    int64_t bytes;
};
constexpr size_t kMaxBindings = 256;
WsBinding g_ws[kMaxBindings];
size_t g_ws_count = 0;
std::atomic<uint64_t> g_wait_limit_ns{1000000000ull};
std::atomic<int> g_force_timeout{0};
std::atomic<int> g_quant_staging{1};
std::atomic<int> g_pdl{1};
std::atomic<int> g_sm_budget{0};   // SMs the compute launches may fill (0: all)
thread_local char g_last_err[256] = "";

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

int cuda_fail(cudaError_t e, const char *what) {
    snprintf(g_last_err, sizeof g_last_err, "%s: %s", what, cudaGetErrorString(e));
    return CLEF_ERR_CUDA;
}

int arg_fail(const char *what) {
    snprintf(g_last_err, sizeof g_last_err, "invalid argument: %s", what);
    return CLEF_ERR_INVALID_ARG;
}

// Device checks and per-device set-up (status-word address, SM count).
int device_state(DeviceState **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return arg_fail("device index");
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceState &d = g_dev[dev];
    d.index = dev;
    if (!d.ready) {
        int major = 0, minor = 0;
        if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess)
            return cuda_fail(e, "compute capability");
        if ((e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
            return cuda_fail(e, "compute capability");
        d.supported = (major == 10 && minor == 3);
        if ((e = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return cuda_fail(e, "SM count");
        if (d.supported) {
            void *p = nullptr;
            if ((e = cudaGetSymbolAddress(&p, g_status)) != cudaSuccess)
                return cuda_fail(e, "status word address");
            d.status = static_cast<unsigned int *>(p);
        }
        if (!g_encode) {
            void *fn = nullptr;
            cudaDriverEntryPointQueryResult q;
            e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                 cudaEnableDefault, &q);
            if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
                return cuda_fail(e == cudaSuccess ? cudaErrorNotSupported : e, "cuTensorMapEncodeTiled");
            g_encode = reinterpret_cast<EncodeTiledFn>(fn);
        }
        d.ready = true;
    }
    if (!d.supported) {
        snprintf(g_last_err, sizeof g_last_err, "device %d is not sm_103 (GB300)", dev);
        return CLEF_ERR_UNSUPPORTED;
    }
    *out = &d;
    return CLEF_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// 2-D tensor map over a row-major [rows][inner] tensor with the given row
// pitch; zero fill outside the tensor.
int make_tmap(CUtensorMap *m, CUtensorMapDataType dt, const void *base, uint64_t inner,
              uint64_t rows, uint64_t pitch_bytes, uint32_t box_inner, uint32_t box_rows,
              CUtensorMapSwizzle sw) {
    const cuuint64_t dims[2] = {inner, rows};
    const cuuint64_t strides[1] = {pitch_bytes};
    const cuuint32_t box[2] = {box_inner, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    if (!g_encode) {
        snprintf(g_last_err, sizeof g_last_err, "tensor-map encoder not initialised (no device set-up)");
        return CLEF_ERR_CUDA;
    }
    CUresult r = g_encode(m, dt, 2, const_cast<void *>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        snprintf(g_last_err, sizeof g_last_err, "cuTensorMapEncodeTiled failed (%d)", (int)r);
        return CLEF_ERR_INVALID_ARG;
    }
    return CLEF_OK;
}

// SMs a compute launch may fill: the device's, or the caller's budget
// (clef_set_sm_budget) where that is fewer.
int launch_sms(const DeviceState *d) {
    const int b = g_sm_budget.load();
    return (b > 0 && b < d->num_sms) ? b : d->num_sms;
}

// The workspace bound to this device and stream, if any, which lets a launch
// split tiles across CTA pairs (INT8 stream-K, the K parts of the FP8 linear
// and of the LoRA x A^T).
void attach_workspace(GemmArgs &a, const DeviceState *d, const void *stream) {
    std::lock_guard<std::mutex> lk(g_mu);
    for (size_t i = 0; i < g_ws_count; ++i)
        if (g_ws[i].dev == d->index && g_ws[i].stream == stream) {
            a.sk_cnt = static_cast<int *>(g_ws[i].ptr);
            a.sk_ws = reinterpret_cast<int4 *>(static_cast<char *>(g_ws[i].ptr) + kSkCounterBytes);
            a.sk_ws_bytes = g_ws[i].bytes - kSkCounterBytes;
            return;
        }
}

GemmArgs base_args(const DeviceState *d, int64_t M, int64_t N, int64_t K) {
    GemmArgs a;
    memset(&a, 0, sizeof a);
    a.M = (int)M;
    a.N = (int)N;
    a.K = (int)K;
    a.status = d->status;
    a.wait_limit_ns = g_wait_limit_ns.load();
    a.force_timeout = g_force_timeout.load();
    return a;
}

constexpr int64_t kMaxDim = (int64_t)1 << 30;

// LoRA stage 1 (arguments already checked): t = bf16(x A^T), [M][r_pad] at
// pitch ldt; rows of A past r read as zeros.  N-fastest tiles: the column
// tiles of one row block run side by side and share its x rows in L2, so x
// (the large operand) streams from HBM once.
int lora_shrink_launch(DeviceState *d, const void *x, int64_t ldx, const void *A, int64_t M, int64_t K,
                       int64_t r, void *t, int64_t ldt, cudaStream_t st) {
    const int64_t r_pad = (r + 63) / 64 * 64;
    GemmArgs a1 = base_args(d, M, r_pad, K);
    a1.out = t;
    a1.ldo = ldt;
    a1.n_fastest = 1;
    attach_workspace(a1, d, st);
    return launch_gemm(kOpBF16, kEpiStoreBF16, lora_shrink_width(M, r_pad, launch_sms(d), 0),
                       Operand{x, (uint64_t)K, (uint64_t)M, (uint64_t)ldx * 2},
                       Operand{A, (uint64_t)K, (uint64_t)r, (uint64_t)K * 2}, a1, launch_sms(d), st);
}

// LoRA stage 2 (arguments already checked): y = bf16(y + t B^T) over K =
// r_pad; columns of B past r read as zeros, so t's columns r .. r_pad - 1
// add nothing.
int lora_expand_launch(DeviceState *d, const void *t, int64_t ldt, const void *B, int64_t M, int64_t N,
                       int64_t r, void *y, int64_t ldy, cudaStream_t st) {
    const int64_t r_pad = (r + 63) / 64 * 64;
    GemmArgs a2 = base_args(d, M, N, r_pad);
    a2.out = y;
    a2.ldo = ldy;
    // N-fastest: the CTAs running together cover neighbouring column blocks of
    // the same rows of y (q adapter at 24,032 tokens: 96.5 -> 93.1 us)
    a2.n_fastest = 1;
    return launch_gemm(kOpBF16, kEpiAddBF16, 128, Operand{t, (uint64_t)r_pad, (uint64_t)M, (uint64_t)ldt * 2},
                       Operand{B, (uint64_t)r, (uint64_t)N, (uint64_t)r * 2}, a2, launch_sms(d), st);
}

// Shared checks of the W8A8 GEMM entry points.  b_rows is the row count of
// the weight operand; out_elem the output element size.
// Returns CLEF_OK with *empty = true for a valid M = 0 call (whose row-indexed
// pointers may be null, as empty tensors' are).
int check_gemm(const void *qx, const float *sx, const void *qw, const float *sw, const void *bias,
               int64_t M, int64_t N, int64_t K, const void *out, int64_t ldo, bool scaled,
               bool *empty) {
    if (M < 0 || M > kMaxDim) return arg_fail("M out of range");
    if (N <= 0 || N > kMaxDim || N % 8 != 0) return arg_fail("N must be positive and a multiple of 8");
    if (K <= 0 || K > kMaxDim || K % 16 != 0) return arg_fail("K must be positive and a multiple of 16");
    if (ldo < N || ldo % 8 != 0) return arg_fail("output row pitch must be >= N and a multiple of 8");
    *empty = (M == 0);
    if (*empty) return CLEF_OK;
    if (!qx || !qw || !out) return arg_fail("null operand or output pointer");
    if (scaled && (!sx || !sw)) return arg_fail("null scale pointer");
    if (!aligned16(qx) || !aligned16(qw) || !aligned16(out)) return arg_fail("operand/output not 16-byte aligned");
    if (scaled && (!aligned16(sw) || (reinterpret_cast<uintptr_t>(sx) & 3u)))
        return arg_fail("weight scales must be 16-byte aligned, row scales 4-byte aligned");
    if (bias && !aligned16(bias)) return arg_fail("bias not 16-byte aligned");
    return CLEF_OK;
}

int run_w8a8(int op, int epi, const void *qx, const float *sx, const void *qw, const float *sw,
             const void *bias, int64_t M, int64_t N, int64_t K, void *out, int64_t ldo,
             void *stream) {
    const bool swiglu = (epi == kEpiSwiGLU);
    bool empty = false;
    int rc = check_gemm(qx, sx, qw, sw, bias, M, N, K, out, ldo, epi != kEpiStoreS32, &empty);
    if (rc || empty) return rc;
    if (swiglu && 2 * N > kMaxDim) return arg_fail("2N out of range");
    DeviceState *d = nullptr;
    if ((rc = device_state(&d))) return rc;
    const uint64_t b_rows = swiglu ? 2 * (uint64_t)N : (uint64_t)N;
    const Operand A = {qx, (uint64_t)K, (uint64_t)M, (uint64_t)K};
    const Operand B = {qw, (uint64_t)K, b_rows, (uint64_t)K};
    GemmArgs a = base_args(d, M, N, K);
    a.n_half = swiglu ? (int)N : 0;
    a.sa = sx;
    a.sb = sw;
    a.bias = static_cast<const uint16_t *>(bias);
    a.out = out;
    a.ldo = ldo;
    if (op == kOpI8 || (op == kOpF8 && epi == kEpiScaleBias)) attach_workspace(a, d, stream);
    return launch_gemm(op, epi, 256, A, B, a, launch_sms(d), static_cast<cudaStream_t>(stream));
}

// The INT8 linear or gate/up SwiGLU with the LoRA expand fused (checks,
// then one launch).  Linear: nseg column segments of the output read t at
// their own column offsets (nseg = 0: one segment at column 0).  Gate/up: t
// holds t_gate then t_up (2 r_pad columns) and B2 is the up factor.
int run_w8a8_lora(bool gateup, const void *qx, const float *sx, const void *qw, const float *sw,
                  const void *bias, int64_t M, int64_t N, int64_t K, const void *t, int64_t ldt,
                  const void *B, const void *B2, int64_t r, int nseg, const int64_t *seg_end,
                  const int64_t *seg_tcol, void *out, int64_t ldo, void *stream) {
    bool empty = false;
    int rc = check_gemm(qx, sx, qw, sw, bias, M, N, K, out, ldo, true, &empty);
    if (rc) return rc;
    if (gateup && 2 * N > kMaxDim) return arg_fail("2N out of range");
    if (r <= 0 || r > 1024 || r % 8 != 0) return arg_fail("rank must be in (0, 1024] and a multiple of 8");
    const int64_t r_pad = (r + 63) / 64 * 64;
    if (ldt <= 0 || ldt % 8 != 0 || ldt > kMaxDim) return arg_fail("ldt must be a positive multiple of 8");
    if (gateup && ldt < 2 * r_pad) return arg_fail("ldt must be >= 2 round_up(r, 64)");
    GemmArgs a;
    memset(&a, 0, sizeof a);
    if (gateup) nseg = 0;   // one segment: t_gate | t_up from column 0
    if (nseg < 0 || nseg > kLoraMaxSegs) return arg_fail("nseg must be in 0..4");
    if (nseg > 0 && (!seg_end || !seg_tcol)) return arg_fail("null segment array");
    const int n = nseg > 0 ? nseg : 1;
    int64_t prev = 0;
    for (int i = 0; i < n; ++i) {
        const int64_t end = nseg > 0 ? seg_end[i] : N;
        const int64_t tc = nseg > 0 ? seg_tcol[i] : 0;
        if (end <= prev || end > N) return arg_fail("segment ends must increase and stay within N");
        if (i + 1 < n && end % 256 != 0) return arg_fail("segment ends other than the last must be multiples of 256");
        if (i + 1 == n && end != N) return arg_fail("the last segment must end at N");
        if (tc < 0 || tc % 8 != 0 || tc + r_pad > ldt)
            return arg_fail("segment t columns must be multiples of 8 with tcol + round_up(r, 64) <= ldt");
        a.lora_seg_end[i] = (int)end;
        a.lora_seg_tcol[i] = (int)tc;
        prev = end;
    }
    a.lora_nseg = n;
    if (empty) return CLEF_OK;
    if (!t || !B || (gateup && !B2)) return arg_fail("null LoRA pointer");
    if (!aligned16(t) || !aligned16(B) || (gateup && !aligned16(B2)))
        return arg_fail("LoRA pointers must be 16-byte aligned");
    DeviceState *d = nullptr;
    if ((rc = device_state(&d))) return rc;
    const GemmArgs b = base_args(d, M, N, K);
    a.M = b.M;
    a.N = b.N;
    a.K = b.K;
    a.status = b.status;
    a.wait_limit_ns = b.wait_limit_ns;
    a.force_timeout = b.force_timeout;
    a.n_half = gateup ? (int)N : 0;
    a.sa = sx;
    a.sb = sw;
    a.bias = static_cast<const uint16_t *>(bias);
    a.out = out;
    a.ldo = ldo;
    a.lora_t = t;
    a.lora_ldt = ldt;
    a.lora_b = B;
    a.lora_b2 = B2;
    a.lora_r = (int)r;
    a.lora_nkb = (int)((gateup ? 2 : 1) * r_pad / 64);
    const Operand A = {qx, (uint64_t)K, (uint64_t)M, (uint64_t)K};
    const Operand W = {qw, (uint64_t)K, (gateup ? 2 : 1) * (uint64_t)N, (uint64_t)K};
    return launch_gemm(kOpI8, gateup ? kEpiSwiGLULora : kEpiScaleBiasLora, 256, A, W, a, launch_sms(d),
                       static_cast<cudaStream_t>(stream));
}

}  // namespace

// Internal services for other translation units of this library.
int internal_device(int *num_sms, unsigned int **status) {
    DeviceState *d = nullptr;
    int rc = device_state(&d);
    if (rc) return rc;
    *num_sms = d->num_sms;
    *status = d->status;
    return CLEF_OK;
}

int internal_lora_add(const void *x, int64_t ldx, const void *A, const void *B, int64_t M, int64_t K,
                      int64_t N, int64_t r, void *t, void *y, int64_t ldy, cudaStream_t st) {
    DeviceState *d = nullptr;
    int rc = device_state(&d);
    if (rc) return rc;
    const int64_t r_pad = (r + 63) / 64 * 64;
    if ((rc = lora_shrink_launch(d, x, ldx, A, M, K, r, t, r_pad, st))) return rc;
    return lora_expand_launch(d, t, r_pad, B, M, N, r, y, ldy, st);
}

int internal_make_tmap(CUtensorMap *m, CUtensorMapDataType dt, const void *base, uint64_t inner,
                       uint64_t rows, uint64_t pitch_bytes, uint32_t box_inner, uint32_t box_rows,
                       CUtensorMapSwizzle sw) {
    return make_tmap(m, dt, base, inner, rows, pitch_bytes, box_inner, box_rows, sw);
}

int internal_make_tmap_nd(CUtensorMap *m, CUtensorMapDataType dt, int rank, const void *base,
                          const uint64_t *dims, const uint64_t *strides, const uint32_t *box,
                          CUtensorMapSwizzle sw) {
    if (rank < 1 || rank > 5) return arg_fail("tensor-map rank");
    cuuint64_t d[5], st[4];
    cuuint32_t b[5], es[5];
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        b[i] = box[i];
        es[i] = 1;
        if (i + 1 < rank) st[i] = strides[i];
    }
    if (!g_encode) {
        snprintf(g_last_err, sizeof g_last_err, "tensor-map encoder not initialised (no device set-up)");
        return CLEF_ERR_CUDA;
    }
    CUresult r = g_encode(m, dt, (cuuint32_t)rank, const_cast<void *>(base), d, st, b, es,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        snprintf(g_last_err, sizeof g_last_err, "cuTensorMapEncodeTiled failed (%d)", (int)r);
        return CLEF_ERR_INVALID_ARG;
    }
    return CLEF_OK;
}

int internal_cuda_error(cudaError_t e, const char *what) { return cuda_fail(e, what); }

void internal_set_error(const char *msg) { snprintf(g_last_err, sizeof g_last_err, "%s", msg); }

bool internal_pdl() { return g_pdl.load() != 0; }

}  // namespace clef

using namespace clef;

namespace {

// Checks and launch shared by the dynamic and static quantizer entry points
// (static_s > 0: one static scale for every row).
int quant_common(const void *x, int64_t M, int64_t K, int64_t ldx, int mode, void *q, float *scale,
                 float static_s, void *stream) {
    if (mode != CLEF_ACT_INT8_H128 && mode != CLEF_ACT_FP8_E4M3 && mode != CLEF_ACT_FP8_E4M3_H128)
        return arg_fail("unknown quantizer mode");
    if (M < 0 || M > 0x7FFFFFFF) return arg_fail("M out of range");
    const bool rot = (mode != CLEF_ACT_FP8_E4M3);
    if (K <= 0 || K > 65536 || K % (rot ? 128 : 32) != 0)
        return arg_fail("K must be in (0, 65536] and a multiple of 128 (rotated) or 32");
    if (ldx < K || ldx % 8 != 0) return arg_fail("ldx must be >= K and a multiple of 8");
    if (M == 0) return CLEF_OK;
    if (!x || !q || !scale) return arg_fail("null pointer");
    if (!aligned16(x) || !aligned16(q)) return arg_fail("x and q must be 16-byte aligned");
    if (reinterpret_cast<uintptr_t>(scale) & 3u) return arg_fail("scale not 4-byte aligned");
    DeviceState *d = nullptr;
    int rc = device_state(&d);
    if (rc) return rc;
    QuantEnv env;
    env.num_sms = launch_sms(d);
    env.status = d->status;
    env.wait_limit_ns = g_wait_limit_ns.load();
    env.staging = g_quant_staging.load();
    if (static_s > 0.0f) {
        volatile float one = 1.0f;   // one IEEE fp32 division, as the definition states
        env.static_r = one / static_s;
        env.static_s = static_s;
    }
    cudaError_t e = launch_quant_act(mode, static_cast<const uint16_t *>(x), M, K, ldx,
                                     static_cast<uint8_t *>(q), scale, env,
                                     static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? CLEF_OK : cuda_fail(e, "quantizer launch");
}

}  // namespace

extern "C" {

int clef_quant_act(const void *x, int64_t M, int64_t K, int64_t ldx, int mode, void *q,
                   float *scale, void *stream) {
    return quant_common(x, M, K, ldx, mode, q, scale, 0.0f, stream);
}

int clef_quant_act_static(const void *x, int64_t M, int64_t K, int64_t ldx, int mode, float s,
                          void *q, float *scale, void *stream) {
    if (!(s > 0.0f) || s > 3.0e38f) return arg_fail("static scale must be positive and finite");
    return quant_common(x, M, K, ldx, mode, q, scale, s, stream);
}

int clef_w8a8_linear(const int8_t *qx, const float *sx, const int8_t *qw, const float *sw,
                     const void *bias, int64_t M, int64_t N, int64_t K, void *y, int64_t ldy,
                     void *stream) {
    return run_w8a8(kOpI8, kEpiScaleBias, qx, sx, qw, sw, bias, M, N, K, y, ldy, stream);
}

int clef_w8a8_gateup_swiglu(const int8_t *qx, const float *sx, const int8_t *qw_gu,
                            const float *sw_gu, const void *bias_gu, int64_t M, int64_t N,
                            int64_t K, void *h, int64_t ldh, void *stream) {
    return run_w8a8(kOpI8, kEpiSwiGLU, qx, sx, qw_gu, sw_gu, bias_gu, M, N, K, h, ldh, stream);
}

int clef_fp8_linear(const void *qx, const float *sx, const void *qw, const float *sw,
                    const void *bias, int64_t M, int64_t N, int64_t K, void *y, int64_t ldy,
                    void *stream) {
    return run_w8a8(kOpF8, kEpiScaleBias, qx, sx, qw, sw, bias, M, N, K, y, ldy, stream);
}

int clef_fp8_gateup_swiglu(const void *qx, const float *sx, const void *qw_gu, const float *sw_gu,
                           const void *bias_gu, int64_t M, int64_t N, int64_t K, void *h,
                           int64_t ldh, void *stream) {
    return run_w8a8(kOpF8, kEpiSwiGLU, qx, sx, qw_gu, sw_gu, bias_gu, M, N, K, h, ldh, stream);
}

int clef_w8a8_linear_lora(const int8_t *qx, const float *sx, const int8_t *qw, const float *sw,
                          const void *bias, int64_t M, int64_t N, int64_t K, const void *t, int64_t ldt,
                          const void *B, int64_t r, int nseg, const int64_t *seg_end,
                          const int64_t *seg_tcol, void *y, int64_t ldy, void *stream) {
    return run_w8a8_lora(false, qx, sx, qw, sw, bias, M, N, K, t, ldt, B, nullptr, r, nseg, seg_end, seg_tcol,
                         y, ldy, stream);
}

int clef_w8a8_gateup_swiglu_lora(const int8_t *qx, const float *sx, const int8_t *qw_gu, const float *sw_gu,
                                 const void *bias_gu, int64_t M, int64_t N, int64_t K, const void *t_gu,
                                 int64_t ldt, const void *B_gate, const void *B_up, int64_t r, void *h,
                                 int64_t ldh, void *stream) {
    return run_w8a8_lora(true, qx, sx, qw_gu, sw_gu, bias_gu, M, N, K, t_gu, ldt, B_gate, B_up, r, 0, nullptr,
                         nullptr, h, ldh, stream);
}

int clef_w8a8_gemm_s32(const int8_t *qx, const int8_t *qw, int64_t M, int64_t N, int64_t K,
                       int32_t *acc, int64_t ldc, void *stream) {
    return run_w8a8(kOpI8, kEpiStoreS32, qx, nullptr, qw, nullptr, nullptr, M, N, K, acc, ldc, stream);
}

int clef_lora_add(const void *x, int64_t ldx, const void *A, const void *B, int64_t M, int64_t K,
                  int64_t N, int64_t r, void *t_scratch, void *y, int64_t ldy, void *stream) {
    if (M < 0 || M > kMaxDim) return arg_fail("M out of range");
    if (K <= 0 || K > kMaxDim || K % 8 != 0) return arg_fail("K must be positive and a multiple of 8");
    if (N <= 0 || N > kMaxDim || N % 8 != 0) return arg_fail("N must be positive and a multiple of 8");
    if (r <= 0 || r > 1024 || r % 8 != 0) return arg_fail("rank must be in (0, 1024] and a multiple of 8");
    if (ldx < K || ldx % 8 != 0) return arg_fail("ldx must be >= K and a multiple of 8");
    if (ldy < N || ldy % 8 != 0) return arg_fail("ldy must be >= N and a multiple of 8");
    if (M == 0) return CLEF_OK;
    if (!x || !A || !B || !t_scratch || !y) return arg_fail("null pointer");
    if (!aligned16(x) || !aligned16(A) || !aligned16(B) || !aligned16(t_scratch) || !aligned16(y))
        return arg_fail("pointers must be 16-byte aligned");
    return internal_lora_add(x, ldx, A, B, M, K, N, r, t_scratch, y, ldy, static_cast<cudaStream_t>(stream));
}

int clef_lora_shrink(const void *x, int64_t ldx, const void *A, int64_t M, int64_t K, int64_t r,
                     void *t, int64_t ldt, void *stream) {
    if (M < 0 || M > kMaxDim) return arg_fail("M out of range");
    if (K <= 0 || K > kMaxDim || K % 8 != 0) return arg_fail("K must be positive and a multiple of 8");
    if (r <= 0 || r > 4096 || r % 8 != 0) return arg_fail("rank must be in (0, 4096] and a multiple of 8");
    if (ldx < K || ldx % 8 != 0) return arg_fail("ldx must be >= K and a multiple of 8");
    if (ldt < (r + 63) / 64 * 64 || ldt % 8 != 0)
        return arg_fail("ldt must be >= round_up(r, 64) and a multiple of 8");
    if (M == 0) return CLEF_OK;
    if (!x || !A || !t) return arg_fail("null pointer");
    if (!aligned16(x) || !aligned16(A) || !aligned16(t)) return arg_fail("pointers must be 16-byte aligned");
    DeviceState *d = nullptr;
    int rc = device_state(&d);
    if (rc) return rc;
    return lora_shrink_launch(d, x, ldx, A, M, K, r, t, ldt, static_cast<cudaStream_t>(stream));
}

int clef_lora_expand_add(const void *t, int64_t ldt, const void *B, int64_t M, int64_t N, int64_t r,
                         void *y, int64_t ldy, void *stream) {
    if (M < 0 || M > kMaxDim) return arg_fail("M out of range");
    if (N <= 0 || N > kMaxDim || N % 8 != 0) return arg_fail("N must be positive and a multiple of 8");
    if (r <= 0 || r > 4096 || r % 8 != 0) return arg_fail("rank must be in (0, 4096] and a multiple of 8");
    if (ldt < (r + 63) / 64 * 64 || ldt % 8 != 0)
        return arg_fail("ldt must be >= round_up(r, 64) and a multiple of 8");
    if (ldy < N || ldy % 8 != 0) return arg_fail("ldy must be >= N and a multiple of 8");
    if (M == 0) return CLEF_OK;
    if (!t || !B || !y) return arg_fail("null pointer");
    if (!aligned16(t) || !aligned16(B) || !aligned16(y)) return arg_fail("pointers must be 16-byte aligned");
    DeviceState *d = nullptr;
    int rc = device_state(&d);
    if (rc) return rc;
    return lora_expand_launch(d, t, ldt, B, M, N, r, y, ldy, static_cast<cudaStream_t>(stream));
}

int clef_lora_gateup_swiglu(const void *x, int64_t ldx, const void *A_gate, const void *B_gate,
                            const void *A_up, const void *B_up, int64_t M, int64_t K, int64_t N,
                            int64_t r, void *t_scratch, const void *y_gu, int64_t ld_gu, void *h,
                            int64_t ldh, void *stream) {
    if (M < 0 || M > kMaxDim) return arg_fail("M out of range");
    if (K <= 0 || K > kMaxDim || K % 8 != 0) return arg_fail("K must be positive and a multiple of 8");
    if (N <= 0 || 2 * N > kMaxDim || N % 8 != 0) return arg_fail("N must be positive and a multiple of 8");
    if (r <= 0 || r > 1024 || r % 8 != 0) return arg_fail("rank must be in (0, 1024] and a multiple of 8");
    if (ldx < K || ldx % 8 != 0) return arg_fail("ldx must be >= K and a multiple of 8");
    if (ld_gu < 2 * N || ld_gu % 8 != 0) return arg_fail("ld_gu must be >= 2N and a multiple of 8");
    if (ldh < N || ldh % 8 != 0) return arg_fail("ldh must be >= N and a multiple of 8");
    if (M == 0) return CLEF_OK;
    if (!x || !A_gate || !B_gate || !A_up || !B_up || !t_scratch || !y_gu || !h)
        return arg_fail("null pointer");
    if (!aligned16(x) || !aligned16(A_gate) || !aligned16(B_gate) || !aligned16(A_up) ||
        !aligned16(B_up) || !aligned16(t_scratch) || !aligned16(y_gu) || !aligned16(h))
        return arg_fail("pointers must be 16-byte aligned");
    DeviceState *d = nullptr;
    int rc = device_state(&d);
    if (rc) return rc;
    const int64_t r_pad = (r + 63) / 64 * 64;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // stage 1: t = [bf16(x A_gate^T) | bf16(x A_up^T)], [M][2 r_pad], as one
    // GEMM whose B rows r_pad .. 2 r_pad - 1 are A_up's (x streams once)
    {
        GemmArgs a1 = base_args(d, M, 2 * r_pad, K);
        a1.out = t_scratch;
        a1.ldo = 2 * r_pad;
        a1.n_fastest = 1;
        a1.b2_row0 = (int)r_pad;
        attach_workspace(a1, d, st);
        const Operand Au{A_up, (uint64_t)K, (uint64_t)r, (uint64_t)K * 2};
        rc = launch_gemm(kOpBF16, kEpiStoreBF16, lora_shrink_width(M, 2 * r_pad, launch_sms(d), r_pad),
                         Operand{x, (uint64_t)K, (uint64_t)M, (uint64_t)ldx * 2},
                         Operand{A_gate, (uint64_t)K, (uint64_t)r, (uint64_t)K * 2}, a1, launch_sms(d), st, &Au);
        if (rc) return rc;
    }
    // stage 2: one GEMM over K = 2 r_pad; gate rows see B_gate in the first
    // r_pad columns and zeros after (past the end of B_gate), up rows zeros
    // first (before the start of B_up) and B_up after, so each half sums only
    // its own adapter's products; the epilogue adds them to the base gate and
    // up values and forms h
    GemmArgs a2 = base_args(d, M, N, 2 * r_pad);
    a2.n_half = (int)N;
    a2.aux = y_gu;
    a2.ld_aux = ld_gu;
    a2.k_shift = (int)r_pad;
    a2.out = h;
    a2.ldo = ldh;
    const Operand Bu{B_up, (uint64_t)r, (uint64_t)N, (uint64_t)r * 2};
    return launch_gemm(kOpBF16, kEpiLoraSwiGLU, 256,
                       Operand{t_scratch, (uint64_t)(2 * r_pad), (uint64_t)M, (uint64_t)(2 * r_pad) * 2},
                       Operand{B_gate, (uint64_t)r, (uint64_t)N, (uint64_t)r * 2}, a2, launch_sms(d), st, &Bu);
}

int clef_swiglu_bf16(const void *y_gu, int64_t M, int64_t N, int64_t ldg, void *h, int64_t ldh,
                     void *stream) {
    if (M < 0 || M > kMaxDim) return arg_fail("M out of range");
    if (N <= 0 || N > kMaxDim || N % 8 != 0) return arg_fail("N must be positive and a multiple of 8");
    if (ldg < 2 * N || ldg % 8 != 0) return arg_fail("ldg must be >= 2N and a multiple of 8");
    if (ldh < N || ldh % 8 != 0) return arg_fail("ldh must be >= N and a multiple of 8");
    if (M == 0) return CLEF_OK;
    if (!y_gu || !h) return arg_fail("null pointer");
    if (!aligned16(y_gu) || !aligned16(h)) return arg_fail("pointers must be 16-byte aligned");
    DeviceState *d = nullptr;
    int rc = device_state(&d);
    if (rc) return rc;
    cudaError_t e = launch_swiglu_bf16(static_cast<const uint16_t *>(y_gu), M, N, ldg,
                                       static_cast<uint16_t *>(h), ldh, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? CLEF_OK : cuda_fail(e, "swiglu launch");
}

int clef_gemm_workspace_bytes(int64_t *bytes) {
    if (!bytes) return arg_fail("null pointer");
    DeviceState *d = nullptr;
    int rc = device_state(&d);
    if (rc) return rc;
    *bytes = kSkCounterBytes + (int64_t)(d->num_sms / 2) * kSkBytesPerPair;
    return CLEF_OK;
}

int clef_bind_workspace(void *stream, void *ws, int64_t bytes) {
    if (ws && !aligned16(ws)) return arg_fail("workspace must be 16-byte aligned");
    if (ws && bytes < kSkCounterBytes) return arg_fail("workspace smaller than its counter block");
    DeviceState *d = nullptr;
    int rc = device_state(&d);
    if (rc) return rc;
    std::lock_guard<std::mutex> lk(g_mu);
    size_t i = 0;
    while (i < g_ws_count && !(g_ws[i].dev == d->index && g_ws[i].stream == stream)) ++i;
    if (!ws) {   // unbind
        if (i < g_ws_count) g_ws[i] = g_ws[--g_ws_count];
        return CLEF_OK;
    }
    if (i == g_ws_count) {
        if (g_ws_count == kMaxBindings) return arg_fail("too many bound workspaces (256)");
        ++g_ws_count;
    }
    g_ws[i] = WsBinding{d->index, stream, ws, bytes};
    return CLEF_OK;
}

int clef_poll_status(void) {
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
    unsigned int w = 0, zero = 0;
    if ((e = cudaMemcpyFromSymbol(&w, g_status, sizeof w)) != cudaSuccess) return cuda_fail(e, "read status");
    if ((e = cudaMemcpyToSymbol(g_status, &zero, sizeof zero)) != cudaSuccess) return cuda_fail(e, "clear status");
    if (w) snprintf(g_last_err, sizeof g_last_err, "device status word 0x%08x (site %u)", w, (w >> 8) & 0xFFu);
    return (int)(w & 0xFFu);
}

void clef_set_wait_limit_ns(uint64_t ns) { g_wait_limit_ns.store(ns ? ns : 1); }

void clef_test_force_timeout(int on) { g_force_timeout.store(on < 0 ? 0 : on); }

void clef_set_quant_staging(int mode) { g_quant_staging.store(mode < 0 ? 0 : (mode > 2 ? 2 : mode)); }

void clef_set_pdl(int on) { g_pdl.store(on ? 1 : 0); }

int clef_set_sm_budget(int sms) {
    if (sms < 0 || sms == 1) return arg_fail("sms must be 0 (all) or at least 2");
    g_sm_budget.store(sms & ~1);
    return CLEF_OK;
}

const char *clef_status_string(int status) {
    switch (status) {
        case CLEF_OK: return "CLEF_OK";
        case CLEF_ERR_INVALID_ARG: return "CLEF_ERR_INVALID_ARG";
        case CLEF_ERR_UNSUPPORTED: return "CLEF_ERR_UNSUPPORTED";
        case CLEF_ERR_CUDA: return "CLEF_ERR_CUDA";
        case CLEF_ERR_TIMEOUT: return "CLEF_ERR_TIMEOUT";
        default: return "CLEF_ERR_UNKNOWN";
    }
}

const char *clef_last_error(void) { return g_last_err; }

int clef_abi_version(void) { return 100; }

}  // extern "C"
