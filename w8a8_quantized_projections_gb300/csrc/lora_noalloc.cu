// lora_noalloc.cu -- clef_lora_add_noalloc: the runtime LoRA add for callers
// that cannot hand the library a scratch buffer.
//
// clef_lora_add needs a caller-owned scratch of M x round_up(r, 64) bf16 for
// the intermediate t = bf16(x A^T).  Some callers cannot provide one: a host
// whose serving runtime owns a fixed device-memory budget and forbids
// allocations outside it, a plugin running inside another framework's
// allocator, or code that must not pay the device-wide synchronisation that
// cudaMalloc / cudaFree can imply.  This entry point keeps t in a
// library-owned, statically sized device array instead, so neither the caller
// nor the library allocates anything.
//
// The array is a file-scope static __device__ symbol: every GPU that loads the
// library holds its 8 MiB until the process exits.  In host code the symbol's
// name is only a host-side stand-in, so its device address is looked up with
// cudaGetSymbolAddress once per device (with that device current), on the
// first call of this entry point on that device, and passed to the kernels.
// That first call should therefore happen before any stream capture.
//
// Every call shares the one array, which keeps whatever the previous call
// left there.  Nothing has to start at zero: the first kernel of each call
// writes every element of t that the second kernel reads (including the
// padded columns past the rank, written as exact zeros).  Calls whose
// kernels overlap on the GPU (different streams without ordering between
// them, or different host threads) race on the array: serialise them.
#include <cstdint>
#include <cstdio>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/clef.h"
#include "clef_kernels.h"

namespace clef {

// 4 Mi bf16 elements = 8 MiB: rows x round_up(rank, 64) must not exceed it
// (for example 16,384 tokens at rank 256, or 65,536 tokens at rank 64).
static constexpr int64_t kNoAllocScratchElems = (int64_t)4 << 20;
static __device__ __align__(256) uint16_t g_lora_noalloc_scratch[kNoAllocScratchElems];

namespace {

constexpr int kMaxDev = 64;
uint16_t *g_scratch_ptr[kMaxDev] = {};
std::mutex g_setup_mu;

int fail(const char *msg) {
    internal_set_error(msg);
    return CLEF_ERR_INVALID_ARG;
}

// Device address of the scratch array on the current device (looked up once).
int scratch_address(uint16_t **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= kMaxDev) {
        internal_set_error("clef_lora_add_noalloc: no usable current device");
        return CLEF_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lk(g_setup_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_lora_noalloc_scratch);
        if (e != cudaSuccess || !p) {
            char buf[160];
            snprintf(buf, sizeof buf, "clef_lora_add_noalloc: cudaGetSymbolAddress failed: %s",
                     cudaGetErrorString(e));
            internal_set_error(buf);
            return CLEF_ERR_CUDA;
        }
        g_scratch_ptr[dev] = static_cast<uint16_t *>(p);
    }
    *out = g_scratch_ptr[dev];
    return CLEF_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace clef

using namespace clef;

extern "C" int clef_lora_add_noalloc(const void *x, int64_t ldx, const void *A, const void *B,
                                     int64_t M, int64_t K, int64_t N, int64_t r, void *y,
                                     int64_t ldy, void *stream) {
    const int64_t kMaxDim = (int64_t)1 << 30;
    if (M < 0 || M > kMaxDim) return fail("invalid argument: M out of range");
    if (K <= 0 || K > kMaxDim || K % 8 != 0) return fail("invalid argument: K must be positive and a multiple of 8");
    if (N <= 0 || N > kMaxDim || N % 8 != 0) return fail("invalid argument: N must be positive and a multiple of 8");
    if (r <= 0 || r > 1024 || r % 8 != 0) return fail("invalid argument: rank must be in (0, 1024] and a multiple of 8");
    if (ldx < K || ldx % 8 != 0) return fail("invalid argument: ldx must be >= K and a multiple of 8");
    if (ldy < N || ldy % 8 != 0) return fail("invalid argument: ldy must be >= N and a multiple of 8");
    const int64_t r_pad = (r + 63) / 64 * 64;
    if (M * r_pad > kNoAllocScratchElems)
        return fail("invalid argument: M * round_up(rank, 64) exceeds the 4,194,304-element "
                    "built-in scratch of clef_lora_add_noalloc (use clef_lora_add with a scratch buffer)");
    if (M == 0) return CLEF_OK;
    if (!x || !A || !B || !y) return fail("invalid argument: null pointer");
    if (!aligned16(x) || !aligned16(A) || !aligned16(B) || !aligned16(y))
        return fail("invalid argument: pointers must be 16-byte aligned");
    int num_sms = 0;
    unsigned int *status = nullptr;
    int rc = internal_device(&num_sms, &status);   // device checks (sm_103) first
    if (rc) return rc;
    uint16_t *t = nullptr;
    if ((rc = scratch_address(&t))) return rc;
    // the launches of clef_lora_add (tile widths, wait limit and test knob
    // included), on the built-in array in place of a caller scratch
    return internal_lora_add(x, ldx, A, B, M, K, N, r, t, y, ldy, static_cast<cudaStream_t>(stream));
}
