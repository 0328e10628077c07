// ttt_api.cu -- the C ABI of include/ttt.h: argument validation, kernel
// selection, launch, status codes and the device status word.
//
// Every entry point validates all arguments before launching anything, so an
// invalid call has no side effect on the device.  Kernel selection is by shape
// and dtype only; there is exactly one implementation per shape.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "../../include/ttt.h"
#include "ttt_internal.h"

namespace {

thread_local char g_last_error[256] = "";

ttt_status fail(ttt_status s, const char* fmt, const char* detail = "") {
    snprintf(g_last_error, sizeof(g_last_error), fmt, detail);
    return s;
}

ttt_status cuda_fail(cudaError_t e, const char* where) {
    snprintf(g_last_error, sizeof(g_last_error), "%s: %s", where, cudaGetErrorString(e));
    return TTT_ERR_CUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool supported_d(int d) { return d == 16 || d == 32 || d == 64 || d == 128; }

// Device status word: written by kernels (first error wins), read and cleared
// by ttt_get_device_status().  One copy per device (a __device__ variable is
// instantiated in every context that loads the module).  Its address is looked
// up on every call, in the context current then, so no address outlives a
// device reset or a re-created primary context.
__device__ int g_device_status;

cudaError_t status_ptr(int** out) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_device_status);
    if (e != cudaSuccess) return e;
    *out = static_cast<int*>(p);
    return cudaSuccess;
}

// Diagnostic bound of the fused TTT-Linear prefill's barrier waits, from the environment variable
// TTT_WAIT_LIMIT_NS (1 ns .. 4 s; 0 or unset: the default 4 s).  A tiny bound makes a real
// prefill's waits expire, which exercises its failure path (status word, clean exit) without
// faulting anything.
uint64_t wait_limit_from_env() {
    const char* v = getenv("TTT_WAIT_LIMIT_NS");
    if (!v) return 0;
    const unsigned long long n = strtoull(v, nullptr, 10);
    return n > 4000000000ull ? 4000000000ull : n;
}

#define CHECK_PTR(p)                                                              \
    do {                                                                          \
        if (!(p)) return fail(TTT_ERR_INVALID_ARG, "null pointer argument: %s", #p); \
        if (!aligned16(p)) return fail(TTT_ERR_INVALID_ARG, "pointer not 16-byte aligned: %s", #p); \
    } while (0)

}  // namespace

extern "C" {

// First kernel of a prefill dispatch from the environment variable `var`: 0 (`k0`), 1 (`k1`),
// 2 ("generic"), or -1 when unset or unknown (the default choice by shape).
static int kernel_choice(const char* var, const char* k0, const char* k1, const char* k2 = nullptr) {
    const char* v = getenv(var);
    if (!v) return -1;
    if (!strcmp(v, k0)) return 0;
    if (!strcmp(v, k1)) return 1;
    if (k2 && !strcmp(v, k2)) return 2;
    if (!strcmp(v, "generic")) return k2 ? 3 : 2;
    return -1;
}

ttt_status ttt_linear_prefill(const void* Q, const void* K, const void* V, const float* eta, const float* W0,
                              void* Z, float* W_out, int B, int H, int T, int d, int chunk, ttt_dtype dtype,
                              void* stream) {
    g_last_error[0] = 0;
    if (B < 0 || H < 0 || T < 0) return fail(TTT_ERR_INVALID_ARG, "negative size%s");
    if (chunk < 1 || chunk > 512) return fail(TTT_ERR_INVALID_ARG, "chunk must be in 1..512%s");
    if (dtype != TTT_F32 && dtype != TTT_BF16) return fail(TTT_ERR_INVALID_ARG, "unknown dtype%s");
    if (d <= 0) return fail(TTT_ERR_INVALID_ARG, "head dim must be positive%s");
    if (!supported_d(d)) return fail(TTT_ERR_UNSUPPORTED, "head dim must be 16, 32, 64 or 128%s");
    if (size_t(B) * H == 0) return TTT_OK;
    CHECK_PTR(W0);
    CHECK_PTR(W_out);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (T == 0) {
        if (W_out != W0) {
            cudaError_t e = cudaMemcpyAsync(W_out, W0, size_t(B) * H * d * d * sizeof(float),
                                            cudaMemcpyDeviceToDevice, s);
            if (e != cudaSuccess) return cuda_fail(e, "ttt_linear_prefill copy");
        }
        return TTT_OK;
    }
    CHECK_PTR(Q);
    CHECK_PTR(K);
    CHECK_PTR(V);
    CHECK_PTR(eta);
    CHECK_PTR(Z);
    ttt::LinearArgs a{Q, K, V, eta, W0, Z, W_out, B, H, T, d, chunk, dtype == TTT_BF16 ? 1 : 0};
    a.wait_ns = wait_limit_from_env();
    int* status = nullptr;
    cudaError_t e = status_ptr(&status);
    if (e != cudaSuccess) return cuda_fail(e, "ttt_linear_prefill status word");
    // bf16, 16 | chunk, any T: the fused warp-MMA kernel at d = 64, the split warp-MMA kernel at
    // d = 128; the generic kernel otherwise.  TTT_LINEAR_PREFILL_KERNEL = "fused", "tc", "mma"
    // or "generic" makes the dispatch start at that kernel (the next one takes the shapes it does
    // not cover); "tc" is the kernel with the read-out on tcgen05.
    const int first = kernel_choice("TTT_LINEAR_PREFILL_KERNEL", "fused", "tc", "mma");
    e = cudaErrorNotSupported;
    if (first <= 0) e = ttt::launch_linear_prefill_fused(a, s, status);
    if (e == cudaErrorNotSupported && first == 1) e = ttt::launch_linear_prefill_tc(a, s, status);
    if (e == cudaErrorNotSupported && first <= 2) e = ttt::launch_linear_prefill_mma(a, s, status);
    if (e == cudaErrorNotSupported) e = ttt::launch_linear_prefill_generic(a, s);
    if (e != cudaSuccess) return cuda_fail(e, "ttt_linear_prefill launch");
    return TTT_OK;
}

// Segment plan of the split prefill for this shape (TTT_LINEAR_SEGMENTS = n asks for n segments).
static ttt::SegPlan seg_plan_for(const ttt::LinearArgs& a) {
    const char* v = getenv("TTT_LINEAR_SEGMENTS");
    const int force = v ? atoi(v) : 0;
    return ttt::linear_segment_plan(a, force > 0 ? force : 0);
}

size_t ttt_linear_prefill_workspace_size(int B, int H, int T, int d, int chunk, ttt_dtype dtype) {
    if (B <= 0 || H <= 0 || T <= 0 || chunk < 1 || chunk > 512 || !supported_d(d) ||
        (dtype != TTT_F32 && dtype != TTT_BF16))
        return 0;
    ttt::LinearArgs a{nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, B, H, T, d, chunk,
                      dtype == TTT_BF16 ? 1 : 0};
    return ttt::linear_segment_workspace_bytes(a, seg_plan_for(a));
}

ttt_status ttt_linear_prefill_ws(const void* Q, const void* K, const void* V, const float* eta, const float* W0,
                                 void* Z, float* W_out, int B, int H, int T, int d, int chunk, ttt_dtype dtype,
                                 void* workspace, size_t workspace_bytes, void* stream) {
    g_last_error[0] = 0;
    if (B < 0 || H < 0 || T < 0) return fail(TTT_ERR_INVALID_ARG, "negative size%s");
    if (chunk < 1 || chunk > 512) return fail(TTT_ERR_INVALID_ARG, "chunk must be in 1..512%s");
    if (dtype != TTT_F32 && dtype != TTT_BF16) return fail(TTT_ERR_INVALID_ARG, "unknown dtype%s");
    if (d <= 0) return fail(TTT_ERR_INVALID_ARG, "head dim must be positive%s");
    if (!supported_d(d)) return fail(TTT_ERR_UNSUPPORTED, "head dim must be 16, 32, 64 or 128%s");
    const size_t need = ttt_linear_prefill_workspace_size(B, H, T, d, chunk, dtype);
    if (need == 0)  // no split for this shape: the one-pass scan
        return ttt_linear_prefill(Q, K, V, eta, W0, Z, W_out, B, H, T, d, chunk, dtype, stream);
    CHECK_PTR(Q);
    CHECK_PTR(K);
    CHECK_PTR(V);
    CHECK_PTR(eta);
    CHECK_PTR(W0);
    CHECK_PTR(Z);
    CHECK_PTR(W_out);
    if (!workspace || workspace_bytes < need)
        return fail(TTT_ERR_INVALID_ARG, "workspace smaller than ttt_linear_prefill_workspace_size()%s");
    CHECK_PTR(workspace);
    ttt::LinearArgs a{Q, K, V, eta, W0, Z, W_out, B, H, T, d, chunk, dtype == TTT_BF16 ? 1 : 0};
    int* status = nullptr;
    cudaError_t e = status_ptr(&status);
    if (e != cudaSuccess) return cuda_fail(e, "ttt_linear_prefill_ws status word");
    e = ttt::launch_linear_prefill_segmented(a, seg_plan_for(a), workspace, static_cast<cudaStream_t>(stream), status);
    if (e != cudaSuccess) return cuda_fail(e, "ttt_linear_prefill_ws launch");
    return TTT_OK;
}

// ---------------------------------------------------------------- split prefill, built-in scratch
//
// For callers that cannot allocate device memory at the moment they run the scan: a serving loop
// that must never reach the device allocator (cudaMalloc may synchronise the whole device and stall
// every stream), or code whose device memory is handed out by another allocator it may not go
// around.  ttt_linear_prefill_noalloc runs the split prefill with its maps and start states in this
// fixed array instead of caller scratch.  Every GPU that loads the library holds the array until the
// process exits.  Nothing in it has to start at zero: each call writes every word it later reads.
// All calls share it, so calls that overlap on the GPU (other streams, other host threads) race.
constexpr size_t kSplitScratchBytes = size_t(16) << 20;  // 16 MiB
static __device__ __align__(256) float g_split_scratch[kSplitScratchBytes / sizeof(float)];

// Device address of g_split_scratch for the current device, looked up with that device current on
// the first call there (and again if the device's context changed since, e.g. after a reset); the
// lookup is a runtime call, so that first call belongs before any stream capture.
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);

static cudaError_t split_scratch_ptr(void** out) {
    constexpr int kMaxDev = 64;
    static std::mutex mu;
    static void* ctx_of[kMaxDev] = {};
    static void* ptr_of[kMaxDev] = {};
    static CtxGetCurrentFn get_ctx = nullptr;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(mu);
    if (!get_ctx) {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        e = cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q);
        if (e != cudaSuccess) return e;
        if (q != cudaDriverEntryPointSuccess || !f) return cudaErrorSymbolNotFound;
        get_ctx = reinterpret_cast<CtxGetCurrentFn>(f);
    }
    CUcontext ctx = nullptr;
    if (get_ctx(&ctx) != CUDA_SUCCESS) return cudaErrorDeviceUninitialized;
    if (!ptr_of[dev] || ctx_of[dev] != static_cast<void*>(ctx)) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_split_scratch);
        if (e != cudaSuccess) return e;
        ptr_of[dev] = p;
        ctx_of[dev] = static_cast<void*>(ctx);
    }
    *out = ptr_of[dev];
    return cudaSuccess;
}

ttt_status ttt_linear_prefill_noalloc(const void* Q, const void* K, const void* V, const float* eta, const float* W0,
                                      void* Z, float* W_out, int B, int H, int T, int d, int chunk, ttt_dtype dtype,
                                      void* stream) {
    g_last_error[0] = 0;
    if (B < 0 || H < 0 || T < 0) return fail(TTT_ERR_INVALID_ARG, "negative size%s");
    if (chunk < 1 || chunk > 512) return fail(TTT_ERR_INVALID_ARG, "chunk must be in 1..512%s");
    if (dtype != TTT_F32 && dtype != TTT_BF16) return fail(TTT_ERR_INVALID_ARG, "unknown dtype%s");
    if (d <= 0) return fail(TTT_ERR_INVALID_ARG, "head dim must be positive%s");
    if (!supported_d(d)) return fail(TTT_ERR_UNSUPPORTED, "head dim must be 16, 32, 64 or 128%s");
    const size_t need = ttt_linear_prefill_workspace_size(B, H, T, d, chunk, dtype);
    if (need == 0)  // no split for this shape: the one-pass scan, which needs no scratch either
        return ttt_linear_prefill(Q, K, V, eta, W0, Z, W_out, B, H, T, d, chunk, dtype, stream);
    if (need > kSplitScratchBytes) {
        snprintf(g_last_error, sizeof(g_last_error),
                 "the split of this shape needs %zu bytes of scratch, more than the %zu of the built-in scratch "
                 "(use ttt_linear_prefill_ws with caller scratch)",
                 need, kSplitScratchBytes);
        return TTT_ERR_UNSUPPORTED;
    }
    CHECK_PTR(Q);
    CHECK_PTR(K);
    CHECK_PTR(V);
    CHECK_PTR(eta);
    CHECK_PTR(W0);
    CHECK_PTR(Z);
    CHECK_PTR(W_out);
    void* scratch = nullptr;
    cudaError_t e = split_scratch_ptr(&scratch);
    if (e != cudaSuccess) return cuda_fail(e, "ttt_linear_prefill_noalloc scratch address");
    int* status = nullptr;
    e = status_ptr(&status);
    if (e != cudaSuccess) return cuda_fail(e, "ttt_linear_prefill_noalloc status word");
    ttt::LinearArgs a{Q, K, V, eta, W0, Z, W_out, B, H, T, d, chunk, dtype == TTT_BF16 ? 1 : 0};
    e = ttt::launch_linear_prefill_segmented(a, seg_plan_for(a), scratch, static_cast<cudaStream_t>(stream), status);
    if (e != cudaSuccess) return cuda_fail(e, "ttt_linear_prefill_noalloc launch");
    return TTT_OK;
}

ttt_status ttt_linear_momentum_prefill(const void* Q, const void* K, const void* V, const float* eta,
                                      const float* W0, const float* M0, void* Z, float* W_out, float* M_out, int B,
                                      int H, int T, int d, int chunk, float beta, ttt_dtype dtype, void* stream) {
    g_last_error[0] = 0;
    if (B < 0 || H < 0 || T < 0) return fail(TTT_ERR_INVALID_ARG, "negative size%s");
    if (chunk < 1 || chunk > 512) return fail(TTT_ERR_INVALID_ARG, "chunk must be in 1..512%s");
    if (dtype != TTT_F32 && dtype != TTT_BF16) return fail(TTT_ERR_INVALID_ARG, "unknown dtype%s");
    if (d <= 0) return fail(TTT_ERR_INVALID_ARG, "head dim must be positive%s");
    if (!(beta >= 0.f && beta <= 1.f)) return fail(TTT_ERR_INVALID_ARG, "beta must be in [0, 1]%s");
    if (!supported_d(d)) return fail(TTT_ERR_UNSUPPORTED, "head dim must be 16, 32, 64 or 128%s");
    if (size_t(B) * H == 0) return TTT_OK;
    CHECK_PTR(W0);
    CHECK_PTR(W_out);
    CHECK_PTR(M_out);
    if (M0 && !aligned16(M0)) return fail(TTT_ERR_INVALID_ARG, "pointer not 16-byte aligned: %s", "M0");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (T == 0) {  // no tokens: the state and the momentum pass through
        const size_t bytes = size_t(B) * H * d * d * sizeof(float);
        cudaError_t e = W_out != W0 ? cudaMemcpyAsync(W_out, W0, bytes, cudaMemcpyDeviceToDevice, s) : cudaSuccess;
        if (e == cudaSuccess)
            e = M0 ? (M_out != M0 ? cudaMemcpyAsync(M_out, M0, bytes, cudaMemcpyDeviceToDevice, s) : cudaSuccess)
                   : cudaMemsetAsync(M_out, 0, bytes, s);
        if (e != cudaSuccess) return cuda_fail(e, "ttt_linear_momentum_prefill copy");
        return TTT_OK;
    }
    CHECK_PTR(Q);
    CHECK_PTR(K);
    CHECK_PTR(V);
    CHECK_PTR(eta);
    CHECK_PTR(Z);
    ttt::LinearArgs a{Q, K, V, eta, W0, Z, W_out, B, H, T, d, chunk, dtype == TTT_BF16 ? 1 : 0};
    a.momentum = true;
    a.M0 = M0;
    a.M_out = M_out;
    a.beta = beta;
    // bf16, d = 64, chunk 16, any T: the warp-MMA kernel; the SIMT kernel otherwise
    // (TTT_LINEAR_MOMENTUM_KERNEL = "simt" forces the SIMT kernel)
    const char* kv = getenv("TTT_LINEAR_MOMENTUM_KERNEL");
    cudaError_t e = cudaErrorNotSupported;
    if (!(kv && !strcmp(kv, "simt"))) e = ttt::launch_linear_momentum_mma(a, s);
    if (e == cudaErrorNotSupported) e = ttt::launch_linear_prefill_generic(a, s);
    if (e != cudaSuccess) return cuda_fail(e, "ttt_linear_momentum_prefill launch");
    return TTT_OK;
}

ttt_status ttt_linear_prefill_hist(const void* Q, const void* K, const void* V, const float* eta, const float* W0,
                                   void* Z, float* W_out, void* W_hist, int B, int H, int T, int d, int chunk,
                                   ttt_dtype dtype, void* stream) {
    g_last_error[0] = 0;
    if (B < 0 || H < 0 || T < 0) return fail(TTT_ERR_INVALID_ARG, "negative size%s");
    if (chunk < 1 || chunk > 512) return fail(TTT_ERR_INVALID_ARG, "chunk must be in 1..512%s");
    if (dtype != TTT_F32 && dtype != TTT_BF16) return fail(TTT_ERR_INVALID_ARG, "unknown dtype%s");
    if (d <= 0) return fail(TTT_ERR_INVALID_ARG, "head dim must be positive%s");
    if (!supported_d(d)) return fail(TTT_ERR_UNSUPPORTED, "head dim must be 16, 32, 64 or 128%s");
    if (size_t(B) * H == 0) return TTT_OK;
    if (T == 0) return ttt_linear_prefill(Q, K, V, eta, W0, Z, W_out, B, H, T, d, chunk, dtype, stream);
    CHECK_PTR(Q);
    CHECK_PTR(K);
    CHECK_PTR(V);
    CHECK_PTR(eta);
    CHECK_PTR(W0);
    CHECK_PTR(Z);
    CHECK_PTR(W_out);
    CHECK_PTR(W_hist);
    ttt::LinearArgs a{Q, K, V, eta, W0, Z, W_out, B, H, T, d, chunk, dtype == TTT_BF16 ? 1 : 0};
    a.W_hist = W_hist;
    // the warp-MMA kernels record the block-start states for bf16, chunk 16, any T, d = 64 (the
    // fused kernel) or d = 128 (the split kernel); the generic kernel for every other shape
    int* status = nullptr;
    cudaError_t e = status_ptr(&status);
    if (e != cudaSuccess) return cuda_fail(e, "ttt_linear_prefill_hist status word");
    e = ttt::launch_linear_prefill_fused(a, static_cast<cudaStream_t>(stream), status);
    if (e == cudaErrorNotSupported) e = ttt::launch_linear_prefill_mma(a, static_cast<cudaStream_t>(stream), status);
    if (e == cudaErrorNotSupported) e = ttt::launch_linear_prefill_generic(a, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "ttt_linear_prefill_hist launch");
    return TTT_OK;
}

ttt_status ttt_linear_prefill_backward(const void* Q, const void* K, const void* V, const float* eta,
                                       const void* W_hist, const void* dZ, const float* dW_T, void* dQ, void* dK,
                                       void* dV, float* deta, float* dW0, int B, int H, int T, int d, int chunk,
                                       ttt_dtype dtype, void* stream) {
    g_last_error[0] = 0;
    if (B < 0 || H < 0 || T < 0) return fail(TTT_ERR_INVALID_ARG, "negative size%s");
    if (chunk < 1 || chunk > 512) return fail(TTT_ERR_INVALID_ARG, "chunk must be in 1..512%s");
    if (dtype != TTT_F32 && dtype != TTT_BF16) return fail(TTT_ERR_INVALID_ARG, "unknown dtype%s");
    if (d <= 0) return fail(TTT_ERR_INVALID_ARG, "head dim must be positive%s");
    if (!supported_d(d)) return fail(TTT_ERR_UNSUPPORTED, "head dim must be 16, 32, 64 or 128%s");
    if (!ttt::linear_backward_supported(d, chunk))
        return fail(TTT_ERR_UNSUPPORTED, "backward: the block tiles of this chunk and head dim exceed shared memory%s");
    if (size_t(B) * H == 0) return TTT_OK;
    CHECK_PTR(dW0);
    if (dW_T && !aligned16(dW_T)) return fail(TTT_ERR_INVALID_ARG, "pointer not 16-byte aligned: %s", "dW_T");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (T == 0) {  // no tokens: the state passes through unchanged
        const size_t bytes = size_t(B) * H * d * d * sizeof(float);
        cudaError_t e = dW_T ? (dW_T != dW0 ? cudaMemcpyAsync(dW0, dW_T, bytes, cudaMemcpyDeviceToDevice, s)
                                            : cudaSuccess)
                             : cudaMemsetAsync(dW0, 0, bytes, s);
        if (e != cudaSuccess) return cuda_fail(e, "ttt_linear_prefill_backward copy");
        return TTT_OK;
    }
    CHECK_PTR(Q);
    CHECK_PTR(K);
    CHECK_PTR(V);
    CHECK_PTR(eta);
    CHECK_PTR(W_hist);
    CHECK_PTR(dZ);
    CHECK_PTR(dQ);
    CHECK_PTR(dK);
    CHECK_PTR(dV);
    CHECK_PTR(deta);
    ttt::LinearBwdArgs a{Q, K, V, eta, W_hist, dZ, dW_T, dQ, dK, dV, deta, dW0, B, H, T, d, chunk,
                         dtype == TTT_BF16 ? 1 : 0};
    // bf16, d = 64, chunk 16, any T: the tensor-core kernel; the SIMT kernel otherwise
    // (TTT_LINEAR_BACKWARD_KERNEL = "simt" forces the SIMT kernel)
    const char* kv = getenv("TTT_LINEAR_BACKWARD_KERNEL");
    cudaError_t e = cudaErrorNotSupported;
    if (!(kv && !strcmp(kv, "simt"))) {
        int* status = nullptr;
        e = status_ptr(&status);
        if (e != cudaSuccess) return cuda_fail(e, "ttt_linear_prefill_backward status word");
        e = ttt::launch_linear_backward_mma(a, s, status);
    }
    if (e == cudaErrorNotSupported) e = ttt::launch_linear_backward(a, s);
    if (e != cudaSuccess) return cuda_fail(e, "ttt_linear_prefill_backward launch");
    return TTT_OK;
}

ttt_status ttt_mlp_prefill(const void* Q, const void* K, const void* V, const float* eta, const float* W1_0,
                           const float* W2_0, void* Z, float* W1_out, float* W2_out, int B, int H, int T, int d,
                           int hidden, int chunk, ttt_dtype dtype, void* stream) {
    g_last_error[0] = 0;
    if (B < 0 || H < 0 || T < 0) return fail(TTT_ERR_INVALID_ARG, "negative size%s");
    if (chunk < 1 || chunk > 512) return fail(TTT_ERR_INVALID_ARG, "chunk must be in 1..512%s");
    if (dtype != TTT_F32 && dtype != TTT_BF16) return fail(TTT_ERR_INVALID_ARG, "unknown dtype%s");
    if (d <= 0 || hidden <= 0) return fail(TTT_ERR_INVALID_ARG, "dimensions must be positive%s");
    if (!(d == 16 || d == 32 || d == 64)) return fail(TTT_ERR_UNSUPPORTED, "MLP head dim must be 16, 32 or 64%s");
    if (hidden % 16 != 0 || size_t(d) * hidden > 16384)
        return fail(TTT_ERR_UNSUPPORTED, "MLP hidden must be a multiple of 16 with d*hidden <= 16384%s");
    if (size_t(chunk) * hidden > 4096 || chunk > 64)
        return fail(TTT_ERR_UNSUPPORTED, "MLP chunk must satisfy chunk <= 64 and chunk*hidden <= 4096%s");
    if (size_t(B) * H == 0) return TTT_OK;
    CHECK_PTR(W1_0);
    CHECK_PTR(W2_0);
    CHECK_PTR(W1_out);
    CHECK_PTR(W2_out);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t nw = size_t(B) * H * d * hidden * sizeof(float);
    if (T == 0) {
        cudaError_t e = cudaSuccess;
        if (W1_out != W1_0) e = cudaMemcpyAsync(W1_out, W1_0, nw, cudaMemcpyDeviceToDevice, s);
        if (e == cudaSuccess && W2_out != W2_0) e = cudaMemcpyAsync(W2_out, W2_0, nw, cudaMemcpyDeviceToDevice, s);
        if (e != cudaSuccess) return cuda_fail(e, "ttt_mlp_prefill copy");
        return TTT_OK;
    }
    CHECK_PTR(Q);
    CHECK_PTR(K);
    CHECK_PTR(V);
    CHECK_PTR(eta);
    CHECK_PTR(Z);
    ttt::MlpArgs a{Q, K, V, eta, W1_0, W2_0, Z, W1_out, W2_out, B, H, T, d, hidden, chunk, dtype == TTT_BF16 ? 1 : 0};
    int* status = nullptr;
    cudaError_t e = status_ptr(&status);
    if (e != cudaSuccess) return cuda_fail(e, "ttt_mlp_prefill status word");
    // bf16, d = 64, hidden = 256, chunk = 16, any T: the warp-MMA kernel (state in registers), else
    // the tcgen05 kernel; the generic kernel otherwise.  TTT_MLP_PREFILL_KERNEL = "mma", "tc" or
    // "generic" makes the dispatch start at that kernel.
    const int first = kernel_choice("TTT_MLP_PREFILL_KERNEL", "mma", "tc");
    e = cudaErrorNotSupported;
    if (first <= 0) e = ttt::launch_mlp_prefill_mma(a, s, status);
    if (e == cudaErrorNotSupported && first <= 1) e = ttt::launch_mlp_prefill_tc(a, s, status);
    if (e == cudaErrorNotSupported) e = ttt::launch_mlp_prefill_generic(a, s);
    if (e != cudaSuccess) return cuda_fail(e, "ttt_mlp_prefill launch");
    return TTT_OK;
}

// Validation shared by the TTT-MLP prefill entry points (shapes of ttt_mlp_prefill).
static ttt_status mlp_shape_check(int B, int H, int T, int d, int hidden, int chunk, ttt_dtype dtype) {
    if (B < 0 || H < 0 || T < 0) return fail(TTT_ERR_INVALID_ARG, "negative size%s");
    if (chunk < 1 || chunk > 512) return fail(TTT_ERR_INVALID_ARG, "chunk must be in 1..512%s");
    if (dtype != TTT_F32 && dtype != TTT_BF16) return fail(TTT_ERR_INVALID_ARG, "unknown dtype%s");
    if (d <= 0 || hidden <= 0) return fail(TTT_ERR_INVALID_ARG, "dimensions must be positive%s");
    if (!(d == 16 || d == 32 || d == 64)) return fail(TTT_ERR_UNSUPPORTED, "MLP head dim must be 16, 32 or 64%s");
    if (hidden % 16 != 0 || size_t(d) * hidden > 16384)
        return fail(TTT_ERR_UNSUPPORTED, "MLP hidden must be a multiple of 16 with d*hidden <= 16384%s");
    if (size_t(chunk) * hidden > 4096 || chunk > 64)
        return fail(TTT_ERR_UNSUPPORTED, "MLP chunk must satisfy chunk <= 64 and chunk*hidden <= 4096%s");
    return TTT_OK;
}

ttt_status ttt_mlp_prefill_hist(const void* Q, const void* K, const void* V, const float* eta, const float* W1_0,
                                const float* W2_0, void* Z, float* W1_out, float* W2_out, void* W1_hist,
                                void* W2_hist, int B, int H, int T, int d, int hidden, int chunk, ttt_dtype dtype,
                                void* stream) {
    g_last_error[0] = 0;
    ttt_status st = mlp_shape_check(B, H, T, d, hidden, chunk, dtype);
    if (st != TTT_OK) return st;
    if (size_t(B) * H == 0) return TTT_OK;
    if (T == 0)
        return ttt_mlp_prefill(Q, K, V, eta, W1_0, W2_0, Z, W1_out, W2_out, B, H, T, d, hidden, chunk, dtype, stream);
    CHECK_PTR(Q);
    CHECK_PTR(K);
    CHECK_PTR(V);
    CHECK_PTR(eta);
    CHECK_PTR(W1_0);
    CHECK_PTR(W2_0);
    CHECK_PTR(Z);
    CHECK_PTR(W1_out);
    CHECK_PTR(W2_out);
    CHECK_PTR(W1_hist);
    CHECK_PTR(W2_hist);
    ttt::MlpArgs a{Q, K, V, eta, W1_0, W2_0, Z, W1_out, W2_out, B, H, T, d, hidden, chunk, dtype == TTT_BF16 ? 1 : 0};
    a.W1_hist = W1_hist;
    a.W2_hist = W2_hist;
    int* status = nullptr;
    cudaError_t e = status_ptr(&status);
    if (e != cudaSuccess) return cuda_fail(e, "ttt_mlp_prefill_hist status word");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // the warp-MMA kernel records the states for its shape (bf16, d 64, hidden 256, chunk 16); the
    // generic kernel for every other shape
    e = ttt::launch_mlp_prefill_mma(a, s, status);
    if (e == cudaErrorNotSupported) e = ttt::launch_mlp_prefill_generic(a, s);
    if (e != cudaSuccess) return cuda_fail(e, "ttt_mlp_prefill_hist launch");
    return TTT_OK;
}

ttt_status ttt_mlp_prefill_backward(const void* Q, const void* K, const void* V, const float* eta,
                                    const void* W1_hist, const void* W2_hist, const void* dZ, const float* dW1_T,
                                    const float* dW2_T, void* dQ, void* dK, void* dV, float* deta, float* dW1_0,
                                    float* dW2_0, int B, int H, int T, int d, int hidden, int chunk, ttt_dtype dtype,
                                    void* stream) {
    g_last_error[0] = 0;
    ttt_status st = mlp_shape_check(B, H, T, d, hidden, chunk, dtype);
    if (st != TTT_OK) return st;
    if (!ttt::mlp_backward_supported(d, hidden, chunk))
        return fail(TTT_ERR_UNSUPPORTED, "MLP backward: chunk must be at most 16 and the block tiles fit in shared "
                                         "memory%s");
    if (size_t(B) * H == 0) return TTT_OK;
    CHECK_PTR(dW1_0);
    CHECK_PTR(dW2_0);
    if (dW1_T && !aligned16(dW1_T)) return fail(TTT_ERR_INVALID_ARG, "pointer not 16-byte aligned: %s", "dW1_T");
    if (dW2_T && !aligned16(dW2_T)) return fail(TTT_ERR_INVALID_ARG, "pointer not 16-byte aligned: %s", "dW2_T");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (T == 0) {  // no tokens: the state gradients pass through
        const size_t bytes = size_t(B) * H * d * hidden * sizeof(float);
        cudaError_t e = dW1_T ? (dW1_T != dW1_0 ? cudaMemcpyAsync(dW1_0, dW1_T, bytes, cudaMemcpyDeviceToDevice, s)
                                                 : cudaSuccess)
                              : cudaMemsetAsync(dW1_0, 0, bytes, s);
        if (e == cudaSuccess)
            e = dW2_T ? (dW2_T != dW2_0 ? cudaMemcpyAsync(dW2_0, dW2_T, bytes, cudaMemcpyDeviceToDevice, s)
                                        : cudaSuccess)
                      : cudaMemsetAsync(dW2_0, 0, bytes, s);
        if (e != cudaSuccess) return cuda_fail(e, "ttt_mlp_prefill_backward copy");
        return TTT_OK;
    }
    CHECK_PTR(Q);
    CHECK_PTR(K);
    CHECK_PTR(V);
    CHECK_PTR(eta);
    CHECK_PTR(W1_hist);
    CHECK_PTR(W2_hist);
    CHECK_PTR(dZ);
    CHECK_PTR(dQ);
    CHECK_PTR(dK);
    CHECK_PTR(dV);
    CHECK_PTR(deta);
    ttt::MlpBwdArgs a{Q, K, V, eta, W1_hist, W2_hist, dZ, dW1_T, dW2_T, dQ, dK, dV, deta, dW1_0, dW2_0,
                      B, H, T, d, hidden, chunk, dtype == TTT_BF16 ? 1 : 0};
    // bf16, d = 64, hidden = 256, chunk 16, any T: the warp-MMA kernel; the SIMT kernel otherwise
    // (TTT_MLP_BACKWARD_KERNEL = "simt" forces the SIMT kernel)
    const char* kv = getenv("TTT_MLP_BACKWARD_KERNEL");
    cudaError_t e = cudaErrorNotSupported;
    if (!(kv && !strcmp(kv, "simt"))) e = ttt::launch_mlp_backward_mma(a, s);
    if (e == cudaErrorNotSupported) e = ttt::launch_mlp_backward(a, s);
    if (e != cudaSuccess) return cuda_fail(e, "ttt_mlp_prefill_backward launch");
    return TTT_OK;
}

ttt_status ttt_linear_decode_step(const void* q, const void* k, const void* v, const float* eta, float* W, void* z,
                                  int B, int H, int d, ttt_dtype dtype, void* stream) {
    g_last_error[0] = 0;
    if (B < 0 || H < 0) return fail(TTT_ERR_INVALID_ARG, "negative size%s");
    if (dtype != TTT_F32 && dtype != TTT_BF16) return fail(TTT_ERR_INVALID_ARG, "unknown dtype%s");
    if (d <= 0) return fail(TTT_ERR_INVALID_ARG, "head dim must be positive%s");
    if (!supported_d(d)) return fail(TTT_ERR_UNSUPPORTED, "head dim must be 16, 32, 64 or 128%s");
    if (size_t(B) * H == 0) return TTT_OK;
    if (size_t(B) * H > 0x7fffffffu) return fail(TTT_ERR_UNSUPPORTED, "B*H too large%s");
    CHECK_PTR(q);
    CHECK_PTR(k);
    CHECK_PTR(v);
    CHECK_PTR(eta);
    CHECK_PTR(W);
    CHECK_PTR(z);
    ttt::DecodeArgs a{q, k, v, eta, W, z, B, H, d, dtype == TTT_BF16 ? 1 : 0};
    int* status = nullptr;
    cudaError_t e = status_ptr(&status);
    if (e != cudaSuccess) return cuda_fail(e, "ttt_linear_decode_step status word");
    e = ttt::launch_linear_decode(a, static_cast<cudaStream_t>(stream), status);
    if (e != cudaSuccess) return cuda_fail(e, "ttt_linear_decode_step launch");
    return TTT_OK;
}

ttt_status ttt_mlp_decode_step(const void* q, const void* k, const void* v, const float* eta, float* W1, float* W2,
                               void* z, int B, int H, int d, int hidden, ttt_dtype dtype, void* stream) {
    g_last_error[0] = 0;
    if (B < 0 || H < 0) return fail(TTT_ERR_INVALID_ARG, "negative size%s");
    if (dtype != TTT_F32 && dtype != TTT_BF16) return fail(TTT_ERR_INVALID_ARG, "unknown dtype%s");
    if (d <= 0 || hidden <= 0) return fail(TTT_ERR_INVALID_ARG, "dimensions must be positive%s");
    if (!(d == 16 || d == 32 || d == 64)) return fail(TTT_ERR_UNSUPPORTED, "MLP head dim must be 16, 32 or 64%s");
    if (!(hidden == 64 || hidden == 128 || hidden == 256))
        return fail(TTT_ERR_UNSUPPORTED, "MLP decode hidden must be 64, 128 or 256%s");
    if (size_t(B) * H == 0) return TTT_OK;
    if (size_t(B) * H > 0x7fffffffu) return fail(TTT_ERR_UNSUPPORTED, "B*H too large%s");
    CHECK_PTR(q);
    CHECK_PTR(k);
    CHECK_PTR(v);
    CHECK_PTR(eta);
    CHECK_PTR(W1);
    CHECK_PTR(W2);
    CHECK_PTR(z);
    ttt::MlpDecodeArgs a{q, k, v, eta, W1, W2, z, B, H, d, hidden, dtype == TTT_BF16 ? 1 : 0};
    cudaError_t e = ttt::launch_mlp_decode(a, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "ttt_mlp_decode_step launch");
    return TTT_OK;
}

ttt_status ttt_selftest_wait_timeout(uint64_t limit_ns, void* stream) {
    g_last_error[0] = 0;
    if (limit_ns == 0 || limit_ns > 2000000000ull)
        return fail(TTT_ERR_INVALID_ARG, "limit must be in 1 ns .. 2 s%s");
    int* status = nullptr;
    cudaError_t e = status_ptr(&status);
    if (e != cudaSuccess) return cuda_fail(e, "ttt_selftest_wait_timeout status word");
    e = ttt::launch_wait_timeout_selftest(limit_ns, static_cast<cudaStream_t>(stream), status);
    if (e != cudaSuccess) return cuda_fail(e, "ttt_selftest_wait_timeout launch");
    return TTT_OK;
}

ttt_status ttt_get_device_status(void* stream) {
    int* p = nullptr;
    cudaError_t e = status_ptr(&p);
    if (e != cudaSuccess) return cuda_fail(e, "ttt_get_device_status");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int h = 0;
    e = cudaMemcpyAsync(&h, p, sizeof(int), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(p, 0, sizeof(int), s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "ttt_get_device_status");
    if (h == 0) return TTT_OK;
    if (h == TTT_ERR_TIMEOUT) return fail(TTT_ERR_TIMEOUT, "a bounded device-side wait expired%s");
    return fail(static_cast<ttt_status>(h), "device reported status %s", "");
}

const char* ttt_status_string(ttt_status s) {
    switch (s) {
        case TTT_OK: return "ok";
        case TTT_ERR_INVALID_ARG: return "invalid argument";
        case TTT_ERR_UNSUPPORTED: return "unsupported shape";
        case TTT_ERR_CUDA: return "CUDA error";
        case TTT_ERR_TIMEOUT: return "device-side wait timed out";
    }
    return "unknown status";
}

const char* ttt_last_error(void) { return g_last_error; }

int ttt_version(void) { return 10500; }  // 1.5: the tensor-core kernels take any T

}  // extern "C"
