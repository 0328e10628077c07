// mlp_prefill_generic.cu -- SIMT fp32 TTT-MLP prefill.
//
// Inner model f(x; W1, W2) = GELU(x W1) W2 (tanh form of GELU, no biases)
// ("Test-Time Training (TTT) Layers for Sequence Modeling", section
// "Variants: TTT-Linear vs. TTT-MLP").  Per block of n tokens with start state
// (W1, W2), the dual form of the mini-batch step:
//   Zk = K W1, Hk = GELU(Zk), E2 = Hk W2 - V, E1 = (E2 W2^T) . GELU'(Zk)
//   Hq = GELU(Q W1 - tril(eta . Q K^T) E1)        (layer-1 delta)
//   Z  = Hq W2 - tril(eta . Hq Hk^T) E2           (layer-2 delta)
//   W1 -= K^T diag(eta) E1,  W2 -= Hk^T diag(eta) E2
//
// One CTA per (batch, head).  The state lives in the caller's output buffers
// (W1_out, W2_out, fp32, read-modify-written in place block after block, so it
// stays in L2); block intermediates live in shared memory.  Reference-quality
// GPU path for every supported shape.
#include "ttt_common.cuh"
#include "ttt_internal.h"

namespace ttt {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ float gelu_tanh(float x) {
    const float c = 0.7978845608028654f, a = 0.044715f;
    float t = tanhf(c * (x + a * x * x * x));
    return 0.5f * x * (1.f + t);
}

__device__ __forceinline__ float gelu_tanh_prime(float x) {
    const float c = 0.7978845608028654f, a = 0.044715f;
    float t = tanhf(c * (x + a * x * x * x));
    return 0.5f * (1.f + t) + 0.5f * x * (1.f - t * t) * c * (1.f + 3.f * a * x * x);
}

struct Smem {
    int d, hd, n;
    __device__ float* q(float* b) const { return b; }
    __device__ float* k(float* b) const { return b + n * d; }
    __device__ float* v(float* b) const { return b + 2 * n * d; }
    __device__ float* e2(float* b) const { return b + 3 * n * d; }
    __device__ float* gp(float* b) const { return b + 4 * n * d; }            // GELU'(Zk), then Hq
    __device__ float* hk(float* b) const { return b + 4 * n * d + n * hd; }
    __device__ float* e1(float* b) const { return b + 4 * n * d + 2 * n * hd; }
    __device__ float* a(float* b) const { return b + 4 * n * d + 3 * n * hd; }  // [n][n]
    __device__ float* eta(float* b) const { return b + 4 * n * d + 3 * n * hd + n * n; }
};

template <typename TI>
__global__ void __launch_bounds__(kThreads)
mlp_prefill_generic_kernel(const TI* __restrict__ Q, const TI* __restrict__ K, const TI* __restrict__ V,
                           const float* __restrict__ eta, const float* W1_0, const float* W2_0,
                           TI* __restrict__ Z, float* W1, float* W2, int T, int d, int hd, int chunk,
                           TI* __restrict__ W1_hist, TI* __restrict__ W2_hist) {
    extern __shared__ float smem[];
    const size_t bh = blockIdx.x;
    const size_t nw = size_t(d) * hd;
    W1 += bh * nw;
    W2 += bh * nw;
    if (W1_0 + bh * nw != W1)
        for (size_t i = threadIdx.x; i < nw; i += kThreads) W1[i] = W1_0[bh * nw + i];
    if (W2_0 + bh * nw != W2)
        for (size_t i = threadIdx.x; i < nw; i += kThreads) W2[i] = W2_0[bh * nw + i];
    const TI* Qh = Q + bh * size_t(T) * d;
    const TI* Kh = K + bh * size_t(T) * d;
    const TI* Vh = V + bh * size_t(T) * d;
    const float* eh = eta + bh * size_t(T);
    TI* Zh = Z + bh * size_t(T) * d;
    __syncthreads();

    const int nblk = (T + chunk - 1) / chunk;
    for (int t0 = 0; t0 < T; t0 += chunk) {
        const int n = min(chunk, T - t0);
        const Smem L{d, hd, chunk};
        if (W1_hist) {  // the state at the start of this block, in the element type of Q
            TI* h1 = W1_hist + (bh * nblk + t0 / chunk) * nw;
            TI* h2 = W2_hist + (bh * nblk + t0 / chunk) * nw;
            for (size_t i = threadIdx.x; i < nw; i += kThreads) {
                h1[i] = from_f32<TI>(W1[i]);
                h2[i] = from_f32<TI>(W2[i]);
            }
        }
        float *qs = L.q(smem), *ks = L.k(smem), *vs = L.v(smem), *e2 = L.e2(smem);
        float *gp = L.gp(smem), *hk = L.hk(smem), *e1 = L.e1(smem), *as = L.a(smem), *es = L.eta(smem);

        for (int i = threadIdx.x; i < n * d; i += kThreads) {
            qs[i] = to_f32(Qh[size_t(t0) * d + i]);
            ks[i] = to_f32(Kh[size_t(t0) * d + i]);
            vs[i] = to_f32(Vh[size_t(t0) * d + i]);
        }
        for (int i = threadIdx.x; i < n; i += kThreads) es[i] = eh[t0 + i];
        __syncthreads();

        // Zk = K W1 -> Hk = GELU(Zk), gp = GELU'(Zk)
        for (int idx = threadIdx.x; idx < n * hd; idx += kThreads) {
            int j = idx / hd, m = idx % hd;
            float acc = 0.f;
            for (int i = 0; i < d; ++i) acc += ks[j * d + i] * W1[size_t(i) * hd + m];
            hk[idx] = gelu_tanh(acc);
            gp[idx] = gelu_tanh_prime(acc);
        }
        // A1 = tril(eta . Q K^T)
        for (int idx = threadIdx.x; idx < n * n; idx += kThreads) {
            int i = idx / n, j = idx % n;
            float s = 0.f;
            if (j <= i) {
                for (int c = 0; c < d; ++c) s += qs[i * d + c] * ks[j * d + c];
                s *= es[j];
            }
            as[idx] = s;
        }
        __syncthreads();
        // E2 = Hk W2 - V
        for (int idx = threadIdx.x; idx < n * d; idx += kThreads) {
            int j = idx / d, c = idx % d;
            float acc = 0.f;
            for (int m = 0; m < hd; ++m) acc += hk[j * hd + m] * W2[size_t(m) * d + c];
            e2[idx] = acc - vs[idx];
        }
        __syncthreads();
        // E1 = (E2 W2^T) . GELU'(Zk)
        for (int idx = threadIdx.x; idx < n * hd; idx += kThreads) {
            int j = idx / hd, m = idx % hd;
            float acc = 0.f;
            for (int c = 0; c < d; ++c) acc += e2[j * d + c] * W2[size_t(m) * d + c];
            e1[idx] = acc * gp[idx];
        }
        __syncthreads();
        // Hq = GELU(Q W1 - A1 E1)   (written over gp)
        for (int idx = threadIdx.x; idx < n * hd; idx += kThreads) {
            int i = idx / hd, m = idx % hd;
            float acc = 0.f;
            for (int c = 0; c < d; ++c) acc += qs[i * d + c] * W1[size_t(c) * hd + m];
            for (int j = 0; j <= i; ++j) acc -= as[i * n + j] * e1[j * hd + m];
            gp[idx] = gelu_tanh(acc);
        }
        __syncthreads();
        // A2 = tril(eta . Hq Hk^T)
        for (int idx = threadIdx.x; idx < n * n; idx += kThreads) {
            int i = idx / n, j = idx % n;
            float s = 0.f;
            if (j <= i) {
                for (int m = 0; m < hd; ++m) s += gp[i * hd + m] * hk[j * hd + m];
                s *= es[j];
            }
            as[idx] = s;
        }
        __syncthreads();
        // Z = Hq W2 - A2 E2
        for (int idx = threadIdx.x; idx < n * d; idx += kThreads) {
            int i = idx / d, c = idx % d;
            float acc = 0.f;
            for (int m = 0; m < hd; ++m) acc += gp[i * hd + m] * W2[size_t(m) * d + c];
            for (int j = 0; j <= i; ++j) acc -= as[i * n + j] * e2[j * d + c];
            Zh[size_t(t0 + i) * d + c] = from_f32<TI>(acc);
        }
        __syncthreads();  // every read of this block's (W1, W2) is done
        // W1 -= K^T diag(eta) E1 ; W2 -= Hk^T diag(eta) E2
        for (int idx = threadIdx.x; idx < d * hd; idx += kThreads) {
            int i = idx / hd, m = idx % hd;
            float acc = 0.f;
            for (int j = 0; j < n; ++j) acc += es[j] * ks[j * d + i] * e1[j * hd + m];
            W1[idx] -= acc;
        }
        for (int idx = threadIdx.x; idx < hd * d; idx += kThreads) {
            int m = idx / d, c = idx % d;
            float acc = 0.f;
            for (int j = 0; j < n; ++j) acc += es[j] * hk[j * hd + m] * e2[j * d + c];
            W2[idx] -= acc;
        }
        __syncthreads();  // updated state visible to the whole CTA before the next block
    }
}

}  // namespace

size_t mlp_generic_smem_bytes(int d, int hidden, int chunk) {
    return sizeof(float) * (size_t(4) * chunk * d + size_t(3) * chunk * hidden + size_t(chunk) * chunk + chunk);
}

cudaError_t launch_mlp_prefill_generic(const MlpArgs& a, cudaStream_t s) {
    size_t bytes = mlp_generic_smem_bytes(a.d, a.hidden, a.chunk);
    cudaError_t e;
    if (a.bf16) {
        auto kern = mlp_prefill_generic_kernel<__nv_bfloat16>;
        if ((e = allow_dynamic_smem(reinterpret_cast<const void*>(kern), int(bytes))) != cudaSuccess)
            return e;
        kern<<<unsigned(a.B) * unsigned(a.H), kThreads, bytes, s>>>(
            static_cast<const __nv_bfloat16*>(a.Q), static_cast<const __nv_bfloat16*>(a.K),
            static_cast<const __nv_bfloat16*>(a.V), a.eta, a.W1_0, a.W2_0, static_cast<__nv_bfloat16*>(a.Z),
            a.W1_out, a.W2_out, a.T, a.d, a.hidden, a.chunk, static_cast<__nv_bfloat16*>(a.W1_hist),
            static_cast<__nv_bfloat16*>(a.W2_hist));
    } else {
        auto kern = mlp_prefill_generic_kernel<float>;
        if ((e = allow_dynamic_smem(reinterpret_cast<const void*>(kern), int(bytes))) != cudaSuccess)
            return e;
        kern<<<unsigned(a.B) * unsigned(a.H), kThreads, bytes, s>>>(
            static_cast<const float*>(a.Q), static_cast<const float*>(a.K), static_cast<const float*>(a.V), a.eta,
            a.W1_0, a.W2_0, static_cast<float*>(a.Z), a.W1_out, a.W2_out, a.T, a.d, a.hidden, a.chunk,
            static_cast<float*>(a.W1_hist), static_cast<float*>(a.W2_hist));
    }
    return cudaGetLastError();
}

}  // namespace ttt
