// linear_backward.cu -- gradient of the TTT-Linear chunked scan (SIMT, fp32).
//
// Training the outer model goes through the inner loop: the slow weights learn the
// initialisation and the update rule of the fast weights (TTT essay, ren-xubin.github.io,
// paragraph on the two time scales).  Given the gradients of a scalar loss with respect to the
// outputs Z and to the final state, this computes them with respect to Q, K, V, eta and W0.
//
// Forward definitions, per block of b tokens with start state W (the dual form of the
// mini-batch step: "Test-Time Training Layers ...", sections "The Core Mechanism" and
// "Hardware Parallelization"; TTT essay, paragraph on the dual form):
//     E = K W - V,  A = tril(Q K^T) diag(eta),  Z = Q W - A E,  W' = W - K^T diag(eta) E.
// Their chain rule, block by block in reverse, with dW' the gradient carried back from the next
// block (D = diag(eta), M the causal mask j <= i, S = Q K^T):
//     dE = -A^T dZ - D K dW'          dA = -dZ E^T,  dS = M . dA D
//     dQ = dZ W^T + dS K              dK = dE W^T - D E dW'^T + dS^T Q
//     dV = -dE                        deta_j = -sum_c E_jc (K dW')_jc + sum_i M_ij dA_ij S_ij
//     dW = dW' + Q^T dZ + K^T dE      (carried to the previous block; dW0 at the end)
// The block-start states W come from the forward pass (ttt_linear_prefill_hist), in the element
// type of Q (bf16 runs record the state rounded to bf16, the operand the forward's products used).
//
// One CTA per (batch, head): dQ, dK and deta sum over every output column, so the column split
// of the forward kernels does not apply.  The block's tiles, both states and the b x b score
// tiles live in shared memory (fp32, rows padded by one word against bank conflicts); this
// bounds chunk * d (linear_backward_supported).
#include "ttt_common.cuh"
#include "ttt_internal.h"

namespace ttt {
namespace {

constexpr int kThreads = 256;

template <int D>
struct BwdSmem {
    static constexpr int LD = D + 1;  // padded row of a [*][D] tile
    // floats: W, dW [D][LD]; Q, K, V, dZ, E, dE, K dW' [b][LD]; S, dA [b][b + 1]; eta [b]
    static size_t bytes(int b) {
        return sizeof(float) * (size_t(2) * D * LD + size_t(7) * b * LD + size_t(2) * b * (b + 1) + b);
    }
};

template <typename TI, int D>
__device__ __forceinline__ void load_tile(float* sh, const TI* src, int rows) {
    constexpr int LD = D + 1;
    for (int idx = threadIdx.x; idx < rows * D; idx += kThreads) sh[(idx / D) * LD + idx % D] = to_f32(src[idx]);
}

template <typename TI, int D>
__global__ void __launch_bounds__(kThreads)
linear_backward_kernel(const TI* __restrict__ Q, const TI* __restrict__ K, const TI* __restrict__ V,
                       const float* __restrict__ eta, const TI* __restrict__ W_hist, const TI* __restrict__ dZ,
                       const float* __restrict__ dW_T, TI* __restrict__ dQ, TI* __restrict__ dK,
                       TI* __restrict__ dV, float* __restrict__ deta, float* __restrict__ dW0, int T, int chunk) {
    constexpr int LD = D + 1;
    const int b = chunk, BL = chunk + 1;
    extern __shared__ float sm[];
    float* Ws = sm;                      // [D][LD]   state at the block start
    float* dWs = Ws + D * LD;            // [D][LD]   gradient of the state after the block
    float* Qs = dWs + D * LD;            // [b][LD]
    float* Ks = Qs + b * LD;
    float* Vs = Ks + b * LD;
    float* dZs = Vs + b * LD;
    float* Es = dZs + b * LD;            // E = K W - V
    float* dEs = Es + b * LD;            // dE
    float* KdW = dEs + b * LD;           // K dW'
    float* Ss = KdW + b * LD;            // [b][BL]   S = Q K^T
    float* dAs = Ss + b * BL;            // [b][BL]   dA = -dZ E^T (masked)
    float* es = dAs + b * BL;            // [b]

    const size_t bh = blockIdx.x;
    const int nblk = (T + chunk - 1) / chunk;
    const size_t hd = bh * size_t(T) * D;

    for (int idx = threadIdx.x; idx < D * D; idx += kThreads)
        dWs[(idx / D) * LD + idx % D] = dW_T ? dW_T[bh * D * D + idx] : 0.f;

    for (int n = nblk - 1; n >= 0; --n) {
        const int t0 = n * chunk, rows = min(chunk, T - t0);
        const size_t base = hd + size_t(t0) * D;
        __syncthreads();  // the previous (later) block is done with every tile
        const TI* Wn = W_hist + (bh * nblk + n) * size_t(D) * D;
        for (int idx = threadIdx.x; idx < D * D; idx += kThreads) Ws[(idx / D) * LD + idx % D] = to_f32(Wn[idx]);
        load_tile<TI, D>(Qs, Q + base, rows);
        load_tile<TI, D>(Ks, K + base, rows);
        load_tile<TI, D>(Vs, V + base, rows);
        load_tile<TI, D>(dZs, dZ + base, rows);
        for (int j = threadIdx.x; j < rows; j += kThreads) es[j] = eta[bh * size_t(T) + t0 + j];
        __syncthreads();

        // E = K W - V,  K dW'  (rows x D each);  S = Q K^T  (rows x rows, lower triangle)
        for (int idx = threadIdx.x; idx < rows * D; idx += kThreads) {
            const int j = idx / D, c = idx % D;
            float e = 0.f, kd = 0.f;
#pragma unroll 8
            for (int k = 0; k < D; ++k) {
                const float kv = Ks[j * LD + k];
                e = fmaf(kv, Ws[k * LD + c], e);
                kd = fmaf(kv, dWs[k * LD + c], kd);
            }
            Es[j * LD + c] = e - Vs[j * LD + c];
            KdW[j * LD + c] = kd;
        }
        for (int idx = threadIdx.x; idx < rows * rows; idx += kThreads) {
            const int i = idx / rows, j = idx % rows;
            float s = 0.f;
            if (j <= i) {
#pragma unroll 8
                for (int k = 0; k < D; ++k) s = fmaf(Qs[i * LD + k], Ks[j * LD + k], s);
            }
            Ss[i * BL + j] = s;
        }
        __syncthreads();

        // dA = -dZ E^T on the mask;  dE = -eta_j (K dW')_j - eta_j sum_{i >= j} S_ij dZ_i
        for (int idx = threadIdx.x; idx < rows * rows; idx += kThreads) {
            const int i = idx / rows, j = idx % rows;
            float a = 0.f;
            if (j <= i) {
#pragma unroll 8
                for (int c = 0; c < D; ++c) a = fmaf(dZs[i * LD + c], Es[j * LD + c], a);
            }
            dAs[i * BL + j] = -a;
        }
        for (int idx = threadIdx.x; idx < rows * D; idx += kThreads) {
            const int j = idx / D, c = idx % D;
            float acc = KdW[j * LD + c];
            for (int i = j; i < rows; ++i) acc = fmaf(Ss[i * BL + j], dZs[i * LD + c], acc);
            dEs[j * LD + c] = -es[j] * acc;
        }
        __syncthreads();

        // dQ, dK, dV, deta of this block's tokens
        for (int idx = threadIdx.x; idx < rows * D; idx += kThreads) {
            const int i = idx / D, k = idx % D;
            float q = 0.f, kk = 0.f, ku = 0.f;
#pragma unroll 8
            for (int c = 0; c < D; ++c) {
                q = fmaf(dZs[i * LD + c], Ws[k * LD + c], q);     // (dZ W^T)_ik
                kk = fmaf(dEs[i * LD + c], Ws[k * LD + c], kk);   // (dE W^T)_ik
                ku = fmaf(Es[i * LD + c], dWs[k * LD + c], ku);   // (E dW'^T)_ik
            }
            for (int j = 0; j <= i; ++j) q = fmaf(dAs[i * BL + j] * es[j], Ks[j * LD + k], q);
            kk = fmaf(-es[i], ku, kk);
            for (int r = i; r < rows; ++r) kk = fmaf(dAs[r * BL + i] * es[i], Qs[r * LD + k], kk);
            dQ[base + size_t(i) * D + k] = from_f32<TI>(q);
            dK[base + size_t(i) * D + k] = from_f32<TI>(kk);
            dV[base + size_t(i) * D + k] = from_f32<TI>(-dEs[i * LD + k]);
        }
        for (int j = threadIdx.x; j < rows; j += kThreads) {
            float de = 0.f;
            for (int c = 0; c < D; ++c) de = fmaf(Es[j * LD + c], KdW[j * LD + c], de);
            de = -de;
            for (int i = j; i < rows; ++i) de = fmaf(dAs[i * BL + j], Ss[i * BL + j], de);
            deta[bh * size_t(T) + t0 + j] = de;
        }
        __syncthreads();  // every reader of dW' is done

        // dW = dW' + Q^T dZ + K^T dE
        for (int idx = threadIdx.x; idx < D * D; idx += kThreads) {
            const int k = idx / D, c = idx % D;
            float acc = dWs[k * LD + c];
            for (int i = 0; i < rows; ++i) {
                acc = fmaf(Qs[i * LD + k], dZs[i * LD + c], acc);
                acc = fmaf(Ks[i * LD + k], dEs[i * LD + c], acc);
            }
            dWs[k * LD + c] = acc;
        }
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < D * D; idx += kThreads) dW0[bh * D * D + idx] = dWs[(idx / D) * LD + idx % D];
}

template <typename TI, int D>
cudaError_t launch_d(const LinearBwdArgs& a, cudaStream_t s) {
    auto kern = linear_backward_kernel<TI, D>;
    const size_t bytes = BwdSmem<D>::bytes(a.chunk);
    cudaError_t e = allow_dynamic_smem(reinterpret_cast<const void*>(kern), int(bytes));
    if (e != cudaSuccess) return e;
    kern<<<unsigned(a.B) * unsigned(a.H), kThreads, bytes, s>>>(
        static_cast<const TI*>(a.Q), static_cast<const TI*>(a.K), static_cast<const TI*>(a.V), a.eta,
        static_cast<const TI*>(a.W_hist),
        static_cast<const TI*>(a.dZ), a.dW_T, static_cast<TI*>(a.dQ), static_cast<TI*>(a.dK), static_cast<TI*>(a.dV),
        a.deta, a.dW0, a.T, a.chunk);
    return cudaGetLastError();
}

template <typename TI>
cudaError_t launch_t(const LinearBwdArgs& a, cudaStream_t s) {
    switch (a.d) {
        case 16: return launch_d<TI, 16>(a, s);
        case 32: return launch_d<TI, 32>(a, s);
        case 64: return launch_d<TI, 64>(a, s);
        case 128: return launch_d<TI, 128>(a, s);
        default: return cudaErrorNotSupported;
    }
}

}  // namespace

bool linear_backward_supported(int d, int chunk) {
    size_t bytes = 0;
    switch (d) {
        case 16: bytes = BwdSmem<16>::bytes(chunk); break;
        case 32: bytes = BwdSmem<32>::bytes(chunk); break;
        case 64: bytes = BwdSmem<64>::bytes(chunk); break;
        case 128: bytes = BwdSmem<128>::bytes(chunk); break;
        default: return false;
    }
    return chunk >= 1 && bytes <= 227 * 1024;
}

cudaError_t launch_linear_backward(const LinearBwdArgs& a, cudaStream_t s) {
    if (!linear_backward_supported(a.d, a.chunk)) return cudaErrorNotSupported;
    return a.bf16 ? launch_t<__nv_bfloat16>(a, s) : launch_t<float>(a, s);
}

}  // namespace ttt
