// linear_prefill_generic.cu -- SIMT fp32 TTT-Linear prefill for every supported shape.
//
// Computes, block by block (block = `chunk` tokens, the last one possibly
// shorter), the dual form of the mini-batch step:
//     E = K W0 - V;  Z = Q W0 - tril(eta . Q K^T) E;  W = W0 - K^T diag(eta) E
// ("Test-Time Training Layers ...", sections "The Core Mechanism" and
// "Hardware Parallelization"; TTT essay, paragraph on the dual form).
//
// Work split: one CTA per (batch*head, slice of NS output columns).  For f = kW
// the output columns of W, E and Z only depend on the same columns of W0 and V,
// so the slices run with no communication; each CTA recomputes the (cheap)
// Q K^T scores.  State slice, E and score tiles live in shared memory; Q/K
// tiles of TT tokens are staged through shared memory in fp32.
//
// This kernel is the reference-quality GPU path (fp32 SIMT, any d in
// {16,32,64,128}, any chunk 1..512, ragged tails, fp32 or bf16 I/O).  The
// tensor-core kernel in linear_prefill_mma.cu covers the bf16 fast path.
//
// MOM: the variant with momentum (E^2-TTT article, zhichai.net, "Technical Details and Practical
// Implications": momentum gradient descent with gradients at the chunk start; our reading: every
// token takes its own step M_i = beta M_{i-1} + g_i, W_i = W_{i-1} - eta_i M_i).  Per block of n
// tokens with start state (W, M), the exact closed form (0-based token indices):
//     Z     = Q W - diag(c) Q M - (Gam . tril(Q K^T)) E,   c_i = sum_{l<=i} eta_l beta^(l+1)
//     W_end = W - c_{n-1} M - K^T diag(Bs) E
//     M_end = beta^n M + K^T diag(beta^(n-1-j)) E
// with Bs_j = eta_j + beta Bs_{j+1} (Bs_n = 0) and Gam_ij = Bs_j - beta^(i+1-j) Bs_{i+1}, which is
// sum_{l=j..i} eta_l beta^(l-j) written without negative powers of beta.  beta = 0 gives the plain
// scan.  Column slices stay independent: M's columns evolve with E's columns.
#include "ttt_common.cuh"
#include "ttt_internal.h"

namespace ttt {
namespace {

constexpr int kThreads = 256;
constexpr int kTT = 32;       // tokens per staged tile
constexpr int kMaxChunk = 512;

template <int D>
struct GenCfg {
    static constexpr int NS = D < 16 ? D : 16;  // output columns per CTA
    static constexpr int SLICES = D / NS;
    // shared memory layout (floats)
    static constexpr int W_OFF = 0;                       // [D][NS]
    static constexpr int E_OFF = W_OFF + D * NS;          // [kMaxChunk][NS]
    static constexpr int QT_OFF = E_OFF + kMaxChunk * NS; // [kTT][D+1]
    static constexpr int KT_OFF = QT_OFF + kTT * (D + 1); // [kTT][D+1]
    static constexpr int S_OFF = KT_OFF + kTT * (D + 1);  // [kTT][kTT]
    static constexpr int ETA_OFF = S_OFF + kTT * kTT;     // [kMaxChunk]
    // momentum only: M slice, c, Bs (one more entry: Bs_n = 0)
    static constexpr int M_OFF = ETA_OFF + kMaxChunk;     // [D][NS]
    static constexpr int C_OFF = M_OFF + D * NS;          // [kMaxChunk]
    static constexpr int BS_OFF = C_OFF + kMaxChunk;      // [kMaxChunk + 1]
    static constexpr int FLOATS = BS_OFF + kMaxChunk + 1;
    static constexpr size_t BYTES = size_t(FLOATS) * sizeof(float);
};

// Stage rows [row0, row0+rows) of a [T][D] head tile into sh[kTT][D+1] (fp32).
template <typename TI, int D>
__device__ __forceinline__ void stage_rows(float* sh, const TI* src, int row0, int rows) {
    for (int idx = threadIdx.x; idx < kTT * D; idx += kThreads) {
        int r = idx / D, c = idx % D;
        sh[r * (D + 1) + c] = (r < rows) ? to_f32(src[size_t(row0 + r) * D + c]) : 0.f;
    }
}

template <typename TI, int D, bool MOM>
__global__ void __launch_bounds__(kThreads)
linear_prefill_generic_kernel(const TI* __restrict__ Q, const TI* __restrict__ K,
                              const TI* __restrict__ V, const float* __restrict__ eta,
                              const float* W0, TI* __restrict__ Z, float* W_out, int T, int chunk,
                              TI* __restrict__ W_hist, const float* M0, float* M_out, float beta) {
    using C = GenCfg<D>;
    constexpr int NS = C::NS;
    extern __shared__ float smem[];
    float* Ws = smem + C::W_OFF;
    float* Es = smem + C::E_OFF;
    float* Qt = smem + C::QT_OFF;
    float* Kt = smem + C::KT_OFF;
    float* St = smem + C::S_OFF;
    float* Et = smem + C::ETA_OFF;
    float* Ms = smem + C::M_OFF;
    float* Cs = smem + C::C_OFF;
    float* Bs = smem + C::BS_OFF;

    const size_t bh = blockIdx.x;
    const int col0 = blockIdx.y * NS;
    const TI* Qh = Q + bh * size_t(T) * D;
    const TI* Kh = K + bh * size_t(T) * D;
    const TI* Vh = V + bh * size_t(T) * D;
    const float* eh = eta + bh * size_t(T);
    TI* Zh = Z + bh * size_t(T) * D;

    for (int idx = threadIdx.x; idx < D * NS; idx += kThreads) {
        const size_t at = bh * D * D + size_t(idx / NS) * D + col0 + idx % NS;
        Ws[idx] = W0[at];
        if constexpr (MOM) Ms[idx] = M0 ? M0[at] : 0.f;
    }
    __syncthreads();

    const int nblk = (T + chunk - 1) / chunk;
    for (int t0 = 0; t0 < T; t0 += chunk) {
        const int n = min(chunk, T - t0);
        for (int j = threadIdx.x; j < n; j += kThreads) Et[j] = eh[t0 + j];
        if constexpr (MOM) {
            __syncthreads();
            if (threadIdx.x == 0) {  // the block's momentum weights: c (forward), Bs (backward)
                float acc = 0.f, bp = 1.f;
                for (int i = 0; i < n; ++i) {
                    bp *= beta;
                    acc = fmaf(Et[i], bp, acc);
                    Cs[i] = acc;
                }
                float b = 0.f;
                Bs[n] = 0.f;
                for (int j = n - 1; j >= 0; --j) {
                    b = fmaf(beta, b, Et[j]);
                    Bs[j] = b;
                }
            }
        }
        if (W_hist) {  // the state at the start of this block (this CTA's columns), as TI
            TI* wh = W_hist + (bh * nblk + t0 / chunk) * size_t(D) * D;
            for (int idx = threadIdx.x; idx < D * NS; idx += kThreads)
                wh[size_t(idx / NS) * D + col0 + idx % NS] = from_f32<TI>(Ws[idx]);
        }

        // E = K W0 - V  (this slice's columns)
        for (int jt = 0; jt < n; jt += kTT) {
            const int rows = min(kTT, n - jt);
            __syncthreads();
            stage_rows<TI, D>(Kt, Kh, t0 + jt, rows);
            __syncthreads();
            for (int idx = threadIdx.x; idx < rows * NS; idx += kThreads) {
                int j = idx / NS, c = idx % NS;
                float acc = 0.f;
#pragma unroll 8
                for (int i = 0; i < D; ++i) acc += Kt[j * (D + 1) + i] * Ws[i * NS + c];
                Es[(jt + j) * NS + c] = acc - to_f32(Vh[size_t(t0 + jt + j) * D + col0 + c]);
            }
        }

        // Z = Q W0 - tril(eta . Q K^T) E
        constexpr int ZPT = (kTT * NS + kThreads - 1) / kThreads;  // outputs per thread
        for (int it = 0; it < n; it += kTT) {
            const int rows = min(kTT, n - it);
            __syncthreads();
            stage_rows<TI, D>(Qt, Qh, t0 + it, rows);
            __syncthreads();
            float zacc[ZPT];
#pragma unroll
            for (int u = 0; u < ZPT; ++u) {
                int idx = threadIdx.x + u * kThreads;
                zacc[u] = 0.f;
                if (idx < kTT * NS) {
                    int i = idx / NS, c = idx % NS;
                    float acc = 0.f, accm = 0.f;
#pragma unroll 8
                    for (int k = 0; k < D; ++k) {
                        acc += Qt[i * (D + 1) + k] * Ws[k * NS + c];
                        if constexpr (MOM) accm += Qt[i * (D + 1) + k] * Ms[k * NS + c];
                    }
                    if constexpr (MOM) {
                        if (i < rows) acc = fmaf(-Cs[it + i], accm, acc);
                    }
                    zacc[u] = acc;
                }
            }
            for (int jt = 0; jt <= it; jt += kTT) {
                const int krows = min(kTT, n - jt);
                __syncthreads();
                stage_rows<TI, D>(Kt, Kh, t0 + jt, krows);
                __syncthreads();
                for (int idx = threadIdx.x; idx < kTT * kTT; idx += kThreads) {
                    int i = idx / kTT, j = idx % kTT;
                    float s = 0.f;
                    if (i < rows && j < krows && jt + j <= it + i) {
#pragma unroll 8
                        for (int k = 0; k < D; ++k) s += Qt[i * (D + 1) + k] * Kt[j * (D + 1) + k];
                        if constexpr (MOM) {
                            const int qi = it + i, kj = jt + j;  // Gam_ij = Bs_j - beta^(i+1-j) Bs_{i+1}
                            s *= Bs[kj] - powf(beta, float(qi + 1 - kj)) * Bs[qi + 1];
                        } else {
                            s *= Et[jt + j];
                        }
                    }
                    St[idx] = s;
                }
                __syncthreads();
#pragma unroll
                for (int u = 0; u < ZPT; ++u) {
                    int idx = threadIdx.x + u * kThreads;
                    if (idx < kTT * NS) {
                        int i = idx / NS, c = idx % NS;
                        float acc = 0.f;
                        for (int j = 0; j < krows; ++j) acc += St[i * kTT + j] * Es[(jt + j) * NS + c];
                        zacc[u] -= acc;
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < ZPT; ++u) {
                int idx = threadIdx.x + u * kThreads;
                if (idx < kTT * NS) {
                    int i = idx / NS, c = idx % NS;
                    if (i < rows) Zh[size_t(t0 + it + i) * D + col0 + c] = from_f32<TI>(zacc[u]);
                }
            }
        }

        // W = W0 - K^T diag(eta) E  (momentum: W0 - c_{n-1} M - K^T diag(Bs) E and
        // M = beta^n M + K^T diag(beta^(n-1-j)) E)
        constexpr int WPT = (D * NS + kThreads - 1) / kThreads;
        float wacc[WPT], macc[WPT];
#pragma unroll
        for (int u = 0; u < WPT; ++u) wacc[u] = macc[u] = 0.f;
        for (int jt = 0; jt < n; jt += kTT) {
            const int rows = min(kTT, n - jt);
            __syncthreads();
            stage_rows<TI, D>(Kt, Kh, t0 + jt, rows);
            __syncthreads();
#pragma unroll
            for (int u = 0; u < WPT; ++u) {
                int idx = threadIdx.x + u * kThreads;
                if (idx < D * NS) {
                    int k = idx / NS, c = idx % NS;
                    float acc = 0.f, accm = 0.f;
                    for (int j = 0; j < rows; ++j) {
                        const float ke = Kt[j * (D + 1) + k] * Es[(jt + j) * NS + c];
                        if constexpr (MOM) {
                            acc += Bs[jt + j] * ke;
                            accm += powf(beta, float(n - 1 - (jt + j))) * ke;
                        } else {
                            acc += Et[jt + j] * ke;
                        }
                    }
                    wacc[u] += acc;
                    macc[u] += accm;
                }
            }
        }
        __syncthreads();
#pragma unroll
        for (int u = 0; u < WPT; ++u) {
            int idx = threadIdx.x + u * kThreads;
            if (idx < D * NS) {
                if constexpr (MOM) {
                    const float m = Ms[idx];
                    Ws[idx] -= fmaf(Cs[n - 1], m, wacc[u]);
                    Ms[idx] = fmaf(powf(beta, float(n)), m, macc[u]);
                } else {
                    Ws[idx] -= wacc[u];
                }
            }
        }
        __syncthreads();
    }

    for (int idx = threadIdx.x; idx < D * NS; idx += kThreads) {
        const size_t at = bh * D * D + size_t(idx / NS) * D + col0 + idx % NS;
        W_out[at] = Ws[idx];
        if constexpr (MOM) M_out[at] = Ms[idx];
    }
}

template <typename TI, int D>
cudaError_t launch_d(const LinearArgs& a, cudaStream_t s) {
    using C = GenCfg<D>;
    if (a.momentum) {
        auto kern = linear_prefill_generic_kernel<TI, D, true>;
        cudaError_t e = allow_dynamic_smem(reinterpret_cast<const void*>(kern), int(C::BYTES));
        if (e != cudaSuccess) return e;
        dim3 grid(unsigned(a.B) * unsigned(a.H), C::SLICES);
        kern<<<grid, kThreads, C::BYTES, s>>>(static_cast<const TI*>(a.Q), static_cast<const TI*>(a.K),
                                              static_cast<const TI*>(a.V), a.eta, a.W0, static_cast<TI*>(a.Z),
                                              a.W_out, a.T, a.chunk, nullptr, a.M0, a.M_out, a.beta);
        return cudaGetLastError();
    }
    auto kern = linear_prefill_generic_kernel<TI, D, false>;
    cudaError_t e = allow_dynamic_smem(reinterpret_cast<const void*>(kern), int(C::BYTES));
    if (e != cudaSuccess) return e;
    dim3 grid(unsigned(a.B) * unsigned(a.H), C::SLICES);
    kern<<<grid, kThreads, C::BYTES, s>>>(static_cast<const TI*>(a.Q), static_cast<const TI*>(a.K),
                                          static_cast<const TI*>(a.V), a.eta, a.W0,
                                          static_cast<TI*>(a.Z), a.W_out, a.T, a.chunk, static_cast<TI*>(a.W_hist),
                                          nullptr, nullptr, 0.f);
    return cudaGetLastError();
}

template <typename TI>
cudaError_t launch_t(const LinearArgs& a, cudaStream_t s) {
    switch (a.d) {
        case 16: return launch_d<TI, 16>(a, s);
        case 32: return launch_d<TI, 32>(a, s);
        case 64: return launch_d<TI, 64>(a, s);
        case 128: return launch_d<TI, 128>(a, s);
        default: return cudaErrorNotSupported;
    }
}

}  // namespace

cudaError_t launch_linear_prefill_generic(const LinearArgs& a, cudaStream_t s) {
    if (a.chunk > kMaxChunk) return cudaErrorNotSupported;
    return a.bf16 ? launch_t<__nv_bfloat16>(a, s) : launch_t<float>(a, s);
}

}  // namespace ttt
