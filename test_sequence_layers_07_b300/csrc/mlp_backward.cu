// mlp_backward.cu -- gradient of the TTT-MLP chunked scan (SIMT, fp32 accumulation).
//
// Training the outer model goes through the inner loop (TTT essay, ren-xubin.github.io, paragraph on
// the two time scales).  Given dZ and the gradients of the final state (dW1_T, dW2_T), this computes
// dQ, dK, dV, deta and the gradients of the initial state.
//
// Forward, per block with start state (W1, W2), D = diag(eta), M the causal mask (j <= i), g = GELU
// in its tanh form ("Test-Time Training (TTT) Layers for Sequence Modeling", section "Variants:
// TTT-Linear vs. TTT-MLP"; loss, step and read-out of "Test-Time Training Layers ...", section
// "The Core Mechanism"):
//   Zk = K W1, Hk = g(Zk), E2 = Hk W2 - V, Gk = E2 W2^T, E1 = Gk . g'(Zk),
//   Zq = Q W1 - (M . Q K^T) D E1, Hq = g(Zq), Z = Hq W2 - (M . Hq Hk^T) D E2,
//   W1' = W1 - K^T D E1, W2' = W2 - Hk^T D E2.
// Chain rule, block by block in reverse (dW1', dW2' the gradients of the state after the block):
//   W':  dHk = -D E2 dW2'^T, dE2 = -D Hk dW2', dK = -D E1 dW1'^T, dE1 = -D K dW1',
//        deta_j = -(Hk dW2')_j . E2_j - (K dW1')_j . E1_j
//   Z:   dHq = dZ W2^T, dA2 = -dZ E2^T (masked), dE2 -= (M . Hq Hk^T D)^T dZ
//   A2:  deta_j += sum_i M_ij (Hq Hk^T)_ij dA2_ij, dS2 = M . dA2 D, dHq += dS2 Hk, dHk += dS2^T Hq
//   Zq:  dZq = dHq . g'(Zq), dQ = dZq W1^T, dA1 = -dZq E1^T (masked), dE1 -= (M . Q K^T D)^T dZq
//   A1:  deta_j += sum_i M_ij (Q K^T)_ij dA1_ij, dS1 = M . dA1 D, dQ += dS1 K, dK += dS1^T Q
//   E1:  dGk = dE1 . g'(Zk), dZk = dE1 . Gk . g''(Zk)
//   Gk:  dE2 += dGk W2;   E2: dV = -dE2, dHk += dE2 W2^T;   dZk += dHk . g'(Zk);   dK += dZk W1^T
//   dW2 = dW2' + Hq^T dZ + dGk^T E2 + Hk^T dE2,   dW1 = dW1' + Q^T dZq + K^T dZk.
// The block-start states come from the forward (ttt_mlp_prefill_hist), in the element type of Q.
//
// One CTA of 512 threads per (batch, head).  The block's intermediates (ten b x h tiles, six b x d,
// four b x b) live in shared memory in fp32; W1, W2 of the block are read from the recorded states
// (L2).  A thread that needs a whole row of W2 (or of the running dW2) reads it with 16-byte loads:
// one element per load would touch a 32-byte sector per 2- or 4-byte value, neighbouring threads
// being a row (128 or 256 bytes) apart.  The running state gradient lives in dW1_0 / dW2_0 (fp32, L2-resident): every thread owns a
// fixed set of their entries and adds its updates once per block, after the block's products have
// read them as dW1', dW2'.  Products that sum over the hidden dimension are split over groups of
// threads and summed through shared memory.
#include "ttt_common.cuh"
#include "ttt_internal.h"

namespace ttt {
namespace {

constexpr int kNT = 512;
constexpr int kRed = 4096;  // floats of the buffer through which sums over the hidden dimension are reduced

__device__ __forceinline__ float g_tanh(float x, float* gp, float* gpp) {
    const float c = 0.7978845608028654f, a = 0.044715f;
    const float t = tanhf(c * (x + a * x * x * x));
    const float u1 = c * (1.f + 3.f * a * x * x), s = 1.f - t * t;
    if (gp) *gp = 0.5f * (1.f + t) + 0.5f * x * s * u1;
    if (gpp) *gpp = s * u1 + 0.5f * x * s * (6.f * a * c * x - 2.f * t * u1 * u1);
    return 0.5f * x * (1.f + t);
}
__device__ __forceinline__ float g_prime(float x) {
    float gp;
    g_tanh(x, &gp, nullptr);
    return gp;
}

// the D elements of a row that starts on a 16-byte boundary into registers, in 16-byte pieces (the
// entry point rejects buffers that do not start on one; d, h and d * h are multiples of 16)
template <int D>
__device__ __forceinline__ void load_row(const float* p, float (&out)[D]) {
    const float4* q = reinterpret_cast<const float4*>(p);
#pragma unroll
    for (int u = 0; u < D / 4; ++u) {
        const float4 v = q[u];
        out[4 * u] = v.x, out[4 * u + 1] = v.y, out[4 * u + 2] = v.z, out[4 * u + 3] = v.w;
    }
}
template <int D>
__device__ __forceinline__ void load_row(const __nv_bfloat16* p, float (&out)[D]) {
    const uint4* q = reinterpret_cast<const uint4*>(p);
#pragma unroll
    for (int u = 0; u < D / 8; ++u) {
        const uint4 v = q[u];
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {  // a bf16 is the top half of an fp32
            out[8 * u + 2 * e] = __uint_as_float(w[e] << 16);
            out[8 * u + 2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
        }
    }
}

// the second operand of a sum over the hidden index, Y(m, c): a [h][d] matrix (W2 and dW2: the eight
// values of m..m+7 for column c sit d apart, one load each, coalesced across c) or a [d][h] one (W1
// and dW1: the eight sit side by side in row c, read as 16-byte pieces when m is a multiple of 8)
template <typename E>
struct ByRow {
    const E* p;
    int ld;
    __device__ float operator()(int m, int c) const { return to_f32(p[size_t(m) * ld + c]); }
    __device__ void eight(int m, int c, bool, float (&y)[8]) const {
#pragma unroll
        for (int u = 0; u < 8; ++u) y[u] = (*this)(m + u, c);
    }
};
template <typename E>
struct ByCol {
    const E* p;
    int ld;
    __device__ float operator()(int m, int c) const { return to_f32(p[size_t(c) * ld + m]); }
    __device__ void eight(int m, int c, bool vec, float (&y)[8]) const {
        if (vec) {
            load_row<8>(p + size_t(c) * ld + m, y);
        } else {
#pragma unroll
            for (int u = 0; u < 8; ++u) y[u] = (*this)(m + u, c);
        }
    }
};

struct Lay {
    int b, d, h, LD, LH, LB;
    size_t off[24];
    size_t floats;
    __host__ __device__ Lay(int b_, int d_, int h_) : b(b_), d(d_), h(h_), LD(d_ + 1), LH(h_ + 1), LB(b_ + 1) {
        size_t o = 0;
        for (int i = 0; i < 6; ++i) { off[i] = o; o += size_t(b) * LD; }        // Q K V dZ E2 dE2
        for (int i = 6; i < 16; ++i) { off[i] = o; o += size_t(b) * LH; }       // 10 b x h tiles
        for (int i = 16; i < 20; ++i) { off[i] = o; o += size_t(b) * LB; }      // S1 S2 dA1 dA2
        off[20] = o; o += size_t(b) * LD;                                        // dQ
        off[21] = o; o += size_t(b) * LD;                                        // dK
        off[22] = o; o += kRed;                                                  // sums over hidden groups
        off[23] = o; o += 2 * size_t(b);                                         // eta, deta
        floats = o;
    }
};

// sum over the hidden index m of X[j][m] * Y(m, c) for all j < b, c < d, into out[j][c] (+= when add):
// thread t takes column c = t % d, hidden group (t / d) % groups (as many groups as `red` holds
// partials for) and the tokens j = js, js + split, ... (js = t / (d * groups)), so that every thread
// has a share; partials go through `red`.
template <typename FY>
__device__ void hidden_sum(const float* X, int LH, int b, int d, int h, FY Y, float* red, float* out, int LD,
                           bool add, float scale) {
    const int groups = min(kNT / d, kRed / (b * d)), per = (h + groups - 1) / groups;
    const bool v8 = per % 8 == 0;  // every group's first m, and so every eight, on a 16-byte boundary
    const int split = kNT / (groups * d);
    const int t = threadIdx.x, c = t % d, grp = (t / d) % groups, js = t / (d * groups);
    float acc[16];
#pragma unroll
    for (int u = 0; u < 16; ++u) acc[u] = 0.f;
    {
        const int m0 = grp * per, m1 = min(h, m0 + per);
        // eight Y values in flight at a time: Y reads the block's recorded state or the running
        // gradient from L2, so loading them one dependent step at a time would be latency-bound
        int m = m0;
        for (; m + 8 <= m1; m += 8) {
            float y[8];
            Y.eight(m, c, v8, y);
#pragma unroll
            for (int u = 0; u < 8; ++u)
#pragma unroll
                for (int q = 0; q < 16; ++q)
                    if (js + q * split < b) acc[q] = fmaf(X[(js + q * split) * LH + m + u], y[u], acc[q]);
        }
        for (; m < m1; ++m) {
            const float y = Y(m, c);
#pragma unroll
            for (int q = 0; q < 16; ++q)
                if (js + q * split < b) acc[q] = fmaf(X[(js + q * split) * LH + m], y, acc[q]);
        }
#pragma unroll
        for (int q = 0; q < 16; ++q)
            if (js + q * split < b) red[(size_t(grp) * b + js + q * split) * d + c] = acc[q];
    }
    __syncthreads();
    for (int idx = t; idx < b * d; idx += kNT) {
        const int j = idx / d, cc = idx % d;
        float s = 0.f;
        for (int gg = 0; gg < groups; ++gg) s += red[(size_t(gg) * b + j) * d + cc];
        out[j * LD + cc] = add ? fmaf(scale, s, out[j * LD + cc]) : scale * s;
    }
    __syncthreads();
}

template <typename TI, int D>
__global__ void __launch_bounds__(kNT, 1)
mlp_backward_kernel(const TI* __restrict__ Q, const TI* __restrict__ K, const TI* __restrict__ V,
                    const float* __restrict__ eta, const TI* __restrict__ W1_hist, const TI* __restrict__ W2_hist,
                    const TI* __restrict__ dZ, const float* dW1_T, const float* dW2_T, TI* __restrict__ dQ,
                    TI* __restrict__ dK, TI* __restrict__ dV, float* __restrict__ deta, float* dW1g, float* dW2g,
                    int T, int h, int chunk) {
    constexpr int d = D;  // compile-time, so the per-thread rows of W stay in registers
    extern __shared__ float sm[];
    const Lay L(chunk, d, h);
    const int LD = L.LD, LH = L.LH, LB = L.LB;
    float *Qs = sm + L.off[0], *Ks = sm + L.off[1], *Vs = sm + L.off[2], *dZs = sm + L.off[3];
    float *E2 = sm + L.off[4], *dE2 = sm + L.off[5];
    float *Zk = sm + L.off[6], *Hk = sm + L.off[7], *Gk = sm + L.off[8], *E1 = sm + L.off[9];
    float *Zq = sm + L.off[10], *Hq = sm + L.off[11], *dHk = sm + L.off[12], *dHq = sm + L.off[13];
    float *dE1 = sm + L.off[14], *dZk = sm + L.off[15];
    float *S1 = sm + L.off[16], *S2 = sm + L.off[17], *dA1 = sm + L.off[18], *dA2 = sm + L.off[19];
    float *dQs = sm + L.off[20], *dKs = sm + L.off[21], *red = sm + L.off[22];
    float *es = sm + L.off[23], *des = es + chunk;

    const int t = threadIdx.x;
    const size_t bh = blockIdx.x;
    const size_t nw = size_t(d) * h;
    const int nblk = (T + chunk - 1) / chunk;
    dW1g += bh * nw;
    dW2g += bh * nw;
    // the running gradient starts at dW_T (zero when absent); dW_T may be the same buffer as dW_0
    // this thread's entries of dW1 ([d][h], idx -> (idx / h, idx % h)) and dW2 ([h][d], (idx / d, idx % d)):
    // idx = t, t + kNT, ...
    for (size_t idx = t; idx < nw; idx += kNT) {
        const float a1 = dW1_T ? dW1_T[bh * nw + idx] : 0.f;
        const float a2 = dW2_T ? dW2_T[bh * nw + idx] : 0.f;
        dW1g[idx] = a1;
        dW2g[idx] = a2;
    }

    // thread -> (hidden unit m, token group): the "row of W" products
    const int jgroups = kNT / h, mm = t % h, jg = t / h;

    for (int n = nblk - 1; n >= 0; --n) {
        const int t0 = n * chunk, b = min(chunk, T - t0);
        const size_t base = bh * size_t(T) * d + size_t(t0) * d;
        const TI* W1 = W1_hist + (bh * nblk + n) * nw;  // [d][h]
        const TI* W2 = W2_hist + (bh * nblk + n) * nw;  // [h][d]
        __syncthreads();  // the previous block is done with every tile and its dW writes are visible
        for (int idx = t; idx < chunk * d; idx += kNT) {
            const int j = idx / d, c = idx % d;
            const bool in = j < b;
            Qs[j * LD + c] = in ? to_f32(Q[base + idx]) : 0.f;
            Ks[j * LD + c] = in ? to_f32(K[base + idx]) : 0.f;
            Vs[j * LD + c] = in ? to_f32(V[base + idx]) : 0.f;
            dZs[j * LD + c] = in ? to_f32(dZ[base + idx]) : 0.f;
            dQs[j * LD + c] = 0.f;
            dKs[j * LD + c] = 0.f;
        }
        for (int j = t; j < chunk; j += kNT) {
            es[j] = j < b ? eta[bh * size_t(T) + t0 + j] : 0.f;
            des[j] = 0.f;
        }
        __syncthreads();

        // ---- forward quantities of the block at its start state
        // Zk = K W1, Zq = Q W1 (thread: hidden unit mm, tokens jg, jg + jgroups, ...)
        if (jg < jgroups) {
            float wcol[D];
            for (int k = 0; k < d; ++k) wcol[k] = to_f32(W1[size_t(k) * h + mm]);
            for (int j = jg; j < b; j += jgroups) {
                float zk = 0.f, zq = 0.f;
                for (int k = 0; k < d; ++k) {
                    zk = fmaf(Ks[j * LD + k], wcol[k], zk);
                    zq = fmaf(Qs[j * LD + k], wcol[k], zq);
                }
                Zk[j * LH + mm] = zk;
                Hk[j * LH + mm] = g_tanh(zk, nullptr, nullptr);
                Zq[j * LH + mm] = zq;
            }
        }
        __syncthreads();
        // E2 = Hk W2 - V
        hidden_sum(Hk, LH, b, d, h, ByRow<TI>{W2, d}, red, E2, LD, false, 1.f);
        for (int idx = t; idx < b * d; idx += kNT) E2[(idx / d) * LD + idx % d] -= Vs[(idx / d) * LD + idx % d];
        // S1 = Q K^T on the mask
        for (int idx = t; idx < b * b; idx += kNT) {
            const int i = idx / b, j = idx % b;
            float s = 0.f;
            if (j <= i)
                for (int k = 0; k < d; ++k) s = fmaf(Qs[i * LD + k], Ks[j * LD + k], s);
            S1[i * LB + j] = s;
        }
        __syncthreads();
        // Gk = E2 W2^T, E1 = Gk . g'(Zk)
        if (jg < jgroups) {
            float wrow[D];
            load_row(W2 + size_t(mm) * d, wrow);
            for (int j = jg; j < b; j += jgroups) {
                float gk = 0.f;
                for (int c = 0; c < d; ++c) gk = fmaf(E2[j * LD + c], wrow[c], gk);
                Gk[j * LH + mm] = gk;
                E1[j * LH + mm] = gk * g_prime(Zk[j * LH + mm]);
            }
        }
        __syncthreads();
        // Zq -= (M . S1 D) E1; Hq = g(Zq)
        for (int idx = t; idx < b * h; idx += kNT) {
            const int i = idx / h, m = idx % h;
            float z = Zq[i * LH + m];
            for (int j = 0; j <= i; ++j) z = fmaf(-es[j] * S1[i * LB + j], E1[j * LH + m], z);
            Zq[i * LH + m] = z;
            Hq[i * LH + m] = g_tanh(z, nullptr, nullptr);
        }
        __syncthreads();
        // S2 = Hq Hk^T on the mask
        for (int idx = t; idx < b * b; idx += kNT) {
            const int i = idx / b, j = idx % b;
            float s = 0.f;
            if (j <= i)
                for (int m = 0; m < h; ++m) s = fmaf(Hq[i * LH + m], Hk[j * LH + m], s);
            S2[i * LB + j] = s;
        }
        __syncthreads();

        // ---- the state update W2' = W2 - Hk^T D E2, W1' = W1 - K^T D E1 (dW' in dW1g / dW2g)
        // dHk = -D E2 dW2'^T and dE1 = -D K dW1' (thread: hidden unit mm)
        if (jg < jgroups) {
            float r[D];  // row mm of dW2', then column mm of dW1' (one at a time: both would spill)
            load_row(dW2g + size_t(mm) * d, r);
            for (int j = jg; j < b; j += jgroups) {
                float a2 = 0.f;
                for (int c = 0; c < d; ++c) a2 = fmaf(E2[j * LD + c], r[c], a2);
                dHk[j * LH + mm] = -es[j] * a2;
            }
            for (int k = 0; k < d; ++k) r[k] = dW1g[size_t(k) * h + mm];
            for (int j = jg; j < b; j += jgroups) {
                float a1 = 0.f;
                for (int k = 0; k < d; ++k) a1 = fmaf(Ks[j * LD + k], r[k], a1);
                dE1[j * LH + mm] = -es[j] * a1;
                dZk[j * LH + mm] = a1 * E1[j * LH + mm];  // (K dW1')_jm E1_jm, summed over m below
            }
        }
        // dE2 = -D (Hk dW2'), with deta_j -= (Hk dW2')_j . E2_j
        hidden_sum(Hk, LH, b, d, h, ByRow<float>{dW2g, d}, red, dE2, LD, false, 1.f);
        // deta_j = -(Hk dW2')_j . E2_j - (K dW1')_j . E1_j, summed in a fixed order (deterministic)
        for (int j = t; j < b; j += kNT) {
            float s = 0.f, s1 = 0.f;
            for (int c = 0; c < d; ++c) s = fmaf(dE2[j * LD + c], E2[j * LD + c], s);
            for (int m = 0; m < h; ++m) s1 += dZk[j * LH + m];
            des[j] = -s - s1;
        }
        __syncthreads();
        for (int idx = t; idx < b * d; idx += kNT) dE2[(idx / d) * LD + idx % d] *= -es[idx / d];
        // dK = -D E1 dW1'^T: sum over m of E1[j][m] dW1'[k][m]
        hidden_sum(E1, LH, b, d, h, ByCol<float>{dW1g, h}, red, dKs, LD, false, 1.f);
        for (int idx = t; idx < b * d; idx += kNT) dKs[(idx / d) * LD + idx % d] *= -es[idx / d];

        // ---- Z = Hq W2 - (M . S2 D) E2
        // dHq = dZ W2^T
        if (jg < jgroups) {
            float wrow[D];
            load_row(W2 + size_t(mm) * d, wrow);
            for (int i = jg; i < b; i += jgroups) {
                float a = 0.f;
                for (int c = 0; c < d; ++c) a = fmaf(dZs[i * LD + c], wrow[c], a);
                dHq[i * LH + mm] = a;
            }
        }
        // dA2 = -dZ E2^T on the mask
        for (int idx = t; idx < b * b; idx += kNT) {
            const int i = idx / b, j = idx % b;
            float s = 0.f;
            if (j <= i)
                for (int c = 0; c < d; ++c) s = fmaf(dZs[i * LD + c], E2[j * LD + c], s);
            dA2[i * LB + j] = -s;
        }
        __syncthreads();
        // dE2 -= (M . S2 D)^T dZ;  deta_j += sum_i M dA2 S2
        for (int idx = t; idx < b * d; idx += kNT) {
            const int j = idx / d, c = idx % d;
            float a = 0.f;
            for (int i = j; i < b; ++i) a = fmaf(S2[i * LB + j], dZs[i * LD + c], a);
            dE2[j * LD + c] = fmaf(-es[j], a, dE2[j * LD + c]);
        }
        for (int j = t; j < b; j += kNT) {
            float s = 0.f;
            for (int i = j; i < b; ++i) s = fmaf(dA2[i * LB + j], S2[i * LB + j], s);
            des[j] += s;
        }
        // dHq += dS2 Hk, dHk += dS2^T Hq with dS2 = M . dA2 D
        for (int idx = t; idx < b * h; idx += kNT) {
            const int i = idx / h, m = idx % h;
            float aq = 0.f, ak = 0.f;
            for (int j = 0; j <= i; ++j) aq = fmaf(dA2[i * LB + j] * es[j], Hk[j * LH + m], aq);
            for (int r = i; r < b; ++r) ak = fmaf(dA2[r * LB + i] * es[i], Hq[r * LH + m], ak);
            dHq[i * LH + m] += aq;
            dHk[i * LH + m] += ak;
        }
        __syncthreads();
        // dZq = dHq . g'(Zq) (in place)
        for (int idx = t; idx < b * h; idx += kNT) {
            const int i = idx / h, m = idx % h;
            dHq[i * LH + m] *= g_prime(Zq[i * LH + m]);
        }
        __syncthreads();
        float* dZq = dHq;

        // ---- Zq = Q W1 - (M . S1 D) E1
        // dQ += dZq W1^T (sum over m of dZq[i][m] W1[k][m])
        hidden_sum(dZq, LH, b, d, h, ByCol<TI>{W1, h}, red, dQs, LD, true, 1.f);
        // dA1 = -dZq E1^T on the mask
        for (int idx = t; idx < b * b; idx += kNT) {
            const int i = idx / b, j = idx % b;
            float s = 0.f;
            if (j <= i)
                for (int m = 0; m < h; ++m) s = fmaf(dZq[i * LH + m], E1[j * LH + m], s);
            dA1[i * LB + j] = -s;
        }
        __syncthreads();
        // dE1 -= (M . S1 D)^T dZq
        for (int idx = t; idx < b * h; idx += kNT) {
            const int j = idx / h, m = idx % h;
            float a = 0.f;
            for (int i = j; i < b; ++i) a = fmaf(S1[i * LB + j], dZq[i * LH + m], a);
            dE1[j * LH + m] = fmaf(-es[j], a, dE1[j * LH + m]);
        }
        // A1: deta_j += sum_i M dA1 S1;  dQ += dS1 K;  dK += dS1^T Q   (dS1 = M . dA1 D)
        for (int j = t; j < b; j += kNT) {
            float s = 0.f;
            for (int i = j; i < b; ++i) s = fmaf(dA1[i * LB + j], S1[i * LB + j], s);
            des[j] += s;
        }
        for (int idx = t; idx < b * d; idx += kNT) {
            const int i = idx / d, k = idx % d;
            float aq = 0.f, ak = 0.f;
            for (int j = 0; j <= i; ++j) aq = fmaf(dA1[i * LB + j] * es[j], Ks[j * LD + k], aq);
            for (int r = i; r < b; ++r) ak = fmaf(dA1[r * LB + i] * es[i], Qs[r * LD + k], ak);
            dQs[i * LD + k] += aq;
            dKs[i * LD + k] += ak;
        }
        __syncthreads();

        // ---- E1 = Gk . g'(Zk):  dGk = dE1 . g'(Zk) (in place), dZk = dE1 . Gk . g''(Zk)
        for (int idx = t; idx < b * h; idx += kNT) {
            const int j = idx / h, m = idx % h;
            float gp, gpp;
            g_tanh(Zk[j * LH + m], &gp, &gpp);
            const float de1 = dE1[j * LH + m];
            dZk[j * LH + m] = de1 * Gk[j * LH + m] * gpp;
            dE1[j * LH + m] = de1 * gp;
        }
        __syncthreads();
        float* dGk = dE1;
        // dE2 += dGk W2
        hidden_sum(dGk, LH, b, d, h, ByRow<TI>{W2, d}, red, dE2, LD, true, 1.f);
        // E2: dHk += dE2 W2^T; then dZk += dHk . g'(Zk)
        if (jg < jgroups) {
            float wrow[D];
            load_row(W2 + size_t(mm) * d, wrow);
            for (int j = jg; j < b; j += jgroups) {
                float a = 0.f;
                for (int c = 0; c < d; ++c) a = fmaf(dE2[j * LD + c], wrow[c], a);
                const float dhk = dHk[j * LH + mm] + a;
                dHk[j * LH + mm] = dhk;
                dZk[j * LH + mm] = fmaf(dhk, g_prime(Zk[j * LH + mm]), dZk[j * LH + mm]);
            }
        }
        __syncthreads();
        // dK += dZk W1^T
        hidden_sum(dZk, LH, b, d, h, ByCol<TI>{W1, h}, red, dKs, LD, true, 1.f);

        // ---- outputs of the block's tokens
        for (int idx = t; idx < b * d; idx += kNT) {
            const int j = idx / d, c = idx % d;
            dQ[base + idx] = from_f32<TI>(dQs[j * LD + c]);
            dK[base + idx] = from_f32<TI>(dKs[j * LD + c]);
            dV[base + idx] = from_f32<TI>(-dE2[j * LD + c]);
        }
        for (int j = t; j < b; j += kNT) deta[bh * size_t(T) + t0 + j] = des[j];

        // ---- dW1 += Q^T dZq + K^T dZk,  dW2 += Hq^T dZ + dGk^T E2 + Hk^T dE2 (owned entries; every
        // read of dW1' / dW2' by this block's products happened before the last barrier)
        for (size_t idx = t; idx < nw; idx += kNT) {
            const int k1 = int(idx / h), m1 = int(idx % h);
            const int m2 = int(idx / d), c2 = int(idx % d);
            float a1 = 0.f, a2 = 0.f;
            for (int j = 0; j < b; ++j) {
                a1 = fmaf(Qs[j * LD + k1], dZq[j * LH + m1], a1);
                a1 = fmaf(Ks[j * LD + k1], dZk[j * LH + m1], a1);
                a2 = fmaf(Hq[j * LH + m2], dZs[j * LD + c2], a2);
                a2 = fmaf(dGk[j * LH + m2], E2[j * LD + c2], a2);
                a2 = fmaf(Hk[j * LH + m2], dE2[j * LD + c2], a2);
            }
            dW1g[idx] += a1;
            dW2g[idx] += a2;
        }
    }
}

template <typename TI, int D>
cudaError_t launch_d(const MlpBwdArgs& a, cudaStream_t s) {
    const Lay L(a.chunk, a.d, a.hidden);
    const size_t bytes = L.floats * sizeof(float);
    auto kern = mlp_backward_kernel<TI, D>;
    cudaError_t e = allow_dynamic_smem(reinterpret_cast<const void*>(kern), int(bytes));
    if (e != cudaSuccess) return e;
    kern<<<unsigned(a.B) * unsigned(a.H), kNT, bytes, s>>>(
        static_cast<const TI*>(a.Q), static_cast<const TI*>(a.K), static_cast<const TI*>(a.V), a.eta,
        static_cast<const TI*>(a.W1_hist), static_cast<const TI*>(a.W2_hist), static_cast<const TI*>(a.dZ), a.dW1_T,
        a.dW2_T, static_cast<TI*>(a.dQ), static_cast<TI*>(a.dK), static_cast<TI*>(a.dV), a.deta, a.dW1_0, a.dW2_0, a.T,
        a.hidden, a.chunk);
    return cudaGetLastError();
}

template <typename TI>
cudaError_t launch_t(const MlpBwdArgs& a, cudaStream_t s) {
    switch (a.d) {
        case 16: return launch_d<TI, 16>(a, s);
        case 32: return launch_d<TI, 32>(a, s);
        case 64: return launch_d<TI, 64>(a, s);
        default: return cudaErrorNotSupported;
    }
}

}  // namespace

bool mlp_backward_supported(int d, int hidden, int chunk) {
    if (!(d == 16 || d == 32 || d == 64) || hidden < 16 || hidden % 16 != 0 || hidden > kNT) return false;
    if (size_t(d) * hidden > 16384 || chunk < 1 || chunk > 16) return false;
    return Lay(chunk, d, hidden).floats * sizeof(float) <= 227 * 1024;
}

cudaError_t launch_mlp_backward(const MlpBwdArgs& a, cudaStream_t s) {
    if (!mlp_backward_supported(a.d, a.hidden, a.chunk)) return cudaErrorNotSupported;
    return a.bf16 ? launch_t<__nv_bfloat16>(a, s) : launch_t<float>(a, s);
}

}  // namespace ttt
