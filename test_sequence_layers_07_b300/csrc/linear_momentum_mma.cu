// linear_momentum_mma.cu -- TTT-Linear prefill with momentum for bf16 Q/K/V/Z, d = 64, chunks of 16
// tokens, fp32 state and momentum, on warp-level tensor-core MMAs.
//
// What is computed (momentum gradient descent on the TTT-Linear inner loss, the gradient of every
// token of a chunk taken at the chunk-start state; E^2-TTT article, passage on momentum and the
// closed-form chunk-end states; loss, step and read-out of "Test-Time Training Layers ...", section
// "The Core Mechanism"): with W, M the state and momentum at the chunk start, e_j = k_j W - v_j,
//   M_i = beta M_{i-1} + k_i^T e_i,   W_i = W_{i-1} - eta_i M_i,   z_i = q_i W_i.
// Closed form over a chunk of n = 16 tokens (ours), with Bs_j = eta_j + beta Bs_{j+1} (Bs_n = 0) and
// c_i = sum_{l <= i} eta_l beta^(l+1):
//   Z = Q W - diag(c) Q M - (Gamma . tril(Q K^T)) E,   Gamma_ij = Bs_j - beta^(i+1-j) Bs_{i+1}
//   W <- W - c_{n-1} M - K^T diag(Bs) E,   M <- beta^n M + K^T diag(beta^(n-1-j)) E.
//
// Design (ours): one warp per 16-column group (the recurrence is separable over output columns),
// W^T and M^T of its columns in registers in the m16n8k16 accumulator layout; read as bf16 pairs
// they are the A operand of W^T K^T and the B operand of Q W, Q M.  E^T stays in registers: scaled
// per token it is the A operand of the two rank-16 updates, unscaled the B operand of the
// correction.  Chunks run in stages of SPS: the state-independent part of a chunk (the chunk weights
// by four-step warp scans over its step sizes, and the masked, weighted scores -(Gamma . tril(Q K^T))
// as a bf16 A fragment) is formed once per CTA, each warp taking every CG-th chunk of the stage, and
// shared through shared memory; Q/K/V/eta of the next stage arrive by cp.async meanwhile.  Two CTA
// barriers per stage.
#include "ptx.cuh"
#include "ttt_common.cuh"
#include "ttt_internal.h"

namespace ttt {
namespace {

using namespace ptx;

constexpr int D = 64, KS = D / 16, NT = D / 8, TILE = 16 * D * 2;
constexpr int SPS = 4;                   // chunks per stage
constexpr int CHUNK = 3 * TILE + 64;     // Q K V [16][64] bf16, eta
constexpr int STAGE = SPS * CHUNK;
constexpr int OFF_AC = 2 * STAGE;        // per chunk of the stage: the correction's A fragment, 16 B per lane
constexpr int OFF_TW = OFF_AC + SPS * 512;  // per chunk: c[16], Bs[17], beta^k (k = 0..16)
constexpr int SMEM_BYTES = OFF_TW + SPS * 64 * 4;

// byte offset of (row, col) in a [16][64] bf16 tile (128-byte rows, 16-byte chunk XOR row % 8)
__device__ __forceinline__ uint32_t sw(int row, int col) {
    return uint32_t(row * 128 + ((((col >> 3) ^ row) & 7) << 4));
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
// the same with zeros instead of the source when `valid` is false (nothing is read from src then)
__device__ __forceinline__ void cp_async16_or_zero(uint32_t dst, const void* src, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async4_or_zero(uint32_t dst, const void* src, bool valid) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(valid ? 4 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait0() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// PART: T is not a multiple of 16 (a partial last chunk).  Its tokens past T are copied in as zeros
// (eta too), which leaves W and Z exact, and its momentum takes the chunk's own length n:
// M <- beta^n M + K^T diag(beta^(n-1-j)) E.  The instantiation for 16 | T compiles none of that.
template <int CG, bool PART>
__global__ void __launch_bounds__(32 * CG)
linear_momentum_mma_kernel(const __nv_bfloat16* __restrict__ Q, const __nv_bfloat16* __restrict__ K,
                           const __nv_bfloat16* __restrict__ V, const float* __restrict__ eta, const float* W0,
                           const float* M0, __nv_bfloat16* __restrict__ Z, float* W_out, float* M_out, int T,
                           float beta) {
    extern __shared__ __align__(128) uint8_t smem[];
    const uint32_t sb = smem_u32(smem);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
    const int lj = lane >> 3, lr = lane & 7;
    const size_t bh = blockIdx.x;
    const int cw0 = (blockIdx.y * CG + warp) * 16;  // first output column of this warp's group
    const int nblk = PART ? (T + 15) / 16 : T / 16, nstg = (nblk + SPS - 1) / SPS;
    float* tws = reinterpret_cast<float*>(smem + OFF_TW);

    auto issue = [&](int si) {
        const uint32_t b = sb + (si & 1) * STAGE;
        const int n = min(SPS, nblk - si * SPS);
        const size_t row0 = bh * size_t(T) + size_t(si) * SPS * 16;
        const int t0 = si * SPS * 16;  // first token of the stage
        if (PART && t0 + 16 * n > T) {  // the stage holds the partial last chunk: zeros past T
            for (int c = tid; c < n * 384; c += 32 * CG) {
                const int i = c / 384, r = c % 384, tile = r >> 7, row = (r >> 3) & 15, ch = r & 7;
                const __nv_bfloat16* src = tile == 0 ? Q : tile == 1 ? K : V;
                const bool in = t0 + 16 * i + row < T;
                cp_async16_or_zero(b + i * CHUNK + tile * TILE + sw(row, 8 * ch),
                                   src + (row0 + (in ? 16 * i + row : 0)) * D + 8 * ch, in);
            }
        } else {
            for (int c = tid; c < n * 384; c += 32 * CG) {
                const int i = c / 384, r = c % 384, tile = r >> 7, row = (r >> 3) & 15, ch = r & 7;
                const __nv_bfloat16* src = tile == 0 ? Q : tile == 1 ? K : V;
                cp_async16(b + i * CHUNK + tile * TILE + sw(row, 8 * ch), src + (row0 + 16 * i + row) * D + 8 * ch);
            }
        }
        if (PART && ((T & 3) || t0 + 16 * n > T)) {  // eta by 4-byte copies: unaligned, or zeros past T
            for (int c = tid; c < n * 16; c += 32 * CG) {
                const bool in = t0 + c < T;
                cp_async4_or_zero(b + (c >> 4) * CHUNK + 3 * TILE + 4 * (c & 15), eta + row0 + (in ? c : 0), in);
            }
        } else {
            for (int c = tid; c < n * 4; c += 32 * CG)
                cp_async16(b + (c >> 2) * CHUNK + 3 * TILE + 16 * (c & 3), eta + row0 + 4 * c);
        }
    };

    // ldmatrix coordinates: B with n = token, k = d (K in W^T K^T and Q K^T); A with m = token, k = d
    // (Q) and, transposed, B with k = token, n = d (K in the updates)
    uint32_t off_nk[KS], off_tk[KS];
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
        off_nk[ks] = sw(lr + 8 * (lj >> 1), 16 * ks + 8 * (lj & 1));
        off_tk[ks] = sw(lr + 8 * (lj & 1), 16 * ks + 8 * (lj >> 1));
    }
    const uint32_t off_v = sw(lr + 8 * (lj >> 1), cw0 + 8 * (lj & 1));
    const int jc[4] = {2 * t, 2 * t + 1, 8 + 2 * t, 9 + 2 * t};

    // W^T and M^T of the columns: x[nt][0..3] = X[8 nt + 2t (+1)][cw0 + g (+8)]
    float w[NT][4], m[NT][4];
    {
        const float* Wh = W0 + bh * D * D;
        const float* Mh = M0 ? M0 + bh * D * D : nullptr;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int r = 8 * nt + 2 * t;
            const size_t a0 = size_t(r) * D + cw0 + g, a1 = a0 + D;
            w[nt][0] = Wh[a0], w[nt][1] = Wh[a1], w[nt][2] = Wh[a0 + 8], w[nt][3] = Wh[a1 + 8];
            m[nt][0] = Mh ? Mh[a0] : 0.f, m[nt][1] = Mh ? Mh[a1] : 0.f;
            m[nt][2] = Mh ? Mh[a0 + 8] : 0.f, m[nt][3] = Mh ? Mh[a1 + 8] : 0.f;
        }
    }

    if (nstg > 0) issue(0);
    cp_async_commit();
    __nv_bfloat16* zb = Z + bh * size_t(T) * D + cw0 + 2 * t;
    for (int si = 0; si < nstg; ++si) {
        const int n = min(SPS, nblk - si * SPS);
        cp_async_wait0();
        __syncthreads();  // stage si has landed; every warp is done with stage si - 1 and its shared products
        if (si + 1 < nstg) issue(si + 1);
        cp_async_commit();
        const uint32_t st = sb + (si & 1) * STAGE;

        // ---- the state-independent part of each chunk, once per CTA
        for (int i = warp; i < n; i += CG) {
            const uint32_t b = st + i * CHUNK;
            const float* es = reinterpret_cast<const float*>(smem + (b - sb) + 3 * TILE);
            float* tw = tws + i * 64;
            {  // lanes 0..15 hold token k = lane: beta^(k+1), c_k, Bs_k by four-step scans
                const int k = lane & 15;
                const float ek = es[k];
                float p = beta;
#pragma unroll
                for (int o = 1; o < 16; o <<= 1) {
                    const float q = __shfl_up_sync(0xffffffffu, p, o, 16);
                    if (k >= o) p *= q;
                }
                float c = ek * p;
#pragma unroll
                for (int o = 1; o < 16; o <<= 1) {
                    const float q = __shfl_up_sync(0xffffffffu, c, o, 16);
                    if (k >= o) c += q;
                }
                float bs = ek, bo = beta;
#pragma unroll
                for (int o = 1; o < 16; o <<= 1) {
                    const float q = __shfl_down_sync(0xffffffffu, bs, o, 16);
                    if (k + o < 16) bs = fmaf(bo, q, bs);
                    bo *= bo;
                }
                const float pk = __shfl_up_sync(0xffffffffu, p, 1, 16);  // beta^k
                if (lane < 16) {
                    tw[k] = c;
                    tw[16 + k] = bs;
                    tw[33 + k] = k == 0 ? 1.f : pk;
                }
                if (lane == 15) {
                    tw[32] = 0.f;  // Bs_16
                    tw[49] = p;    // beta^16
                }
                __syncwarp();
            }
            // S = Q K^T, then the correction's A fragment -(Gamma . tril(S))
            float sa[2][4];
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                uint32_t kb[4], qa[4];
                ldsm_x4(b + TILE + off_nk[ks], kb);
                ldsm_x4(b + off_tk[ks], qa);
                if (ks == 0) {
                    mma_bf16_16816_z(sa[0], qa, kb[0], kb[1]);
                    mma_bf16_16816_z(sa[1], qa, kb[2], kb[3]);
                } else {
                    mma_bf16_16816(sa[0], qa, kb[0], kb[1]);
                    mma_bf16_16816(sa[1], qa, kb[2], kb[3]);
                }
            }
            uint32_t ac[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {  // register q: rows i = g + 8 (q & 1), cols j = 8 (q >> 1) + 2t (+1)
                float v[2];
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int r = g + 8 * (q & 1), j = 8 * (q >> 1) + 2 * t + u;
                    const float s = sa[q >> 1][2 * (q & 1) + u];
                    v[u] = j <= r ? -(tw[16 + j] - tw[33 + r + 1 - j] * tw[16 + r + 1]) * s : 0.f;
                }
                ac[q] = pack_bf16(v[0], v[1]);
            }
            *reinterpret_cast<uint4*>(smem + OFF_AC + i * 512 + lane * 16) = make_uint4(ac[0], ac[1], ac[2], ac[3]);
        }
        __syncthreads();  // every chunk's weights and correction fragment are written

        // ---- the chain: one chunk at a time through this warp's state; a full stage is unrolled, so
        // the compiler can load the next chunk's fragments while this chunk's products are in flight
        auto chunk = [&](const int i) {
            const uint32_t b = st + i * CHUNK;
            const float* tw = tws + i * 64;
            uint32_t kb[KS][4], qa[KS][4], kt[KS][4], vv[4];
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                ldsm_x4(b + TILE + off_nk[ks], kb[ks]);
                ldsm_x4(b + off_tk[ks], qa[ks]);
                ldsm_x4_trans(b + TILE + off_tk[ks], kt[ks]);
            }
            ldsm_x4_trans(b + 2 * TILE + off_v, vv);
            uint32_t wa[KS][4], ma[KS][4];
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                wa[ks][0] = pack_bf16(w[2 * ks][0], w[2 * ks][1]);
                wa[ks][1] = pack_bf16(w[2 * ks][2], w[2 * ks][3]);
                wa[ks][2] = pack_bf16(w[2 * ks + 1][0], w[2 * ks + 1][1]);
                wa[ks][3] = pack_bf16(w[2 * ks + 1][2], w[2 * ks + 1][3]);
                ma[ks][0] = pack_bf16(m[2 * ks][0], m[2 * ks][1]);
                ma[ks][1] = pack_bf16(m[2 * ks][2], m[2 * ks][3]);
                ma[ks][2] = pack_bf16(m[2 * ks + 1][0], m[2 * ks + 1][1]);
                ma[ks][3] = pack_bf16(m[2 * ks + 1][2], m[2 * ks + 1][3]);
            }
            // P^T = W^T K^T (columns x tokens) at the chunk-start state; Q W and Q M
            float pa[2][2][4], za[2][4], zm[2][4];
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                if (ks < 2) {
                    mma_bf16_16816_z(pa[ks][0], wa[ks], kb[ks][0], kb[ks][1]);
                    mma_bf16_16816_z(pa[ks][1], wa[ks], kb[ks][2], kb[ks][3]);
                } else {
                    mma_bf16_16816(pa[ks & 1][0], wa[ks], kb[ks][0], kb[ks][1]);
                    mma_bf16_16816(pa[ks & 1][1], wa[ks], kb[ks][2], kb[ks][3]);
                }
                if (ks == 0) {
                    mma_bf16_16816_z(za[0], qa[0], wa[0][0], wa[0][2]);
                    mma_bf16_16816_z(za[1], qa[0], wa[0][1], wa[0][3]);
                    mma_bf16_16816_z(zm[0], qa[0], ma[0][0], ma[0][2]);
                    mma_bf16_16816_z(zm[1], qa[0], ma[0][1], ma[0][3]);
                } else {
                    mma_bf16_16816(za[0], qa[ks], wa[ks][0], wa[ks][2]);
                    mma_bf16_16816(za[1], qa[ks], wa[ks][1], wa[ks][3]);
                    mma_bf16_16816(zm[0], qa[ks], ma[ks][0], ma[ks][2]);
                    mma_bf16_16816(zm[1], qa[ks], ma[ks][1], ma[ks][3]);
                }
            }
            // E^T = P^T - V^T: e[h][0..3] = (c = g, j), (g, j + 1), (g + 8, j), (g + 8, j + 1), j = 8 h + 2t
            float e[2][4];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                e[h][0] = (pa[0][h][0] + pa[1][h][0]) - bf16_lo(vv[2 * h]);
                e[h][1] = (pa[0][h][1] + pa[1][h][1]) - bf16_hi(vv[2 * h]);
                e[h][2] = (pa[0][h][2] + pa[1][h][2]) - bf16_lo(vv[2 * h + 1]);
                e[h][3] = (pa[0][h][3] + pa[1][h][3]) - bf16_hi(vv[2 * h + 1]);
            }
            // read-out Z = Q W - diag(c) Q M - (Gamma . tril(S)) E
            {
                const uint4 a4 = *reinterpret_cast<const uint4*>(smem + OFF_AC + i * 512 + lane * 16);
                const uint32_t ac[4] = {a4.x, a4.y, a4.z, a4.w};
                const uint32_t ea[4] = {pack_bf16(e[0][0], e[0][1]), pack_bf16(e[0][2], e[0][3]),
                                        pack_bf16(e[1][0], e[1][1]), pack_bf16(e[1][2], e[1][3])};
                const float cg0 = tw[g], cg8 = tw[g + 8];
                float zp[2][4];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    zp[h][0] = fmaf(-cg0, zm[h][0], za[h][0]);
                    zp[h][1] = fmaf(-cg0, zm[h][1], za[h][1]);
                    zp[h][2] = fmaf(-cg8, zm[h][2], za[h][2]);
                    zp[h][3] = fmaf(-cg8, zm[h][3], za[h][3]);
                }
                mma_bf16_16816(zp[0], ac, ea[0], ea[2]);
                mma_bf16_16816(zp[1], ac, ea[1], ea[3]);
                __nv_bfloat16* zr = zb + size_t(16 * (si * SPS + i) + g) * D;  // rows g (+8), columns cw0 + 2t (+8)
                const bool lo = !PART || 16 * (si * SPS + i) + g < T, hi = !PART || 16 * (si * SPS + i) + g + 8 < T;
                if (lo) *reinterpret_cast<uint32_t*>(zr) = pack_bf16(zp[0][0], zp[0][1]);
                if (hi) *reinterpret_cast<uint32_t*>(zr + 8 * D) = pack_bf16(zp[0][2], zp[0][3]);
                if (lo) *reinterpret_cast<uint32_t*>(zr + 8) = pack_bf16(zp[1][0], zp[1][1]);
                if (hi) *reinterpret_cast<uint32_t*>(zr + 8 * D + 8) = pack_bf16(zp[1][2], zp[1][3]);
            }
            // W^T <- W^T - c_15 M^T - E^T diag(Bs) K;  M^T <- beta^n M^T + E^T diag(beta^(n-1-j)) K, n the
            // chunk's tokens (16 but for a partial last chunk, whose E is zero past n)
            {
                const int ntok = PART ? min(16, T - 16 * (si * SPS + i)) : 16;
                float bsj[4], pj[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    bsj[q] = tw[16 + jc[q]];
                    pj[q] = PART ? (jc[q] < ntok ? tw[33 + ntok - 1 - jc[q]] : 0.f) : tw[33 + 15 - jc[q]];
                }
                const uint32_t gw[4] = {pack_bf16(-bsj[0] * e[0][0], -bsj[1] * e[0][1]),
                                        pack_bf16(-bsj[0] * e[0][2], -bsj[1] * e[0][3]),
                                        pack_bf16(-bsj[2] * e[1][0], -bsj[3] * e[1][1]),
                                        pack_bf16(-bsj[2] * e[1][2], -bsj[3] * e[1][3])};
                const uint32_t gm[4] = {pack_bf16(pj[0] * e[0][0], pj[1] * e[0][1]),
                                        pack_bf16(pj[0] * e[0][2], pj[1] * e[0][3]),
                                        pack_bf16(pj[2] * e[1][0], pj[3] * e[1][1]),
                                        pack_bf16(pj[2] * e[1][2], pj[3] * e[1][3])};
                const float c15 = tw[15], b16 = PART ? tw[33 + ntok] : tw[49];  // beta^n
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        w[nt][r] = fmaf(-c15, m[nt][r], w[nt][r]);
                        m[nt][r] *= b16;
                    }
#pragma unroll
                for (int kk = 0; kk < KS; ++kk) {
                    mma_bf16_16816(w[2 * kk], gw, kt[kk][0], kt[kk][1]);
                    mma_bf16_16816(w[2 * kk + 1], gw, kt[kk][2], kt[kk][3]);
                    mma_bf16_16816(m[2 * kk], gm, kt[kk][0], kt[kk][1]);
                    mma_bf16_16816(m[2 * kk + 1], gm, kt[kk][2], kt[kk][3]);
                }
            }
        };
        if (n == SPS) {
#pragma unroll
            for (int i = 0; i < SPS; ++i) chunk(i);
        } else {
            for (int i = 0; i < n; ++i) chunk(i);
        }
    }
    cp_async_wait0();
    float* Wo = W_out + bh * D * D;
    float* Mo = M_out + bh * D * D;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int r = 8 * nt + 2 * t;
        const size_t a0 = size_t(r) * D + cw0 + g, a1 = a0 + D;
        Wo[a0] = w[nt][0], Wo[a1] = w[nt][1], Wo[a0 + 8] = w[nt][2], Wo[a1 + 8] = w[nt][3];
        Mo[a0] = m[nt][0], Mo[a1] = m[nt][1], Mo[a0 + 8] = m[nt][2], Mo[a1 + 8] = m[nt][3];
    }
}

template <int CG, bool PART>
cudaError_t launch_part(const LinearArgs& a, cudaStream_t s) {
    auto kern = linear_momentum_mma_kernel<CG, PART>;
    cudaError_t e = allow_dynamic_smem(reinterpret_cast<const void*>(kern), SMEM_BYTES);
    if (e != cudaSuccess) return e;
    kern<<<dim3(unsigned(a.B) * unsigned(a.H), 4 / CG), 32 * CG, SMEM_BYTES, s>>>(
        static_cast<const __nv_bfloat16*>(a.Q), static_cast<const __nv_bfloat16*>(a.K),
        static_cast<const __nv_bfloat16*>(a.V), a.eta, a.W0, a.M0, static_cast<__nv_bfloat16*>(a.Z), a.W_out,
        a.M_out, a.T, a.beta);
    return cudaGetLastError();
}

template <int CG>
cudaError_t launch_cg(const LinearArgs& a, cudaStream_t s) {
    return a.T % 16 ? launch_part<CG, true>(a, s) : launch_part<CG, false>(a, s);
}

}  // namespace

bool linear_momentum_mma_supported(const LinearArgs& a) {
    return a.momentum && a.bf16 && a.d == D && a.chunk == 16;  // any T
}

cudaError_t launch_linear_momentum_mma(const LinearArgs& a, cudaStream_t s) {
    if (!linear_momentum_mma_supported(a)) return cudaErrorNotSupported;
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    // four column groups per CTA (one CTA per head) unless that leaves most SMs idle
    const long long bh = (long long)a.B * a.H;
    if (bh * 2 > sms) return launch_cg<4>(a, s);
    if (bh * 4 > sms) return launch_cg<2>(a, s);
    return launch_cg<1>(a, s);
}

}  // namespace ttt
