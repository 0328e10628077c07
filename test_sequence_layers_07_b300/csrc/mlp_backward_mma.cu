// mlp_backward_mma.cu -- gradient of the TTT-MLP chunked scan for bf16, d = 64, hidden = 256, blocks
// of 16 tokens, on warp-level tensor-core MMAs (fp32 accumulation).
//
// What is computed is the chain rule through the block form of the scan ("Test-Time Training (TTT)
// Layers for Sequence Modeling", section "Variants: TTT-Linear vs. TTT-MLP"; loss, step and read-out
// of "Test-Time Training Layers ...", section "The Core Mechanism"; outer-loop training through the
// inner loop as in the TTT essay's paragraph on the two time scales).  Per block, with start state
// (W1, W2), D = diag(eta), M the causal mask (j <= i), g the tanh-form GELU:
//   Zk = K W1, Hk = g(Zk), E2 = Hk W2 - V, Gk = E2 W2^T, E1 = Gk . g'(Zk),
//   Zq = Q W1 - (M . Q K^T) D E1, Hq = g(Zq), Z = Hq W2 - (M . Hq Hk^T) D E2,
//   W1' = W1 - K^T D E1, W2' = W2 - Hk^T D E2,
// and, given the gradients dW1', dW2' of the state after the block and dZ:
//   dHk = -D E2 dW2'^T + dS2^T Hq + dE2 W2^T      dE1 = -D K dW1' - (M . S1 D)^T dZq
//   dHq = dZ W2^T + dS2 Hk, dZq = dHq . g'(Zq)    dGk = dE1 . g'(Zk)
//   dZk = dE1 . Gk . g''(Zk) + dHk . g'(Zk)
//   dE2 = -D Hk dW2' - (M . S2 D)^T dZ + dGk W2    dV = -dE2
//   dQ = dZq W1^T + dS1 K,  dK = -D E1 dW1'^T + dS1^T Q + dZk W1^T
//   (S1 = Q K^T, S2 = Hq Hk^T, dA1 = -dZq E1^T, dA2 = -dZ E2^T, dS = M . dA D)
//   deta_j = -(K dW1')_j . E1_j - (Hk dW2')_j . E2_j + sum_i M (dA2 . S2)_ij + sum_i M (dA1 . S1)_ij
//   dW1 = dW1' + Q^T dZq + K^T dZk,   dW2 = dW2' + Hq^T dZ + dGk^T E2 + Hk^T dE2
// The block-start states come from the forward (ttt_mlp_prefill_hist), recorded in bf16.
//
// Design (ours, for sm_103a):
//  * One CTA of NW warps per (batch, head) (eight by default; sixteen can be chosen), blocks in
//    reverse order.  Warp w owns hidden units [HS w, HS w + HS), HS = 256 / NW: every b x hidden
//    quantity (Zk, Hk, Gk, E1, Zq, Hq, dHk, dHq, dE1, dZk, ...) lives in its registers as the MMA
//    accumulator slice 16 x HS, so the element-wise steps (GELU and its derivatives, the products
//    with g') need no shared memory.  An accumulator slice read
//    as bf16 pairs is the A fragment of the slice over its hidden columns and the B fragment of its
//    transpose; the B fragment over tokens and the A fragment of the transpose come from movmatrix.
//  * Products over d (K W1, Q W1, E2 W2^T, dZ W2^T, K dW1', E2 dW2'^T, dE2 W2^T) take their B
//    operands from the warp's own slices of W1, W2 (the recorded state of the block) and of the bf16
//    copy of dW1', dW2', all in warp-private shared memory: no barrier guards them.
//  * Products over the hidden dimension (E2, Hq Hk^T, dZq W1^T, dZq E1^T, the dE2 and dK sums) are
//    partial per warp and summed in a fixed order through shared memory: five reductions a block,
//    two barriers each (three with sixteen warps, whose partials pair up first).  Small
//    token-by-token products (the masked score terms) run one 8-column tile per warp (warps 0-7).
//  * The running state gradient (fp32) lives in dW1_0 / dW2_0 (L2-resident): each warp reads its
//    slices as accumulator fragments, adds the block's rank-16 terms by MMA, writes them back and
//    refreshes its bf16 copy.
//  * Token tiles are double buffered by cp.async one block ahead; the next block's state slices are
//    prefetched to L2 a block ahead and copied in right after their last use.
#include <stdlib.h>
#include <string.h>

#include "ptx.cuh"
#include "ttt_common.cuh"
#include "ttt_internal.h"

namespace ttt {
namespace {

using namespace ptx;

constexpr int D = 64, HID = 256, BT = 16;
constexpr int TILE = BT * D * 2;       // [16][64] bf16 token tile
constexpr int TOKBUF = 4 * TILE + 64;  // Q K V dZ, eta

// NW warps, each owning HS = 256 / NW hidden units (NJ 8-wide n-tiles, NKH 16-wide k-steps of them).
// The per-warp partials of a sum over the hidden dimension go through 8 slots: with 16 warps, warp
// w + 8 hands its partial to warp w first (two-stage, fixed order).
template <int NW_>
struct BwdCfg {
    static constexpr int NW = NW_, NTH = 32 * NW, HS = HID / NW, NJ = HS / 8, NKH = HS / 16;
    static constexpr int SZ_W1S = 64 * HS * 2;  // a warp's [64][HS] slice of W1 (or dW1'), bf16
    static constexpr int SZ_W2S = HS * 64 * 2;  // a warp's [HS][64] slice of W2 (or dW2'), bf16
    // shared memory (bytes)
    static constexpr int OFF_W1 = 0;
    static constexpr int OFF_W2 = OFF_W1 + NW * SZ_W1S;
    static constexpr int OFF_G1 = OFF_W2 + NW * SZ_W2S;   // bf16 dW1' slices
    static constexpr int OFF_G2 = OFF_G1 + NW * SZ_W1S;   // bf16 dW2' slices
    static constexpr int OFF_TOK = OFF_G2 + NW * SZ_W2S;  // two token buffers
    static constexpr int OFF_E2B = OFF_TOK + 2 * TOKBUF;  // E2, bf16 [16][64]
    static constexpr int OFF_DE2B = OFF_E2B + TILE;       // dE2, bf16 [16][64]
    static constexpr int OFF_PART = OFF_DE2B + TILE;      // 16 x 64 partials [8][8 n-tiles][32 lanes] float4
    static constexpr int OFF_PSM = OFF_PART + 8 * 4096;   // 16 x 16 partials [8][2][32] float4
    static constexpr int OFF_E2F = OFF_PSM + 8 * 1024;    // E2 fp32, fragment order [8][32] float4
    static constexpr int OFF_DE2T = OFF_E2F + 4096;       // -(M . S2 D)^T dZ, fragment order
    static constexpr int OFF_DQ = OFF_DE2T + 4096;        // dQ, fragment order
    static constexpr int OFF_DKT = OFF_DQ + 4096;         // dS1^T Q, fragment order
    static constexpr int OFF_S2 = OFF_DKT + 4096;         // S2 fp32 [16][16]
    static constexpr int OFF_DA1 = OFF_S2 + 1024;         // dA1 fp32 [16][16]
    static constexpr int OFF_DETA = OFF_DA1 + 1024;       // [NW warps][16] partials, then [16] score terms
    static constexpr int SMEM_BYTES = OFF_DETA + (NW + 1) * 64;
    static_assert(SMEM_BYTES <= 232448, "shared memory");
};

// byte offset of (row, col) in a [rows][64] bf16 block (128-byte rows, 16-byte chunk XOR row % 8)
__device__ __forceinline__ uint32_t t64(int row, int col) {
    return uint32_t(row * 128 + ((((col >> 3) ^ row) & 7) << 4) + (col & 7) * 2);
}
// byte offset of (row, col) in a [rows][32] bf16 block (64-byte rows, chunk XOR (row / 2) % 4) or a
// [rows][16] one (32-byte rows, chunk XOR (row / 4) % 2): the eight rows an ldmatrix reads at one chunk
// fall in distinct banks
__device__ __forceinline__ uint32_t t32(int row, int col) {
    return uint32_t(row * 64 + ((((col >> 3) ^ (row >> 1)) & 3) << 4) + (col & 7) * 2);
}
__device__ __forceinline__ uint32_t t16(int row, int col) {
    return uint32_t(row * 32 + ((((col >> 3) ^ (row >> 2)) & 1) << 4) + (col & 7) * 2);
}
// the layout of a warp's [64][HS] slice of W1 or dW1' (RB = 0: a [rows][64] block)
template <int RB>
__device__ __forceinline__ uint32_t tl(int row, int col) {
    return RB == 32 ? t32(row, col) : RB == 16 ? t16(row, col) : t64(row, col);
}

__device__ __forceinline__ uint32_t movt(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}
__device__ __forceinline__ void ldsm_x2_trans(uint32_t addr, uint32_t& r0, uint32_t& r1) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0, %1}, [%2];"
                 : "=r"(r0), "=r"(r1)
                 : "r"(addr)
                 : "memory");
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
__device__ __forceinline__ void cp_async_wait1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait0() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void prefetch_l2(const void* p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// ---- GELU (tanh form) and its first two derivatives
__device__ __forceinline__ float tanh_fast(float x) {
    float y;
    asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
struct Gelu {
    float g, gp, gpp;
};
__device__ __forceinline__ Gelu gelu3(float x) {
    const float c = 0.7978845608028654f, a = 0.044715f;
    const float t = tanh_fast(c * fmaf(a * x, x * x, x));
    const float u1 = c * fmaf(3.f * a, x * x, 1.f), s = 1.f - t * t;
    Gelu r;
    r.g = 0.5f * x * (1.f + t);
    r.gp = 0.5f * (1.f + t) + 0.5f * x * s * u1;
    r.gpp = s * u1 + 0.5f * x * s * (6.f * a * c * x - 2.f * t * u1 * u1);
    return r;
}

// ---- fragment loads (lane l gives the row address of row l % 8 of matrix l / 8)
// A of a [16][64] token tile, k-step kk (columns 16 kk ..)
__device__ __forceinline__ void lda_tok(uint32_t tile, int kk, int lane, uint32_t (&a)[4]) {
    const int q = lane >> 3, r = lane & 7;
    ldsm_x4(tile + t64(r + 8 * (q & 1), 16 * kk + 8 * (q >> 1)), a);
}
// B of two n-tiles (n0, n0 + 8), k-step at k0, from [n][k] storage: b[0..1] for n0, b[2..3] for n0 + 8
template <int RB>
__device__ __forceinline__ void ldb_nk(uint32_t base, int n0, int k0, int lane, uint32_t (&b)[4]) {
    const int q = lane >> 3, r = lane & 7, row = n0 + 8 * (q >> 1) + r, col = k0 + 8 * (q & 1);
    ldsm_x4(base + tl<RB>(row, col), b);
}
// the same from [k][n] storage (transposing load)
template <int RB>
__device__ __forceinline__ void ldb_kn(uint32_t base, int n0, int k0, int lane, uint32_t (&b)[4]) {
    const int q = lane >> 3, r = lane & 7, row = k0 + 8 * (q & 1) + r, col = n0 + 8 * (q >> 1);
    ldsm_x4_trans(base + tl<RB>(row, col), b);
}
// B of one n-tile n0 over the 16 tokens of a [16][64] token tile ([k][n] storage)
__device__ __forceinline__ void ldb_tok1(uint32_t tile, int n0, int lane, uint32_t& b0, uint32_t& b1) {
    const int r = lane & 7, q = (lane >> 3) & 1;
    ldsm_x2_trans(tile + t64(r + 8 * q, n0), b0, b1);
}
// A of the transpose of a [16][64] token tile: m-tile at m0 (columns of the tile), k = the 16 tokens
__device__ __forceinline__ void lda_tokT(uint32_t tile, int m0, int lane, uint32_t (&a)[4]) {
    const int q = lane >> 3, r = lane & 7;
    ldsm_x4_trans(tile + t64(r + 8 * (q >> 1), m0 + 8 * (q & 1)), a);
}

// ---- register slices: X[NJ][4] is a 16 x 8 NJ accumulator slice (n-tile j = columns 8 j ..)
// packed A fragments over its columns, k-step kk = columns 16 kk ..
template <int NJ>
__device__ __forceinline__ void pack_slice(const float (&x)[NJ][4], uint32_t (&xa)[NJ / 2][4]) {
#pragma unroll
    for (int kk = 0; kk < NJ / 2; ++kk) {
        xa[kk][0] = pack_bf16(x[2 * kk][0], x[2 * kk][1]);
        xa[kk][1] = pack_bf16(x[2 * kk][2], x[2 * kk][3]);
        xa[kk][2] = pack_bf16(x[2 * kk + 1][0], x[2 * kk + 1][1]);
        xa[kk][3] = pack_bf16(x[2 * kk + 1][2], x[2 * kk + 1][3]);
    }
}
// the slice as the B operand over tokens (k = token, n = column tile j)
template <int NKH>
__device__ __forceinline__ void btok(const uint32_t (&xa)[NKH][4], int j, uint32_t& b0, uint32_t& b1) {
    b0 = movt(xa[j >> 1][(j & 1) * 2]);
    b1 = movt(xa[j >> 1][(j & 1) * 2 + 1]);
}
// the transposed slice as an A operand: m-tile p = columns 16 p .., k = the 16 tokens
template <int NKH>
__device__ __forceinline__ void atr(const uint32_t (&xa)[NKH][4], int p, uint32_t (&a)[4]) {
    a[0] = movt(xa[p][0]);
    a[1] = movt(xa[p][2]);
    a[2] = movt(xa[p][1]);
    a[3] = movt(xa[p][3]);
}

__device__ __forceinline__ void scale_rows(float (&x)[4], float sg, float sg8) {
    x[0] *= sg, x[1] *= sg, x[2] *= sg8, x[3] *= sg8;
}

// PART: T is not a multiple of 16 (a partial last block, the first processed): its tokens past T
// are copied in as zeros (eta too), so they add nothing to any gradient, and no output row past T is
// stored; the instantiation for 16 | T compiles none of that.
template <int NW_, bool PART>
__global__ void __launch_bounds__(32 * NW_, 1)
mlp_backward_mma_kernel(const __nv_bfloat16* __restrict__ Q, const __nv_bfloat16* __restrict__ K,
                        const __nv_bfloat16* __restrict__ V, const float* __restrict__ eta,
                        const __nv_bfloat16* __restrict__ W1h, const __nv_bfloat16* __restrict__ W2h,
                        const __nv_bfloat16* __restrict__ dZ, const float* dW1_T, const float* dW2_T,
                        __nv_bfloat16* __restrict__ dQ, __nv_bfloat16* __restrict__ dK,
                        __nv_bfloat16* __restrict__ dV, float* __restrict__ deta, float* dW1g, float* dW2g, int T) {
    using C = BwdCfg<NW_>;
    constexpr int NW = C::NW, NTH = C::NTH, HS = C::HS, NJ = C::NJ, NKH = C::NKH;
    constexpr int SZ_W1S = C::SZ_W1S, SZ_W2S = C::SZ_W2S, OFF_W1 = C::OFF_W1, OFF_W2 = C::OFF_W2;
    constexpr int OFF_G1 = C::OFF_G1, OFF_G2 = C::OFF_G2, OFF_TOK = C::OFF_TOK, OFF_E2B = C::OFF_E2B;
    constexpr int OFF_DE2B = C::OFF_DE2B, OFF_PART = C::OFF_PART, OFF_PSM = C::OFF_PSM, OFF_E2F = C::OFF_E2F;
    constexpr int OFF_DE2T = C::OFF_DE2T, OFF_DQ = C::OFF_DQ, OFF_DKT = C::OFF_DKT, OFF_S2 = C::OFF_S2;
    constexpr int OFF_DA1 = C::OFF_DA1, OFF_DETA = C::OFF_DETA;
    extern __shared__ __align__(128) uint8_t smem[];
    const uint32_t sb = smem_u32(smem);
    const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
    const size_t bh = blockIdx.x;
    const int nblk = PART ? (T + BT - 1) / BT : T / BT;
    constexpr size_t NWT = size_t(D) * HID;
    dW1g += bh * NWT;
    dW2g += bh * NWT;
    const uint32_t w1s = sb + OFF_W1 + w * SZ_W1S, w2s = sb + OFF_W2 + w * SZ_W2S;
    const uint32_t g1s = sb + OFF_G1 + w * SZ_W1S, g2s = sb + OFF_G2 + w * SZ_W2S;
    float* part = reinterpret_cast<float*>(smem + OFF_PART);
    float* psm = reinterpret_cast<float*>(smem + OFF_PSM);
    float* e2f = reinterpret_cast<float*>(smem + OFF_E2F);
    float* de2t = reinterpret_cast<float*>(smem + OFF_DE2T);
    float* dqf = reinterpret_cast<float*>(smem + OFF_DQ);
    float* dkt = reinterpret_cast<float*>(smem + OFF_DKT);
    float* s2s = reinterpret_cast<float*>(smem + OFF_S2);
    float* da1s = reinterpret_cast<float*>(smem + OFF_DA1);
    float* detap = reinterpret_cast<float*>(smem + OFF_DETA);  // [NW][16]
    float* detac = detap + NW * 16;                             // [16]
    const int hw = HS * w;  // first hidden unit of this warp
    // this warp's partial of a 16 x 64 (or 16 x 16) sum over the hidden dimension into its slot of
    // `buf` (nt n-tiles x 32 lanes x float4); with 16 warps, warp w + 8 hands its partial to warp w,
    // which adds its own (one more barrier).  The caller's barrier then covers the slots.
    auto put_partial = [&](float* buf, const auto& P) {
        constexpr int ntiles = sizeof(P) / sizeof(P[0]);
        if (NW == 16 && w >= 8) {
#pragma unroll
            for (int nt = 0; nt < ntiles; ++nt)
                *reinterpret_cast<float4*>(buf + (((w - 8) * ntiles + nt) * 32 + lane) * 4) =
                    make_float4(P[nt][0], P[nt][1], P[nt][2], P[nt][3]);
        }
        if (NW == 16) __syncthreads();
        if (w < 8) {
#pragma unroll
            for (int nt = 0; nt < ntiles; ++nt) {
                float4* d = reinterpret_cast<float4*>(buf + ((w * ntiles + nt) * 32 + lane) * 4);
                float4 v = make_float4(P[nt][0], P[nt][1], P[nt][2], P[nt][3]);
                if (NW == 16) {
                    const float4 o = *d;
                    v.x += o.x, v.y += o.y, v.z += o.z, v.w += o.w;
                }
                *d = v;
            }
        }
    };

    auto issue_tokens = [&](int m) {
        const uint32_t tb = sb + OFF_TOK + (m & 1) * TOKBUF;
        const size_t row0 = bh * size_t(T) + size_t(m) * BT;
        if (PART && BT * (m + 1) > T) {  // the partial last block: zeros past T, eta by 4-byte copies
#pragma unroll
            for (int c = tid; c < 4 * 128; c += NTH) {
                const int tile = c >> 7, row = (c >> 3) & 15, ch = c & 7;
                const __nv_bfloat16* src = tile == 0 ? Q : tile == 1 ? K : tile == 2 ? V : dZ;
                const bool in = BT * m + row < T;
                cp_async16_or_zero(tb + tile * TILE + t64(row, 8 * ch), src + (row0 + (in ? row : 0)) * D + 8 * ch, in);
            }
            if (tid < BT) cp_async4_or_zero(tb + 4 * TILE + 4 * tid, eta + row0 + (BT * m + tid < T ? tid : 0), BT * m + tid < T);
            return;
        }
#pragma unroll
        for (int c = tid; c < 4 * 128; c += NTH) {
            const int tile = c >> 7, row = (c >> 3) & 15, ch = c & 7;
            const __nv_bfloat16* src = tile == 0 ? Q : tile == 1 ? K : tile == 2 ? V : dZ;
            cp_async16(tb + tile * TILE + t64(row, 8 * ch), src + (row0 + row) * D + 8 * ch);
        }
        if (PART && (T & 3)) {  // a head's eta not 16-byte aligned: 4-byte copies
            if (tid < BT) cp_async4_or_zero(tb + 4 * TILE + 4 * tid, eta + row0 + tid, true);
        } else if (tid < 4) {
            cp_async16(tb + 4 * TILE + 16 * tid, eta + row0 + 4 * tid);
        }
    };
    auto issue_state = [&](int m) {  // this warp's slices of the block-start state of block m
        const __nv_bfloat16* s1 = W1h + (bh * nblk + m) * NWT;
        const __nv_bfloat16* s2 = W2h + (bh * nblk + m) * NWT;
#pragma unroll
        for (int c = lane; c < 64 * (HS / 8); c += 32) {
            const int r1 = c / (HS / 8), c1 = c % (HS / 8);
            cp_async16(w1s + tl<HS>(r1, 8 * c1), s1 + size_t(r1) * HID + hw + 8 * c1);
        }
#pragma unroll
        for (int c = lane; c < HS * 8; c += 32) {
            const int r2 = c >> 3, c2 = c & 7;
            cp_async16(w2s + t64(r2, 8 * c2), s2 + size_t(hw + r2) * D + 8 * c2);
        }
    };
    auto prefetch_state = [&](int m) {
        const __nv_bfloat16* s1 = W1h + (bh * nblk + m) * NWT;
        const __nv_bfloat16* s2 = W2h + (bh * nblk + m) * NWT;
        prefetch_l2(s1 + size_t(lane) * HID + hw);
        prefetch_l2(s1 + size_t(lane + 32) * HID + hw);
        if (lane < HS) prefetch_l2(s2 + size_t(hw + lane) * D);
    };

    // ---- the running state gradient starts at dW_T (zero when absent); dW_T may be dW_0 itself
    {
#pragma unroll
        for (int mt = 0; mt < 4; ++mt)
#pragma unroll
            for (int j = 0; j < NJ; ++j)
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2) {
                    const int row = 16 * mt + g + 8 * h2, col = 8 * j + 2 * t;
                    const size_t at = size_t(row) * HID + hw + col;
                    float2 v = dW1_T ? *reinterpret_cast<const float2*>(dW1_T + bh * NWT + at) : make_float2(0.f, 0.f);
                    *reinterpret_cast<float2*>(dW1g + at) = v;
                    *reinterpret_cast<uint32_t*>(smem + OFF_G1 + w * SZ_W1S + tl<HS>(row, col)) = pack_bf16(v.x, v.y);
                }
#pragma unroll
        for (int p = 0; p < NKH; ++p)
#pragma unroll
            for (int nt = 0; nt < 8; ++nt)
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2) {
                    const int row = 16 * p + g + 8 * h2, col = 8 * nt + 2 * t;
                    const size_t at = size_t(hw + row) * D + col;
                    float2 v = dW2_T ? *reinterpret_cast<const float2*>(dW2_T + bh * NWT + at) : make_float2(0.f, 0.f);
                    *reinterpret_cast<float2*>(dW2g + at) = v;
                    *reinterpret_cast<uint32_t*>(smem + OFF_G2 + w * SZ_W2S + t64(row, col)) = pack_bf16(v.x, v.y);
                }
    }
    if (nblk > 0) {
        issue_tokens(nblk - 1);
        cp_async_commit();
        issue_state(nblk - 1);
        cp_async_commit();
    }

    for (int n = nblk - 1; n >= 0; --n) {
        if (n >= 1) {
            issue_tokens(n - 1);
            prefetch_state(n - 1);
        }
        cp_async_commit();
        cp_async_wait1();  // this block's tokens and state slices have landed (this thread's copies)
        __syncthreads();   // everyone's have; the previous block's outputs are written
        const uint32_t tb = sb + OFF_TOK + (n & 1) * TOKBUF;
        const uint32_t Qs = tb, Ks = tb + TILE, Vs = tb + 2 * TILE, dZs = tb + 3 * TILE;
        const float* es = reinterpret_cast<const float*>(smem + OFF_TOK + (n & 1) * TOKBUF + 4 * TILE);
        const float eg = es[g], eg8 = es[g + 8];
        const float ec[4] = {es[2 * t], es[2 * t + 1], es[8 + 2 * t], es[9 + 2 * t]};  // columns of the A layout
        const int colj[4] = {2 * t, 2 * t + 1, 8 + 2 * t, 9 + 2 * t};
        const size_t orow = bh * size_t(T) + size_t(n) * BT;

        // ================= F1: Zk = K W1, Zq = Q W1, S1 = Q K^T, E2 partial = Hk W2 (this warp's slice)
        float Zk[NJ][4], Zq[NJ][4], S1[2][4];
        {
            uint32_t aK[4][4], aQ[4][4];
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                lda_tok(Ks, kk, lane, aK[kk]);
                lda_tok(Qs, kk, lane, aQ[kk]);
            }
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
#pragma unroll
                for (int jp = 0; jp < NJ / 2; ++jp) {
                    uint32_t b[4];
                    ldb_kn<HS>(w1s, 16 * jp, 16 * kk, lane, b);
                    if (kk == 0) {
                        mma_bf16_16816_z(Zk[2 * jp], aK[kk], b[0], b[1]);
                        mma_bf16_16816_z(Zk[2 * jp + 1], aK[kk], b[2], b[3]);
                        mma_bf16_16816_z(Zq[2 * jp], aQ[kk], b[0], b[1]);
                        mma_bf16_16816_z(Zq[2 * jp + 1], aQ[kk], b[2], b[3]);
                    } else {
                        mma_bf16_16816(Zk[2 * jp], aK[kk], b[0], b[1]);
                        mma_bf16_16816(Zk[2 * jp + 1], aK[kk], b[2], b[3]);
                        mma_bf16_16816(Zq[2 * jp], aQ[kk], b[0], b[1]);
                        mma_bf16_16816(Zq[2 * jp + 1], aQ[kk], b[2], b[3]);
                    }
                }
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                uint32_t b[4];
                ldb_nk<0>(Ks, 0, 16 * kk, lane, b);
                if (kk == 0) {
                    mma_bf16_16816_z(S1[0], aQ[kk], b[0], b[1]);
                    mma_bf16_16816_z(S1[1], aQ[kk], b[2], b[3]);
                } else {
                    mma_bf16_16816(S1[0], aQ[kk], b[0], b[1]);
                    mma_bf16_16816(S1[1], aQ[kk], b[2], b[3]);
                }
            }
        }
        uint32_t HkA[NKH][4];
        {
            float hk[NJ][4];
#pragma unroll
            for (int j = 0; j < NJ; ++j)
#pragma unroll
                for (int e = 0; e < 4; ++e) hk[j][e] = gelu3(Zk[j][e]).g;
            pack_slice(hk, HkA);
        }
        {
            float P[8][4];
#pragma unroll
            for (int kk = 0; kk < NKH; ++kk)
#pragma unroll
                for (int p = 0; p < 4; ++p) {
                    uint32_t b[4];
                    ldb_kn<0>(w2s, 16 * p, 16 * kk, lane, b);
                    if (kk == 0) {
                        mma_bf16_16816_z(P[2 * p], HkA[kk], b[0], b[1]);
                        mma_bf16_16816_z(P[2 * p + 1], HkA[kk], b[2], b[3]);
                    } else {
                        mma_bf16_16816(P[2 * p], HkA[kk], b[0], b[1]);
                        mma_bf16_16816(P[2 * p + 1], HkA[kk], b[2], b[3]);
                    }
                }
            put_partial(part, P);
        }
        __syncthreads();
        // E2 = sum of the partials - V (thread: n-tile tid / 32, fragment position tid % 32)
        if (tid < 256) {
            const int nt = tid >> 5, gl = (tid & 31) >> 2, tl = tid & 3, col = 8 * nt + 2 * tl;
            float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int ww = 0; ww < 8; ++ww) {
                const float4 v = *reinterpret_cast<const float4*>(part + ((ww * 8 + nt) * 32 + (tid & 31)) * 4);
                s.x += v.x, s.y += v.y, s.z += v.z, s.w += v.w;
            }
            const uint32_t v0 = *reinterpret_cast<const uint32_t*>(smem + (Vs - sb) + t64(gl, col));
            const uint32_t v1 = *reinterpret_cast<const uint32_t*>(smem + (Vs - sb) + t64(gl + 8, col));
            s.x -= bf16_lo(v0), s.y -= bf16_hi(v0), s.z -= bf16_lo(v1), s.w -= bf16_hi(v1);
            *reinterpret_cast<float4*>(e2f + (nt * 32 + (tid & 31)) * 4) = s;
            *reinterpret_cast<uint32_t*>(smem + OFF_E2B + t64(gl, col)) = pack_bf16(s.x, s.y);
            *reinterpret_cast<uint32_t*>(smem + OFF_E2B + t64(gl + 8, col)) = pack_bf16(s.z, s.w);
        }
        __syncthreads();

        // ================= F2
        float Gk[NJ][4], dHk[NJ][4], dE1[NJ][4], dHq[NJ][4];
        uint32_t E1A[NKH][4], HqA[NKH][4];
        {
            uint32_t aE[4][4];
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) lda_tok(sb + OFF_E2B, kk, lane, aE[kk]);
            // Gk = E2 W2^T and dHk = -D E2 dW2'^T (over d)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
#pragma unroll
                for (int jp = 0; jp < NJ / 2; ++jp) {
                    uint32_t b[4], c[4];
                    ldb_nk<0>(w2s, 16 * jp, 16 * kk, lane, b);
                    ldb_nk<0>(g2s, 16 * jp, 16 * kk, lane, c);
                    if (kk == 0) {
                        mma_bf16_16816_z(Gk[2 * jp], aE[kk], b[0], b[1]);
                        mma_bf16_16816_z(Gk[2 * jp + 1], aE[kk], b[2], b[3]);
                        mma_bf16_16816_z(dHk[2 * jp], aE[kk], c[0], c[1]);
                        mma_bf16_16816_z(dHk[2 * jp + 1], aE[kk], c[2], c[3]);
                    } else {
                        mma_bf16_16816(Gk[2 * jp], aE[kk], b[0], b[1]);
                        mma_bf16_16816(Gk[2 * jp + 1], aE[kk], b[2], b[3]);
                        mma_bf16_16816(dHk[2 * jp], aE[kk], c[0], c[1]);
                        mma_bf16_16816(dHk[2 * jp + 1], aE[kk], c[2], c[3]);
                    }
                }
#pragma unroll
            for (int j = 0; j < NJ; ++j) scale_rows(dHk[j], -eg, -eg8);
        }
        float sa_g = 0.f, sa_g8 = 0.f;  // deta partials of this thread's rows: sum (K dW1') . E1 + (Hk dW2') . E2
        {
            // E1 = Gk . g'(Zk); from here on Zk holds g'(Zk) and Gk holds Gk . g''(Zk), all that the
            // later steps need of them.  P1 = K dW1' (over d); dE1 = -D P1
            float e1[NJ][4];
#pragma unroll
            for (int j = 0; j < NJ; ++j)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const Gelu r = gelu3(Zk[j][e]);
                    e1[j][e] = Gk[j][e] * r.gp;
                    Zk[j][e] = r.gp;
                    Gk[j][e] *= r.gpp;
                }
            pack_slice(e1, E1A);
            uint32_t aK[4][4];
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) lda_tok(Ks, kk, lane, aK[kk]);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
#pragma unroll
                for (int jp = 0; jp < NJ / 2; ++jp) {
                    uint32_t b[4];
                    ldb_kn<HS>(g1s, 16 * jp, 16 * kk, lane, b);
                    if (kk == 0) {
                        mma_bf16_16816_z(dE1[2 * jp], aK[kk], b[0], b[1]);
                        mma_bf16_16816_z(dE1[2 * jp + 1], aK[kk], b[2], b[3]);
                    } else {
                        mma_bf16_16816(dE1[2 * jp], aK[kk], b[0], b[1]);
                        mma_bf16_16816(dE1[2 * jp + 1], aK[kk], b[2], b[3]);
                    }
                }
#pragma unroll
            for (int j = 0; j < NJ; ++j) {
                sa_g = fmaf(dE1[j][0], e1[j][0], fmaf(dE1[j][1], e1[j][1], sa_g));
                sa_g8 = fmaf(dE1[j][2], e1[j][2], fmaf(dE1[j][3], e1[j][3], sa_g8));
                scale_rows(dE1[j], -eg, -eg8);
            }
        }
        {
            // Zq -= (M . S1 D) E1; Hq = g(Zq), keep g'(Zq) in Zq
            uint32_t aS[4];
            {
                float v[2][4];
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int i = g + 8 * (e >> 1), j = colj[2 * h + (e & 1)];
                        v[h][e] = j <= i ? -S1[h][e] * ec[2 * h + (e & 1)] : 0.f;
                    }
                aS[0] = pack_bf16(v[0][0], v[0][1]);
                aS[1] = pack_bf16(v[0][2], v[0][3]);
                aS[2] = pack_bf16(v[1][0], v[1][1]);
                aS[3] = pack_bf16(v[1][2], v[1][3]);
            }
#pragma unroll
            for (int j = 0; j < NJ; ++j) {
                uint32_t b0, b1;
                btok(E1A, j, b0, b1);
                mma_bf16_16816(Zq[j], aS, b0, b1);
            }
            float hq[NJ][4];
#pragma unroll
            for (int j = 0; j < NJ; ++j)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const Gelu r = gelu3(Zq[j][e]);
                    hq[j][e] = r.g;
                    Zq[j][e] = r.gp;
                }
            pack_slice(hq, HqA);
        }
        {
            // dHq = dZ W2^T (over d)
            uint32_t aZ[4][4];
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) lda_tok(dZs, kk, lane, aZ[kk]);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
#pragma unroll
                for (int jp = 0; jp < NJ / 2; ++jp) {
                    uint32_t b[4];
                    ldb_nk<0>(w2s, 16 * jp, 16 * kk, lane, b);
                    if (kk == 0) {
                        mma_bf16_16816_z(dHq[2 * jp], aZ[kk], b[0], b[1]);
                        mma_bf16_16816_z(dHq[2 * jp + 1], aZ[kk], b[2], b[3]);
                    } else {
                        mma_bf16_16816(dHq[2 * jp], aZ[kk], b[0], b[1]);
                        mma_bf16_16816(dHq[2 * jp + 1], aZ[kk], b[2], b[3]);
                    }
                }
        }
        {
            // S2 partial = Hq Hk^T over this warp's hidden units
            float S2p[2][4];
#pragma unroll
            for (int tn = 0; tn < 2; ++tn)
#pragma unroll
                for (int kk = 0; kk < NKH; ++kk) {
                    if (kk == 0)
                        mma_bf16_16816_z(S2p[tn], HqA[kk], HkA[kk][tn], HkA[kk][2 + tn]);
                    else
                        mma_bf16_16816(S2p[tn], HqA[kk], HkA[kk][tn], HkA[kk][2 + tn]);
                }
            put_partial(psm, S2p);
        }
        {
            // (Hk dW2')_j . E2_j over this warp's hidden units (the partial P2 dotted with E2)
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                float P[2][4];
#pragma unroll
                for (int kk = 0; kk < NKH; ++kk) {
                    uint32_t b[4];
                    ldb_kn<0>(g2s, 16 * p, 16 * kk, lane, b);
                    if (kk == 0) {
                        mma_bf16_16816_z(P[0], HkA[kk], b[0], b[1]);
                        mma_bf16_16816_z(P[1], HkA[kk], b[2], b[3]);
                    } else {
                        mma_bf16_16816(P[0], HkA[kk], b[0], b[1]);
                        mma_bf16_16816(P[1], HkA[kk], b[2], b[3]);
                    }
                }
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const float4 e = *reinterpret_cast<const float4*>(e2f + ((2 * p + h) * 32 + lane) * 4);
                    sa_g = fmaf(P[h][0], e.x, fmaf(P[h][1], e.y, sa_g));
                    sa_g8 = fmaf(P[h][2], e.z, fmaf(P[h][3], e.w, sa_g8));
                }
            }
            sa_g += __shfl_xor_sync(0xffffffffu, sa_g, 1);
            sa_g += __shfl_xor_sync(0xffffffffu, sa_g, 2);
            sa_g8 += __shfl_xor_sync(0xffffffffu, sa_g8, 1);
            sa_g8 += __shfl_xor_sync(0xffffffffu, sa_g8, 2);
            if (t == 0) {
                detap[w * 16 + g] = -sa_g;
                detap[w * 16 + g + 8] = -sa_g8;
            }
        }
        __syncthreads();
        if (tid < 64) {  // S2 = sum of the partials, row-major [16][16]
            const int tn = tid >> 5, l = tid & 31, gl = l >> 2, tl = l & 3;
            float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int ww = 0; ww < 8; ++ww) {
                const float4 v = *reinterpret_cast<const float4*>(psm + ((ww * 2 + tn) * 32 + l) * 4);
                s.x += v.x, s.y += v.y, s.z += v.z, s.w += v.w;
            }
            const int col = 8 * tn + 2 * tl;
            s2s[gl * 16 + col] = s.x;
            s2s[gl * 16 + col + 1] = s.y;
            s2s[(gl + 8) * 16 + col] = s.z;
            s2s[(gl + 8) * 16 + col + 1] = s.w;
        }
        __syncthreads();

        // ================= B1: the Z = Hq W2 - (M . S2 D) E2 terms
        uint32_t dZqA[NKH][4];
        {
            // dA2 = -dZ E2^T (every warp; 16 x 16)
            float dA2[2][4];
            {
                uint32_t aZ[4][4];
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) lda_tok(dZs, kk, lane, aZ[kk]);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    uint32_t b[4];
                    ldb_nk<0>(sb + OFF_E2B, 0, 16 * kk, lane, b);
                    if (kk == 0) {
                        mma_bf16_16816_z(dA2[0], aZ[kk], b[0], b[1]);
                        mma_bf16_16816_z(dA2[1], aZ[kk], b[2], b[3]);
                    } else {
                        mma_bf16_16816(dA2[0], aZ[kk], b[0], b[1]);
                        mma_bf16_16816(dA2[1], aZ[kk], b[2], b[3]);
                    }
                }
            }
            // deta_j += sum_{i >= j} dA2_ij S2_ij (warp 0: column sums over its fragments)
            if (w == 0) {
                float cs[4];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int h = c >> 1, e0 = c & 1, j = colj[c];
                    float s = 0.f;
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        const int i = g + 8 * r;
                        if (j <= i) s = fmaf(-dA2[h][2 * r + e0], s2s[i * 16 + j], s);
                    }
                    s += __shfl_xor_sync(0xffffffffu, s, 4);
                    s += __shfl_xor_sync(0xffffffffu, s, 8);
                    s += __shfl_xor_sync(0xffffffffu, s, 16);
                    cs[c] = s;
                }
                if (g == 0) {
#pragma unroll
                    for (int c = 0; c < 4; ++c) detac[colj[c]] = cs[c];
                }
            }
            // dS2 = M . dA2 D as A fragments (and of its transpose)
            uint32_t aD[4], aDT[4];
            {
                float v[2][4];
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int i = g + 8 * (e >> 1), j = colj[2 * h + (e & 1)];
                        v[h][e] = j <= i ? -dA2[h][e] * ec[2 * h + (e & 1)] : 0.f;
                    }
                aD[0] = pack_bf16(v[0][0], v[0][1]);
                aD[1] = pack_bf16(v[0][2], v[0][3]);
                aD[2] = pack_bf16(v[1][0], v[1][1]);
                aD[3] = pack_bf16(v[1][2], v[1][3]);
                aDT[0] = movt(aD[0]);
                aDT[1] = movt(aD[2]);
                aDT[2] = movt(aD[1]);
                aDT[3] = movt(aD[3]);
            }
            // dHq += dS2 Hk, dHk += dS2^T Hq (over tokens)
#pragma unroll
            for (int j = 0; j < NJ; ++j) {
                uint32_t b0, b1;
                btok(HkA, j, b0, b1);
                mma_bf16_16816(dHq[j], aD, b0, b1);
                btok(HqA, j, b0, b1);
                mma_bf16_16816(dHk[j], aDT, b0, b1);
            }
            // -(M . S2 D)^T dZ, d-columns 8 w .. 8 w + 7 (row j, over tokens i: -S2_ij eta_j for j <= i)
            if (w < 8) {
                uint32_t a[4];
                float v[4][2];
#pragma unroll
                for (int q = 0; q < 4; ++q)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int j = g + 8 * (q & 1), i = 2 * t + e + 8 * (q >> 1);
                        v[q][e] = j <= i ? -s2s[i * 16 + j] * es[j] : 0.f;
                    }
#pragma unroll
                for (int q = 0; q < 4; ++q) a[q] = pack_bf16(v[q][0], v[q][1]);
                uint32_t b0, b1;
                ldb_tok1(dZs, 8 * w, lane, b0, b1);
                float c[4];
                mma_bf16_16816_z(c, a, b0, b1);
                *reinterpret_cast<float4*>(de2t + (w * 32 + lane) * 4) = make_float4(c[0], c[1], c[2], c[3]);
            }
            // dZq = dHq . g'(Zq)
            float dzq[NJ][4];
#pragma unroll
            for (int j = 0; j < NJ; ++j)
#pragma unroll
                for (int e = 0; e < 4; ++e) dzq[j][e] = dHq[j][e] * Zq[j][e];
            pack_slice(dzq, dZqA);
        }
        {
            // dQ partial = dZq W1^T (over this warp's hidden units)
            float P[8][4];
#pragma unroll
            for (int kk = 0; kk < NKH; ++kk)
#pragma unroll
                for (int p = 0; p < 4; ++p) {
                    uint32_t b[4];
                    ldb_nk<HS>(w1s, 16 * p, 16 * kk, lane, b);
                    if (kk == 0) {
                        mma_bf16_16816_z(P[2 * p], dZqA[kk], b[0], b[1]);
                        mma_bf16_16816_z(P[2 * p + 1], dZqA[kk], b[2], b[3]);
                    } else {
                        mma_bf16_16816(P[2 * p], dZqA[kk], b[0], b[1]);
                        mma_bf16_16816(P[2 * p + 1], dZqA[kk], b[2], b[3]);
                    }
                }
            put_partial(part, P);
            // dA1 partial = -dZq E1^T
            float A1[2][4];
#pragma unroll
            for (int tn = 0; tn < 2; ++tn)
#pragma unroll
                for (int kk = 0; kk < NKH; ++kk) {
                    if (kk == 0)
                        mma_bf16_16816_z(A1[tn], dZqA[kk], E1A[kk][tn], E1A[kk][2 + tn]);
                    else
                        mma_bf16_16816(A1[tn], dZqA[kk], E1A[kk][tn], E1A[kk][2 + tn]);
                }
#pragma unroll
            for (int tn = 0; tn < 2; ++tn)
#pragma unroll
                for (int e = 0; e < 4; ++e) A1[tn][e] = -A1[tn][e];
            put_partial(psm, A1);
        }
        __syncthreads();
        if (tid < 256) {
            const int nt = tid >> 5, l = tid & 31;
            float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int ww = 0; ww < 8; ++ww) {
                const float4 v = *reinterpret_cast<const float4*>(part + ((ww * 8 + nt) * 32 + l) * 4);
                s.x += v.x, s.y += v.y, s.z += v.z, s.w += v.w;
            }
            *reinterpret_cast<float4*>(dqf + (nt * 32 + l) * 4) = s;
            if (tid < 64) {
                const int tn = tid >> 5, gl = l >> 2, tl = l & 3;
                float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int ww = 0; ww < 8; ++ww) {
                    const float4 v = *reinterpret_cast<const float4*>(psm + ((ww * 2 + tn) * 32 + l) * 4);
                    a.x += v.x, a.y += v.y, a.z += v.z, a.w += v.w;
                }
                const int col = 8 * tn + 2 * tl;
                da1s[gl * 16 + col] = a.x;
                da1s[gl * 16 + col + 1] = a.y;
                da1s[(gl + 8) * 16 + col] = a.z;
                da1s[(gl + 8) * 16 + col + 1] = a.w;
            }
        }
        __syncthreads();

        // ================= B2: the Zq = Q W1 - (M . S1 D) E1 terms, then E1 = Gk . g'(Zk)
        uint32_t dGkA[NKH][4];
        {
            if (w == 0) {  // deta_j += sum_{i >= j} dA1_ij S1_ij
                float cs[4];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int h = c >> 1, e0 = c & 1, j = colj[c];
                    float s = 0.f;
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        const int i = g + 8 * r;
                        if (j <= i) s = fmaf(da1s[i * 16 + j], S1[h][2 * r + e0], s);
                    }
                    s += __shfl_xor_sync(0xffffffffu, s, 4);
                    s += __shfl_xor_sync(0xffffffffu, s, 8);
                    s += __shfl_xor_sync(0xffffffffu, s, 16);
                    cs[c] = s;
                }
                if (g == 0) {
#pragma unroll
                    for (int c = 0; c < 4; ++c) detac[colj[c]] += cs[c];
                }
            }
            // dE1 -= (M . S1 D)^T dZq (over tokens)
            {
                uint32_t a[4], aT[4];
                float v[2][4];
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int i = g + 8 * (e >> 1), j = colj[2 * h + (e & 1)];
                        v[h][e] = j <= i ? -S1[h][e] * ec[2 * h + (e & 1)] : 0.f;
                    }
                a[0] = pack_bf16(v[0][0], v[0][1]);
                a[1] = pack_bf16(v[0][2], v[0][3]);
                a[2] = pack_bf16(v[1][0], v[1][1]);
                a[3] = pack_bf16(v[1][2], v[1][3]);
                aT[0] = movt(a[0]);
                aT[1] = movt(a[2]);
                aT[2] = movt(a[1]);
                aT[3] = movt(a[3]);
#pragma unroll
                for (int j = 0; j < NJ; ++j) {
                    uint32_t b0, b1;
                    btok(dZqA, j, b0, b1);
                    mma_bf16_16816(dE1[j], aT, b0, b1);
                }
            }
            // dQ += dS1 K and dS1^T Q, d-columns 8 w .. (dS1 = M . dA1 D)
            if (w < 8) {
                uint32_t a[4], aT[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    float v[2], vt[2];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int r = g + 8 * (q & 1), c = 2 * t + e + 8 * (q >> 1);
                        v[e] = c <= r ? da1s[r * 16 + c] * es[c] : 0.f;    // dS1[r][c]
                        vt[e] = r <= c ? da1s[c * 16 + r] * es[r] : 0.f;   // dS1[c][r]
                    }
                    a[q] = pack_bf16(v[0], v[1]);
                    aT[q] = pack_bf16(vt[0], vt[1]);
                }
                uint32_t b0, b1;
                ldb_tok1(Ks, 8 * w, lane, b0, b1);
                float4* dq4 = reinterpret_cast<float4*>(dqf + (w * 32 + lane) * 4);
                float c[4] = {dq4->x, dq4->y, dq4->z, dq4->w};
                mma_bf16_16816(c, a, b0, b1);
                *dq4 = make_float4(c[0], c[1], c[2], c[3]);
                ldb_tok1(Qs, 8 * w, lane, b0, b1);
                float k4[4];
                mma_bf16_16816_z(k4, aT, b0, b1);
                *reinterpret_cast<float4*>(dkt + (w * 32 + lane) * 4) = make_float4(k4[0], k4[1], k4[2], k4[3]);
            }
            // dGk = dE1 . g'(Zk) (packed), dZk = dE1 . Gk . g''(Zk) (into Gk)
            float dgk[NJ][4];
#pragma unroll
            for (int j = 0; j < NJ; ++j)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    dgk[j][e] = dE1[j][e] * Zk[j][e];
                    Gk[j][e] *= dE1[j][e];
                }
            pack_slice(dgk, dGkA);
        }
        {
            // dE2 partial = -D (Hk dW2') + dGk W2 (over this warp's hidden units)
            float P[8][4];
#pragma unroll
            for (int kk = 0; kk < NKH; ++kk)
#pragma unroll
                for (int p = 0; p < 4; ++p) {
                    uint32_t b[4];
                    ldb_kn<0>(g2s, 16 * p, 16 * kk, lane, b);
                    if (kk == 0) {
                        mma_bf16_16816_z(P[2 * p], HkA[kk], b[0], b[1]);
                        mma_bf16_16816_z(P[2 * p + 1], HkA[kk], b[2], b[3]);
                    } else {
                        mma_bf16_16816(P[2 * p], HkA[kk], b[0], b[1]);
                        mma_bf16_16816(P[2 * p + 1], HkA[kk], b[2], b[3]);
                    }
                }
#pragma unroll
            for (int nt = 0; nt < 8; ++nt) scale_rows(P[nt], -eg, -eg8);
#pragma unroll
            for (int kk = 0; kk < NKH; ++kk)
#pragma unroll
                for (int p = 0; p < 4; ++p) {
                    uint32_t b[4];
                    ldb_kn<0>(w2s, 16 * p, 16 * kk, lane, b);
                    mma_bf16_16816(P[2 * p], dGkA[kk], b[0], b[1]);
                    mma_bf16_16816(P[2 * p + 1], dGkA[kk], b[2], b[3]);
                }
            put_partial(part, P);
        }
        __syncthreads();
        if (tid < 256) {
            // dE2 = sum + the token term; dV = -dE2
            const int nt = tid >> 5, l = tid & 31, gl = l >> 2, tl = l & 3, col = 8 * nt + 2 * tl;
            float4 s = *reinterpret_cast<const float4*>(de2t + (nt * 32 + l) * 4);
#pragma unroll
            for (int ww = 0; ww < 8; ++ww) {
                const float4 v = *reinterpret_cast<const float4*>(part + ((ww * 8 + nt) * 32 + l) * 4);
                s.x += v.x, s.y += v.y, s.z += v.z, s.w += v.w;
            }
            *reinterpret_cast<uint32_t*>(smem + OFF_DE2B + t64(gl, col)) = pack_bf16(s.x, s.y);
            *reinterpret_cast<uint32_t*>(smem + OFF_DE2B + t64(gl + 8, col)) = pack_bf16(s.z, s.w);
            __nv_bfloat162 o0 = __floats2bfloat162_rn(-s.x, -s.y), o1 = __floats2bfloat162_rn(-s.z, -s.w);
            if (!PART || BT * n + gl < T) *reinterpret_cast<__nv_bfloat162*>(dV + (orow + gl) * D + col) = o0;
            if (!PART || BT * n + gl + 8 < T) *reinterpret_cast<__nv_bfloat162*>(dV + (orow + gl + 8) * D + col) = o1;
        }
        __syncthreads();

        // ================= B3: dHk += dE2 W2^T, dZk, the dK partial, the state gradient
        uint32_t dZkA[NKH][4];
        {
            uint32_t aD[4][4];
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) lda_tok(sb + OFF_DE2B, kk, lane, aD[kk]);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
#pragma unroll
                for (int jp = 0; jp < NJ / 2; ++jp) {
                    uint32_t b[4];
                    ldb_nk<0>(w2s, 16 * jp, 16 * kk, lane, b);
                    mma_bf16_16816(dHk[2 * jp], aD[kk], b[0], b[1]);
                    mma_bf16_16816(dHk[2 * jp + 1], aD[kk], b[2], b[3]);
                }
            float dzk[NJ][4];
#pragma unroll
            for (int j = 0; j < NJ; ++j)
#pragma unroll
                for (int e = 0; e < 4; ++e) dzk[j][e] = fmaf(dHk[j][e], Zk[j][e], Gk[j][e]);
            pack_slice(dzk, dZkA);
        }
        // the running dW1 slice, loaded here so that its L2 round trip overlaps the dK partial
        float2 u1[4][NJ][2];
#pragma unroll
        for (int mt = 0; mt < 4; ++mt)
#pragma unroll
            for (int j = 0; j < NJ; ++j) {
                const float* p0 = dW1g + size_t(16 * mt + g) * HID + hw + 8 * j + 2 * t;
                u1[mt][j][0] = *reinterpret_cast<const float2*>(p0);
                u1[mt][j][1] = *reinterpret_cast<const float2*>(p0 + 8 * HID);
            }
        {
            // dK partial = -D (E1 dW1'^T) + dZk W1^T (over this warp's hidden units)
            float P[8][4];
#pragma unroll
            for (int kk = 0; kk < NKH; ++kk)
#pragma unroll
                for (int p = 0; p < 4; ++p) {
                    uint32_t b[4];
                    ldb_nk<HS>(g1s, 16 * p, 16 * kk, lane, b);
                    if (kk == 0) {
                        mma_bf16_16816_z(P[2 * p], E1A[kk], b[0], b[1]);
                        mma_bf16_16816_z(P[2 * p + 1], E1A[kk], b[2], b[3]);
                    } else {
                        mma_bf16_16816(P[2 * p], E1A[kk], b[0], b[1]);
                        mma_bf16_16816(P[2 * p + 1], E1A[kk], b[2], b[3]);
                    }
                }
#pragma unroll
            for (int nt = 0; nt < 8; ++nt) scale_rows(P[nt], -eg, -eg8);
#pragma unroll
            for (int kk = 0; kk < NKH; ++kk)
#pragma unroll
                for (int p = 0; p < 4; ++p) {
                    uint32_t b[4];
                    ldb_nk<HS>(w1s, 16 * p, 16 * kk, lane, b);
                    mma_bf16_16816(P[2 * p], dZkA[kk], b[0], b[1]);
                    mma_bf16_16816(P[2 * p + 1], dZkA[kk], b[2], b[3]);
                }
            put_partial(part, P);
        }
        // the block's state slices are read for the last time above: bring in the next block's
        __syncwarp();
        if (n >= 1) issue_state(n - 1);
        cp_async_commit();
        {
            // the running dW2 slice, loaded before the dW1 products for the same reason
            float2 u2[NKH][8][2];
#pragma unroll
            for (int p = 0; p < NKH; ++p)
#pragma unroll
                for (int nt = 0; nt < 8; ++nt) {
                    const float* p0 = dW2g + size_t(hw + 16 * p + g) * D + 8 * nt + 2 * t;
                    u2[p][nt][0] = *reinterpret_cast<const float2*>(p0);
                    u2[p][nt][1] = *reinterpret_cast<const float2*>(p0 + 8 * D);
                }
            // dW1[:, slice] += Q^T dZq + K^T dZk (over tokens); refresh the bf16 copy
#pragma unroll
            for (int mt = 0; mt < 4; ++mt) {
                uint32_t aQT[4], aKT[4];
                lda_tokT(Qs, 16 * mt, lane, aQT);
                lda_tokT(Ks, 16 * mt, lane, aKT);
#pragma unroll
                for (int j = 0; j < NJ; ++j) {
                    const int r0 = 16 * mt + g, col = 8 * j + 2 * t;
                    float* p0 = dW1g + size_t(r0) * HID + hw + col;
                    float* p1 = p0 + 8 * HID;
                    float c[4] = {u1[mt][j][0].x, u1[mt][j][0].y, u1[mt][j][1].x, u1[mt][j][1].y};
                    uint32_t b0, b1;
                    btok(dZqA, j, b0, b1);
                    mma_bf16_16816(c, aQT, b0, b1);
                    btok(dZkA, j, b0, b1);
                    mma_bf16_16816(c, aKT, b0, b1);
                    *reinterpret_cast<float2*>(p0) = make_float2(c[0], c[1]);
                    *reinterpret_cast<float2*>(p1) = make_float2(c[2], c[3]);
                    *reinterpret_cast<uint32_t*>(smem + OFF_G1 + w * SZ_W1S + tl<HS>(r0, col)) = pack_bf16(c[0], c[1]);
                    *reinterpret_cast<uint32_t*>(smem + OFF_G1 + w * SZ_W1S + tl<HS>(r0 + 8, col)) =
                        pack_bf16(c[2], c[3]);
                }
            }
            // dW2[slice, :] += Hq^T dZ + dGk^T E2 + Hk^T dE2 (over tokens); refresh the bf16 copy
#pragma unroll
            for (int p = 0; p < NKH; ++p) {
                uint32_t aHq[4], aGk[4], aHk[4];
                atr(HqA, p, aHq);
                atr(dGkA, p, aGk);
                atr(HkA, p, aHk);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    uint32_t bz[4], be[4], bd[4];
                    ldb_kn<0>(dZs, 16 * q, 0, lane, bz);
                    ldb_kn<0>(sb + OFF_E2B, 16 * q, 0, lane, be);
                    ldb_kn<0>(sb + OFF_DE2B, 16 * q, 0, lane, bd);
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int r0 = 16 * p + g, col = 16 * q + 8 * h + 2 * t;
                        float* p0 = dW2g + size_t(hw + r0) * D + col;
                        float* p1 = p0 + 8 * D;
                        const int nt = 2 * q + h;
                        float c[4] = {u2[p][nt][0].x, u2[p][nt][0].y, u2[p][nt][1].x, u2[p][nt][1].y};
                        mma_bf16_16816(c, aHq, bz[2 * h], bz[2 * h + 1]);
                        mma_bf16_16816(c, aGk, be[2 * h], be[2 * h + 1]);
                        mma_bf16_16816(c, aHk, bd[2 * h], bd[2 * h + 1]);
                        *reinterpret_cast<float2*>(p0) = make_float2(c[0], c[1]);
                        *reinterpret_cast<float2*>(p1) = make_float2(c[2], c[3]);
                        *reinterpret_cast<uint32_t*>(smem + OFF_G2 + w * SZ_W2S + t64(r0, col)) = pack_bf16(c[0], c[1]);
                        *reinterpret_cast<uint32_t*>(smem + OFF_G2 + w * SZ_W2S + t64(r0 + 8, col)) =
                            pack_bf16(c[2], c[3]);
                    }
                }
            }
        }
        __syncthreads();
        if (tid < 256) {
            // dK = sum + dS1^T Q; dQ; deta
            const int nt = tid >> 5, l = tid & 31, gl = l >> 2, tl = l & 3, col = 8 * nt + 2 * tl;
            float4 s = *reinterpret_cast<const float4*>(dkt + (nt * 32 + l) * 4);
#pragma unroll
            for (int ww = 0; ww < 8; ++ww) {
                const float4 v = *reinterpret_cast<const float4*>(part + ((ww * 8 + nt) * 32 + l) * 4);
                s.x += v.x, s.y += v.y, s.z += v.z, s.w += v.w;
            }
            const float4 q = *reinterpret_cast<const float4*>(dqf + (nt * 32 + l) * 4);
            if (!PART || BT * n + gl < T) {  // rows past T are not stored
                *reinterpret_cast<__nv_bfloat162*>(dK + (orow + gl) * D + col) = __floats2bfloat162_rn(s.x, s.y);
                *reinterpret_cast<__nv_bfloat162*>(dQ + (orow + gl) * D + col) = __floats2bfloat162_rn(q.x, q.y);
            }
            if (!PART || BT * n + gl + 8 < T) {
                *reinterpret_cast<__nv_bfloat162*>(dK + (orow + gl + 8) * D + col) = __floats2bfloat162_rn(s.z, s.w);
                *reinterpret_cast<__nv_bfloat162*>(dQ + (orow + gl + 8) * D + col) = __floats2bfloat162_rn(q.z, q.w);
            }
            if (tid < BT) {
                float d = detac[tid];
#pragma unroll
                for (int ww = 0; ww < NW; ++ww) d += detap[ww * 16 + tid];
                if (!PART || BT * n + tid < T) deta[orow + tid] = d;
            }
        }
    }
    cp_async_wait0();
}

}  // namespace

bool mlp_backward_mma_supported(const MlpBwdArgs& a) {
    return a.bf16 && a.d == D && a.hidden == HID && a.chunk == BT;  // any T
}

template <int NW, bool PART>
cudaError_t launch_nw(const MlpBwdArgs& a, cudaStream_t s) {
    using C = BwdCfg<NW>;
    auto kern = mlp_backward_mma_kernel<NW, PART>;
    cudaError_t e = allow_dynamic_smem(reinterpret_cast<const void*>(kern), C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    kern<<<unsigned(a.B) * unsigned(a.H), C::NTH, C::SMEM_BYTES, s>>>(
        static_cast<const __nv_bfloat16*>(a.Q), static_cast<const __nv_bfloat16*>(a.K),
        static_cast<const __nv_bfloat16*>(a.V), a.eta, static_cast<const __nv_bfloat16*>(a.W1_hist),
        static_cast<const __nv_bfloat16*>(a.W2_hist), static_cast<const __nv_bfloat16*>(a.dZ), a.dW1_T, a.dW2_T,
        static_cast<__nv_bfloat16*>(a.dQ), static_cast<__nv_bfloat16*>(a.dK), static_cast<__nv_bfloat16*>(a.dV),
        a.deta, a.dW1_0, a.dW2_0, a.T);
    return cudaGetLastError();
}

cudaError_t launch_mlp_backward_mma(const MlpBwdArgs& a, cudaStream_t s) {
    if (!mlp_backward_mma_supported(a)) return cudaErrorNotSupported;
    // eight warps of 32 hidden units each; TTT_MLP_BACKWARD_WARPS = 16 selects sixteen of 16 (correct, and
    // measured slower on the TTT-MLP workload shape: 2.12 against 1.65 ms -- the per-warp work on the token
    // side does not shrink, each reduction takes one more barrier, and 128 registers per thread)
    const char* v = getenv("TTT_MLP_BACKWARD_WARPS");
    if (a.T % BT) return (v && !strcmp(v, "16")) ? launch_nw<16, true>(a, s) : launch_nw<8, true>(a, s);
    return (v && !strcmp(v, "16")) ? launch_nw<16, false>(a, s) : launch_nw<8, false>(a, s);
}

}  // namespace ttt
