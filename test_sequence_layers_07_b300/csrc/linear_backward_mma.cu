// linear_backward_mma.cu -- gradient of the TTT-Linear scan on warp-level tensor-core MMAs
// (bf16 Q/K/V/dZ/dQ/dK/dV, fp32 state gradients), d = 64, blocks of 16 tokens.
//
// What is computed (linear_backward.cu states it in full): per block of 16 tokens, in reverse
// order, with W the block-start state, dW' the gradient of the state after the block,
// D = diag(eta), M the causal mask, S = Q K^T, A = (M . S) D, E = K W - V:
//     dE = -A^T dZ - D K dW'          dA = -dZ E^T,  dS = M . dA D
//     dQ = dZ W^T + dS K              dK = dE W^T - D E dW'^T + dS^T Q
//     dV = -dE                        deta_j = -sum_c E_jc (K dW')_jc + sum_i M_ij dA_ij S_ij
//     dW = dW' + Q^T dZ + K^T dE
// (training the outer model through the inner loop: TTT essay, ren-xubin.github.io, paragraph
// on the two time scales).  deta's first term is written -sum_k K_jk (E dW'^T)_jk, the same sum.
//
// Design (ours, for sm_103a), after the forward kernel (linear_prefill_mma.cu):
//  * The dW chain is column-separable (column c of dE and dW needs only column c of dZ and dW'),
//    so four chain warps, one per 16-column group, carry dW^T in registers in the MMA accumulator
//    layout and run the recurrence: P = K dW' (as P^T = dW'^T K^T), dE^T = -(dZ^T A + P^T D),
//    dW^T += dZ^T Q + dE^T K.  They export dE by stmatrix into a [16][64] tile per block.
//  * A scores warp forms S = Q K^T once per block (as K Q^T, whose accumulator fragments are the
//    B fragments of A with K = the query index) and keeps S in fp32 for deta.
//  * Four read-out warps take the sums over all columns (dQ, dK, deta): warp r forms columns
//    [16r, 16r + 16) of E = K W - V and the partial dA, then rows [16r, 16r + 16) of dQ and dK.
//    The term E dW'^T needs dW' with the column index as the contraction: each read-out warp
//    keeps its own copy of rows [16r, 16r + 16) of dW (same updates, dW = dW' + Q^T dZ + K^T dE),
//    whose accumulator fragments are exactly those B fragments.
//  * The block-start states (bf16, as the forward recorded them: 8 KB a block) stream in by
//    cp.async, three blocks ahead, straight into a 4-slot ring of swizzled [64][64] tiles, from
//    which ldmatrix reads both the W and the W^T fragments.
//  * Q/K/V/dZ arrive by TMA in reverse token order, 4 blocks a stage, 3 stages.
//  * All mbarrier waits are bounded; the read-out warps meet at reducing barriers (bar.red.or of
//    the per-thread error flag), so after an expired wait every role leaves its loop.
#include <cuda.h>

#include "ptx.cuh"
#include "ttt_common.cuh"
#include "ttt_internal.h"

namespace ttt {
namespace {

using namespace ptx;

constexpr uint64_t kWaitLimitNs = 4000000000ull;  // 4 s: far beyond any legitimate wait
constexpr int D = 64, CG = 4, SPS = 4, NST = 3, NW = 4;
constexpr int KS = D / 16, NT = D / 8;
constexpr int TILE = 16 * D * 2;  // one [16][64] bf16 block tile (one TMA box)
// stage slot: Q, K, V, dZ tiles of SPS blocks (processing order), then eta (SPS x 16 fp32, token order)
constexpr int QOFF = 0, KOFF = SPS * TILE, VOFF = 2 * SPS * TILE, ZOFF = 3 * SPS * TILE, EOFF = 4 * SPS * TILE;
constexpr int STAGE = (EOFF + SPS * 64 + 1023) / 1024 * 1024;
constexpr int WB_OFF = NST * STAGE;                // W ring: NW x [64][64] bf16, 128-byte swizzled rows
constexpr int WSLOT = D * D * 2;
constexpr int SC_OFF = WB_OFF + NW * WSLOT;        // scores ring [NST][SPS]: A fragments (512 B) + S [16][16] fp32
constexpr int SCSZ = 512 + 1024;
constexpr int DE_OFF = SC_OFF + NST * SPS * SCSZ;  // dE ring [NST][SPS] x [16][64] bf16
constexpr int ET_OFF = DE_OFF + NST * SPS * TILE;  // E [16][64] bf16
constexpr int DAP_OFF = ET_OFF + TILE;             // dA partials [4 warps][32 lanes] x 8 fp32
constexpr int DAS_OFF = DAP_OFF + 4 * 32 * 32;     // summed dA [16][17] fp32 (read-out warp 0)
constexpr int DEP_OFF = DAS_OFF + 1152;            // deta partials [4][16] fp32, then the S-term [16]
constexpr int STG_OFF = DEP_OFF + 5 * 64;          // per read-out warp: dQ, dK staging [16][16] bf16 each
constexpr int BYTES = STG_OFF + 4 * 1024;
constexpr int THREADS = 32 * (2 + 2 * CG);
static_assert(BYTES + 1024 <= 232448, "shared memory");
static_assert(WB_OFF % 1024 == 0, "swizzled W slots must be 1024-byte aligned");

// byte offset of (row, col) in a [rows][64] bf16 tile with 128-byte rows, 16-byte chunk XOR row % 8;
// col % 8 == 0
__device__ __forceinline__ uint32_t swz(int row, int col) {
    return uint32_t(row * 128 + ((((col >> 3) ^ row) & 7) << 4));
}

template <int NK>
__device__ __forceinline__ void pack_state(const float (&w)[2 * NK][4], uint32_t (&wa)[NK][4]) {
#pragma unroll
    for (int ks = 0; ks < NK; ++ks) {
        wa[ks][0] = pack_bf16(w[2 * ks][0], w[2 * ks][1]);
        wa[ks][1] = pack_bf16(w[2 * ks][2], w[2 * ks][3]);
        wa[ks][2] = pack_bf16(w[2 * ks + 1][0], w[2 * ks + 1][1]);
        wa[ks][3] = pack_bf16(w[2 * ks + 1][2], w[2 * ks + 1][3]);
    }
}

__device__ __forceinline__ uint32_t movt(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait2() { asm volatile("cp.async.wait_group 2;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait0() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// barrier over the read-out warps (named barrier 1) that also ORs a per-thread flag
__device__ __forceinline__ bool bar_readout_any(bool c) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, 1, %2, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(uint32_t(c)), "n"(32 * CG)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ float2 bf16x2_at(const uint8_t* tile, int row, int col) {  // col even
    const uint32_t v = *reinterpret_cast<const uint32_t*>(tile + swz(row, col & ~7) + (col & 7) * 2);
    return make_float2(bf16_lo(v), bf16_hi(v));
}

// PART: T is not a multiple of 16 (a partial last block, the first one processed), or the rows of
// all heads exceed the int32 coordinate of a 2D tensor map.  Then Q/K/V/dZ come through per-head 3D
// maps (tokens past a head's end read as zeros, so they add nothing to any gradient), eta by cp.async
// where a bulk copy cannot take it (zeros past T), and no output row past T is stored; the
// instantiation for the common case compiles none of that.
template <bool PART>
__global__ void __launch_bounds__(THREADS, 1)
linear_backward_mma_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                           const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmZ,
                           const float* __restrict__ eta, const __nv_bfloat16* __restrict__ W_hist,
                           const float* __restrict__ dW_T, __nv_bfloat16* __restrict__ dQ,
                           __nv_bfloat16* __restrict__ dK, __nv_bfloat16* __restrict__ dV, float* __restrict__ deta,
                           float* __restrict__ dW0, int T, int* status) {
    extern __shared__ uint8_t smem_dyn[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
    __shared__ __align__(8) uint64_t full_bar[NST];   // TMA tiles and eta of a stage landed
    __shared__ __align__(8) uint64_t sc_bar[NST];     // scores of a stage written
    __shared__ __align__(8) uint64_t xf_bar[NST];     // dE of a stage exported (all chain warps)
    __shared__ __align__(8) uint64_t empty_bar[NST];  // scores and read-out warps done with a stage
    __shared__ volatile int s_err;
    __shared__ volatile int s_zero;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const size_t bh = blockIdx.x;
    const int nsb = PART ? (T + 15) / 16 : T / 16;  // blocks of 16 tokens (with PART the last may be partial)
    const int nstg = (nsb + SPS - 1) / SPS;  // stages
    const uint32_t sbase = smem_u32(smem);
    const int g = lane >> 2, t = lane & 3;
    const int lj = lane >> 3, lr = lane & 7;
    // processing order: stage si holds blocks hi(si), hi(si) - 1, ..., hi(si) - n + 1
    auto subs_in = [&](int si) { return nsb - si * SPS < SPS ? nsb - si * SPS : SPS; };
    auto hi_of = [&](int si) { return nsb - 1 - si * SPS; };

    if (threadIdx.x == 0) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(smem_u32(&full_bar[s]), 1);
            mbar_init(smem_u32(&sc_bar[s]), 1);
            mbar_init(smem_u32(&xf_bar[s]), CG);
            mbar_init(smem_u32(&empty_bar[s]), CG + 1);
        }
        s_err = 0;
        s_zero = 0;
        fence_mbar_init();
    }
    __syncthreads();

    auto wait = [&](uint64_t& bar, uint32_t parity) -> bool {
        if (s_err || !mbar_wait_bounded(smem_u32(&bar), parity, &s_err, kWaitLimitNs)) {
            if (!s_err) record_status(status, kStatusTimeout);
            s_err = 1;
            return false;
        }
        return true;
    };
    // the same wait taken by a whole warp, with a warp-uniform outcome: lanes must never part ways
    // before the warp-wide ldmatrix / mma.sync that follow
    auto wait_all = [&](uint64_t& bar, uint32_t parity) -> bool {
        return __all_sync(0xffffffffu, wait(bar, parity));
    };

    // ldmatrix offsets inside a [16][64] tile, k-step ks:
    //  off_nk: tiles (rows 0-7, k lo), (rows 0-7, k hi), (rows 8-15, k lo), (rows 8-15, k hi): the B
    //          fragments with N = rows (n-tiles 0, 1)
    //  off_tk: tiles (rows 0-7, cols lo), (rows 8-15, cols lo), (rows 0-7, cols hi), (rows 8-15, cols hi):
    //          plain, the A fragment (M = rows); with .trans, the B fragments with K = rows for the
    //          column n-tiles 2 ks, 2 ks + 1
    uint32_t off_nk[KS], off_tk[KS];
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
        off_nk[ks] = swz(lr + 8 * (lj >> 1), 16 * ks + 8 * (lj & 1));
        off_tk[ks] = swz(lr + 8 * (lj & 1), 16 * ks + 8 * (lj >> 1));
    }

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer (reverse order)
        if (lane == 0) {
            prefetch_tensormap(&tmQ);
            prefetch_tensormap(&tmK);
            prefetch_tensormap(&tmV);
            prefetch_tensormap(&tmZ);
            int issued = 0;
            for (int si = 0; si < nstg; ++si) {
                const int s = si % NST, n = subs_in(si), hi = hi_of(si);
                if (si >= NST && !wait(empty_bar[s], ((si / NST) - 1) & 1)) break;
                const uint32_t fb = smem_u32(&full_bar[s]);
                const uint32_t st = sbase + s * STAGE;
                if constexpr (PART) {
                    // eta of blocks hi - n + 1 .. hi (token order): one bulk copy when all their tokens
                    // exist and a head's eta starts on a 16-byte boundary (4 | T); otherwise 4-byte
                    // cp.async copies that the stage's mbarrier tracks, and zeros past T
                    const int t0 = 16 * (hi - n + 1), tok = min(16 * n, T - t0);
                    const bool eb = (T & 3) == 0 && tok == 16 * n;
                    if (!eb) {
                        const float* eg = eta + bh * T + t0;
                        float* es = reinterpret_cast<float*>(smem + s * STAGE + EOFF);
                        for (int j = 0; j < 16 * n; ++j) {
                            if (j < tok) cp_async4(st + EOFF + 4 * j, eg + j);
                            else es[j] = 0.f;
                        }
                        cp_async_mbar_arrive(fb);  // before this thread's own arrive on the phase
                    }
                    mbar_arrive_expect_tx(fb, uint32_t(n) * 4 * TILE + (eb ? uint32_t(n) * 64 : 0u));
                    for (int i = 0; i < n; ++i) {
                        const int y = 16 * (hi - i), z = int(bh);
                        tma_load_3d(st + QOFF + i * TILE, &tmQ, 0, y, z, fb);
                        tma_load_3d(st + KOFF + i * TILE, &tmK, 0, y, z, fb);
                        tma_load_3d(st + VOFF + i * TILE, &tmV, 0, y, z, fb);
                        tma_load_3d(st + ZOFF + i * TILE, &tmZ, 0, y, z, fb);
                    }
                    if (eb) bulk_load(st + EOFF, eta + bh * T + t0, uint32_t(n) * 64, fb);
                } else {
                    mbar_arrive_expect_tx(fb, uint32_t(n) * (4 * TILE + 64));
                    for (int i = 0; i < n; ++i) {
                        const int y = int(bh * T) + 16 * (hi - i);
                        tma_load_2d(st + QOFF + i * TILE, &tmQ, 0, y, fb);
                        tma_load_2d(st + KOFF + i * TILE, &tmK, 0, y, fb);
                        tma_load_2d(st + VOFF + i * TILE, &tmV, 0, y, fb);
                        tma_load_2d(st + ZOFF + i * TILE, &tmZ, 0, y, fb);
                    }
                    bulk_load(st + EOFF, eta + bh * T + 16 * (hi - n + 1), uint32_t(n) * 64, fb);
                }
                ++issued;
            }
            for (int si = issued > NST ? issued - NST : 0; si < issued; ++si)
                mbar_wait_bounded(smem_u32(&full_bar[si % NST]), (si / NST) & 1, &s_zero, kWaitLimitNs);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ scores: X = K Q^T (rows key j, cols query i)
        for (int si = 0; si < nstg; ++si) {
            const int s = si % NST, n = subs_in(si);
            if (!wait_all(full_bar[s], (si / NST) & 1)) break;
            const uint32_t st = sbase + s * STAGE;
            for (int i = 0; i < n; ++i) {
                float x0[2][4] = {}, x1[2][4] = {};
#pragma unroll
                for (int ks = 0; ks < KS; ++ks) {
                    uint32_t ka[4], qb[4];
                    ldsm_x4(st + KOFF + i * TILE + off_tk[ks], ka);
                    ldsm_x4(st + QOFF + i * TILE + off_nk[ks], qb);
                    float(&acc)[2][4] = (ks & 1) ? x1 : x0;
                    mma_bf16_16816(acc[0], ka, qb[0], qb[1]);  // queries 0-7
                    mma_bf16_16816(acc[1], ka, qb[2], qb[3]);  // queries 8-15
                }
#pragma unroll
                for (int j = 0; j < 2; ++j)
#pragma unroll
                    for (int k = 0; k < 4; ++k) x0[j][k] += x1[j][k];
                // x0[it][k]: key j = g (+8 for k >= 2), query i = 8 it + 2t (+1 for odd k)
                const float* es = reinterpret_cast<const float*>(smem + s * STAGE + EOFF + (n - 1 - i) * 64);
                const float eg = es[g], eg8 = es[g + 8];
                // A = (M . S) D as B fragments (K = query i, N = key j): keep key <= query
                uint4 am;
                am.x = pack_bf16(g <= 2 * t ? x0[0][0] * eg : 0.f, g <= 2 * t + 1 ? x0[0][1] * eg : 0.f);
                am.y = pack_bf16(x0[1][0] * eg, x0[1][1] * eg);
                am.z = 0u;
                am.w = pack_bf16(g <= 2 * t ? x0[1][2] * eg8 : 0.f, g <= 2 * t + 1 ? x0[1][3] * eg8 : 0.f);
                uint8_t* sc = smem + SC_OFF + (s * SPS + i) * SCSZ;
                *reinterpret_cast<uint4*>(sc + lane * 16) = am;
                // S[i][j] in fp32 for deta
                float* S = reinterpret_cast<float*>(sc + 512);
#pragma unroll
                for (int it = 0; it < 2; ++it) {
                    const int i0 = 8 * it + 2 * t;
                    S[i0 * 16 + g] = x0[it][0];
                    S[(i0 + 1) * 16 + g] = x0[it][1];
                    S[i0 * 16 + g + 8] = x0[it][2];
                    S[(i0 + 1) * 16 + g + 8] = x0[it][3];
                }
            }
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(smem_u32(&sc_bar[s]));
                mbar_arrive(smem_u32(&empty_bar[s]));
            }
        }
    } else if (warp < 2 + CG) {
        // ------------------------------------------------------------ chain: dW^T of 16 columns
        const int cg = warp - 2, cw0 = 16 * cg;
        float w[NT][4];  // dW^T[c][d_in], c = cw0 + g (+8), d_in = 8 nt + 2t (+1)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int r = 8 * nt + 2 * t;
            const float* src = dW_T + bh * D * D;
            w[nt][0] = dW_T ? src[size_t(r) * D + cw0 + g] : 0.f;
            w[nt][1] = dW_T ? src[size_t(r + 1) * D + cw0 + g] : 0.f;
            w[nt][2] = dW_T ? src[size_t(r) * D + cw0 + g + 8] : 0.f;
            w[nt][3] = dW_T ? src[size_t(r + 1) * D + cw0 + g + 8] : 0.f;
        }
        const uint32_t off_z = swz(lr + 8 * (lj >> 1), cw0 + 8 * (lj & 1));  // dZ^T A fragment of the group
        const int st_row = lr + 8 * (lj >> 1), st_col = cw0 + 8 * (lj & 1);  // stmatrix.trans rows (tokens)
        // prefetched one block ahead: what the first products of a step read (K rows, dZ^T, A, eta);
        // the transposed K and Q fragments of the update load inside the step
        uint32_t kb[KS][4], zt[4];
        uint4 am;
        float e0 = 0, e1 = 0, e2 = 0, e3 = 0;  // eta of tokens 2t, 2t + 1, 8 + 2t, 9 + 2t
        auto load = [&](int s, int i, int n) {
            const uint32_t st = sbase + s * STAGE;
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) ldsm_x4(st + KOFF + i * TILE + off_nk[ks], kb[ks]);
            ldsm_x4_trans(st + ZOFF + i * TILE + off_z, zt);
            am = *reinterpret_cast<const uint4*>(smem + SC_OFF + (s * SPS + i) * SCSZ + lane * 16);
            const float* es = reinterpret_cast<const float*>(smem + s * STAGE + EOFF + (n - 1 - i) * 64);
            const float2 a = *reinterpret_cast<const float2*>(es + 2 * t);
            const float2 b = *reinterpret_cast<const float2*>(es + 8 + 2 * t);
            e0 = a.x; e1 = a.y; e2 = b.x; e3 = b.y;
        };
        bool ok = wait_all(full_bar[0], 0) && wait_all(sc_bar[0], 0);
        if (ok) load(0, 0, subs_in(0));
        for (int si = 0; ok && si < nstg; ++si) {
            const int s = si % NST, n = subs_in(si);
            uint8_t* det = smem + DE_OFF + s * SPS * TILE;
            auto step = [&](int i) {
                const uint32_t st = sbase + s * STAGE;
                uint32_t wa[KS][4];
                pack_state<KS>(w, wa);
                // P^T = dW'^T K^T (16 columns x 16 tokens), in two partial chains
                float pa[2][2][4] = {};
#pragma unroll
                for (int ks = 0; ks < KS; ++ks) {
                    mma_bf16_16816(pa[ks & 1][0], wa[ks], kb[ks][0], kb[ks][1]);
                    mma_bf16_16816(pa[ks & 1][1], wa[ks], kb[ks][2], kb[ks][3]);
                }
                // T1^T = dZ^T A
                float t1[2][4] = {};
                mma_bf16_16816(t1[0], zt, am.x, am.y);
                mma_bf16_16816(t1[1], zt, am.z, am.w);
                float p[2][4];
#pragma unroll
                for (int j = 0; j < 2; ++j)
#pragma unroll
                    for (int k = 0; k < 4; ++k) p[j][k] = pa[0][j][k] + pa[1][j][k];
                // dE^T = -(T1^T + P^T D), as a bf16 A fragment (rows c, K = token)
                uint32_t ge[4];
                ge[0] = pack_bf16(-fmaf(e0, p[0][0], t1[0][0]), -fmaf(e1, p[0][1], t1[0][1]));
                ge[1] = pack_bf16(-fmaf(e0, p[0][2], t1[0][2]), -fmaf(e1, p[0][3], t1[0][3]));
                ge[2] = pack_bf16(-fmaf(e2, p[1][0], t1[1][0]), -fmaf(e3, p[1][1], t1[1][1]));
                ge[3] = pack_bf16(-fmaf(e2, p[1][2], t1[1][2]), -fmaf(e3, p[1][3], t1[1][3]));
                // dW^T += dZ^T Q + dE^T K
#pragma unroll
                for (int kk = 0; kk < KS; ++kk) {
                    uint32_t qt[4], kt[4];
                    ldsm_x4_trans(st + QOFF + i * TILE + off_tk[kk], qt);
                    ldsm_x4_trans(st + KOFF + i * TILE + off_tk[kk], kt);
                    mma_bf16_16816(w[2 * kk], zt, qt[0], qt[1]);
                    mma_bf16_16816(w[2 * kk + 1], zt, qt[2], qt[3]);
                    mma_bf16_16816(w[2 * kk], ge, kt[0], kt[1]);
                    mma_bf16_16816(w[2 * kk + 1], ge, kt[2], kt[3]);
                }
                // dE of this group's columns into the block's [16][64] tile (rows tokens)
                stsm_x4_trans(smem_u32(det + i * TILE) + swz(st_row, st_col), ge[0], ge[1], ge[2], ge[3]);
            };
            if (n == SPS) {
#pragma unroll
                for (int i = 0; i < SPS; ++i) {
                    step(i);
                    if (i + 1 < SPS) load(s, i + 1, n);
                }
            } else {
                for (int i = 0; i < n; ++i) {
                    step(i);
                    if (i + 1 < n) load(s, i + 1, n);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&xf_bar[s]));
            if (si + 1 < nstg) {
                const int s1 = (si + 1) % NST;
                const uint32_t par = ((si + 1) / NST) & 1;
                ok = wait_all(full_bar[s1], par) && wait_all(sc_bar[s1], par);
                if (ok) load(s1, 0, subs_in(si + 1));
            }
        }
        float* out = dW0 + bh * D * D;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int r = 8 * nt + 2 * t;
            out[size_t(r) * D + cw0 + g] = w[nt][0];
            out[size_t(r + 1) * D + cw0 + g] = w[nt][1];
            out[size_t(r) * D + cw0 + g + 8] = w[nt][2];
            out[size_t(r + 1) * D + cw0 + g + 8] = w[nt][3];
        }
    } else {
        // ------------------------------------------------------------ read-out warps
        const int r = warp - 2 - CG;     // column slice of E, row slice of dQ / dK
        const int rt = threadIdx.x - 32 * (2 + CG);  // 0..127
        // dW rows d_in = 16 r + g (+8), columns c = 8 nt + 2t (+1): the same updates as the chain
        float rep[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const float* src = dW_T + bh * D * D;
            const int r0 = 16 * r + g, c0 = 8 * nt + 2 * t;
            rep[nt][0] = dW_T ? src[size_t(r0) * D + c0] : 0.f;
            rep[nt][1] = dW_T ? src[size_t(r0) * D + c0 + 1] : 0.f;
            rep[nt][2] = dW_T ? src[size_t(r0 + 8) * D + c0] : 0.f;
            rep[nt][3] = dW_T ? src[size_t(r0 + 8) * D + c0 + 1] : 0.f;
        }
        // the block-start state of the p-th block in processing order, by cp.async: this thread's
        // four 16-byte chunks of the 8 KB bf16 block, placed in the swizzled layout of slot p % NW
        auto fetch_w = [&](int p) {
            if (p < nsb) {
                const int sb = nsb - 1 - p;
                const __nv_bfloat16* src = W_hist + (bh * nsb + sb) * size_t(D) * D;
                const uint32_t dst = sbase + WB_OFF + (p % NW) * WSLOT;
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int q = rt + 128 * u;  // chunk 0..511: row q >> 3, columns 8 (q & 7) ..
                    const int din = q >> 3, c8 = (q & 7) * 8;
                    cp_async16(dst + swz(din, c8), src + din * D + c8);
                }
            }
            cp_async_commit();
        };
        fetch_w(0);
        fetch_w(1);
        fetch_w(2);
        cp_async_wait2();
        bool err = bar_readout_any(false);  // every thread's chunks of block 0 are in
        const int st_row = lr + 8 * (lj & 1), st_col = 8 * (lj >> 1);  // stmatrix rows of an A-layout tile
        float* dep = reinterpret_cast<float*>(smem + DEP_OFF);           // [4][16] partials, then [16] S-term
        uint8_t* stg = smem + STG_OFF + r * 1024;
        int p = 0;  // processing index
        for (int si = 0; si < nstg; ++si) {
            const int s = si % NST, n = subs_in(si), hi = hi_of(si);
            const uint32_t par = (si / NST) & 1;
            if (!err && !(wait(full_bar[s], par) && wait(sc_bar[s], par) && wait(xf_bar[s], par))) err = true;
            const uint32_t st = sbase + s * STAGE;
            const uint8_t* stp = smem + s * STAGE;
            for (int i = 0; i < n; ++i, ++p) {
                const int sb = hi - i;
                cp_async_wait2();  // this thread's chunks of the state of block p
                // ---- barrier A: the state of block p is in, every warp is done with block p - 1
                if (bar_readout_any(err)) { err = true; break; }
                if (p >= 1 && r == 0 && lane < 16 && (!PART || 16 * (sb + 1) + lane < T))
                    deta[bh * T + 16 * (sb + 1) + lane] =
                        dep[64 + lane] + ((dep[lane] + dep[16 + lane]) + (dep[32 + lane] + dep[48 + lane]));
                fetch_w(p + 3);  // into the slot of block p - 1
                const uint32_t wb = sbase + WB_OFF + (p % NW) * WSLOT;
                const float* es = reinterpret_cast<const float*>(stp + EOFF + (n - 1 - i) * 64);
                const uint8_t* Kt_ = stp + KOFF + i * TILE;
                const uint8_t* Vt_ = stp + VOFF + i * TILE;

                // ---- E columns [16r, 16r + 16) = K W - V; dA partial = -dZ[:, slice] E[:, slice]^T
                float e[2][4] = {};
#pragma unroll
                for (int ks = 0; ks < KS; ++ks) {
                    uint32_t ka[4], wk[4];
                    ldsm_x4(st + KOFF + i * TILE + off_tk[ks], ka);
                    // W as B (K = d_in, N = c 16r ..): transposed loads of the rows d_in
                    ldsm_x4_trans(wb + swz(16 * ks + lr + 8 * (lj & 1), 16 * r + 8 * (lj >> 1)), wk);
                    mma_bf16_16816(e[0], ka, wk[0], wk[1]);
                    mma_bf16_16816(e[1], ka, wk[2], wk[3]);
                }
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    const int c = 16 * r + 8 * nt + 2 * t;
                    const float2 v0 = bf16x2_at(Vt_, g, c), v1 = bf16x2_at(Vt_, g + 8, c);
                    e[nt][0] -= v0.x; e[nt][1] -= v0.y; e[nt][2] -= v1.x; e[nt][3] -= v1.y;
                }
                stsm_x4(sbase + ET_OFF + swz(st_row, 16 * r + st_col), pack_bf16(e[0][0], e[0][1]),
                        pack_bf16(e[0][2], e[0][3]), pack_bf16(e[1][0], e[1][1]), pack_bf16(e[1][2], e[1][3]));
                {
                    uint32_t za[4];
                    ldsm_x4(st + ZOFF + i * TILE + swz(st_row, 16 * r + st_col), za);
                    float da[2][4] = {};
                    mma_bf16_16816(da[0], za, pack_bf16(e[0][0], e[0][1]), pack_bf16(e[1][0], e[1][1]));
                    mma_bf16_16816(da[1], za, pack_bf16(e[0][2], e[0][3]), pack_bf16(e[1][2], e[1][3]));
                    float4* dap = reinterpret_cast<float4*>(smem + DAP_OFF + (r * 32 + lane) * 32);
                    dap[0] = make_float4(-da[0][0], -da[0][1], -da[0][2], -da[0][3]);
                    dap[1] = make_float4(-da[1][0], -da[1][1], -da[1][2], -da[1][3]);
                }
                // ---- barrier B: E and the dA partials of block p are complete
                if (bar_readout_any(err)) { err = true; break; }

                // dA (rows query i, cols key j), dS = M . dA D; dS^T by register transposes
                float ds[2][4];
                {
                    const float4* dap = reinterpret_cast<const float4*>(smem + DAP_OFF);
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt) {
                        float4 a = dap[(0 * 32 + lane) * 2 + nt];
#pragma unroll
                        for (int w2 = 1; w2 < 4; ++w2) {
                            const float4 b = dap[(w2 * 32 + lane) * 2 + nt];
                            a.x += b.x; a.y += b.y; a.z += b.z; a.w += b.w;
                        }
                        ds[nt][0] = a.x; ds[nt][1] = a.y; ds[nt][2] = a.z; ds[nt][3] = a.w;
                    }
                }
                if (r == 0) {
                    // deta's S-term of this block: sum over queries i >= j of dA_ij S_ij, per key j;
                    // this lane's products (i = g, g + 8; j = 8 nt + 2t, + 1), summed over g by shuffles
                    const float* S = reinterpret_cast<const float*>(smem + SC_OFF + (s * SPS + i) * SCSZ + 512);
                    float cs[2][2];
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt) {
                        const int j0 = 8 * nt + 2 * t;
                        const float2 s0 = *reinterpret_cast<const float2*>(S + g * 16 + j0);
                        const float2 s1 = *reinterpret_cast<const float2*>(S + (g + 8) * 16 + j0);
                        cs[nt][0] = (j0 <= g ? ds[nt][0] * s0.x : 0.f) + ds[nt][2] * s1.x;
                        cs[nt][1] = (j0 + 1 <= g ? ds[nt][1] * s0.y : 0.f) + ds[nt][3] * s1.y;
                        if (nt == 1) {  // keys 8..15: query rows 0..7 never reach them
                            cs[1][0] = (j0 <= g + 8 ? ds[1][2] * s1.x : 0.f);
                            cs[1][1] = (j0 + 1 <= g + 8 ? ds[1][3] * s1.y : 0.f);
                        }
                    }
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            float v = cs[nt][h];
                            v += __shfl_xor_sync(0xffffffffu, v, 4);
                            v += __shfl_xor_sync(0xffffffffu, v, 8);
                            v += __shfl_xor_sync(0xffffffffu, v, 16);
                            if (g == 0) dep[64 + 8 * nt + 2 * t + h] = v;
                        }
                }
                uint32_t dsa[4], dst[4];
                {
                    const float ej[4] = {es[2 * t], es[2 * t + 1], es[8 + 2 * t], es[9 + 2 * t]};
                    // (query i = g (+8), key j = 8 nt + 2t (+1)); keep j <= i
                    const float s00 = 2 * t <= g ? ds[0][0] * ej[0] : 0.f, s01 = 2 * t + 1 <= g ? ds[0][1] * ej[1] : 0.f;
                    const float s02 = ds[0][2] * ej[0], s03 = ds[0][3] * ej[1];
                    const float s12 = 2 * t <= g ? ds[1][2] * ej[2] : 0.f, s13 = 2 * t + 1 <= g ? ds[1][3] * ej[3] : 0.f;
                    dsa[0] = pack_bf16(s00, s01);
                    dsa[1] = pack_bf16(s02, s03);
                    dsa[2] = 0u;
                    dsa[3] = pack_bf16(s12, s13);
                    dst[0] = movt(dsa[0]);
                    dst[1] = movt(dsa[2]);
                    dst[2] = movt(dsa[1]);
                    dst[3] = movt(dsa[3]);
                }

                // ---- dQ rows [16r, 16r + 16) = dZ W^T + dS K;  dK = dE W^T - D (E dW'^T) + dS^T Q
                float q[2][4] = {}, k[2][4] = {}, y[2][4] = {};
                const uint32_t det = sbase + DE_OFF + (s * SPS + i) * TILE;
#pragma unroll
                for (int kc = 0; kc < KS; ++kc) {
                    uint32_t za[4], da_[4], ea[4], wt[4];
                    ldsm_x4(st + ZOFF + i * TILE + off_tk[kc], za);
                    ldsm_x4(det + off_tk[kc], da_);
                    ldsm_x4(sbase + ET_OFF + off_tk[kc], ea);
                    // W^T as B (K = column c, N = d_in 16r ..): plain loads of the rows d_in
                    ldsm_x4(wb + swz(16 * r + lr + 8 * (lj >> 1), 16 * kc + 8 * (lj & 1)), wt);
#pragma unroll
                    for (int nd = 0; nd < 2; ++nd) {
                        const uint32_t b0 = wt[2 * nd], b1 = wt[2 * nd + 1];
                        mma_bf16_16816(q[nd], za, b0, b1);
                        mma_bf16_16816(k[nd], da_, b0, b1);
                        // dW'^T as B from the replica (rows d_in, columns c)
                        const int hf = 2 * nd;
                        mma_bf16_16816(y[nd], ea, pack_bf16(rep[2 * kc][hf], rep[2 * kc][hf + 1]),
                                       pack_bf16(rep[2 * kc + 1][hf], rep[2 * kc + 1][hf + 1]));
                    }
                }
                {
                    uint32_t kb_[4], qb_[4];
                    ldsm_x4_trans(st + KOFF + i * TILE + off_tk[r], kb_);  // K as B (K = key j), d_in 16r ..
                    ldsm_x4_trans(st + QOFF + i * TILE + off_tk[r], qb_);  // Q as B (K = query i)
                    mma_bf16_16816(q[0], dsa, kb_[0], kb_[1]);
                    mma_bf16_16816(q[1], dsa, kb_[2], kb_[3]);
                    mma_bf16_16816(k[0], dst, qb_[0], qb_[1]);
                    mma_bf16_16816(k[1], dst, qb_[2], qb_[3]);
                }
                {
                    // dK -= D (E dW'^T); deta partial -sum_{d_in in slice} K_j,d_in (E dW'^T)_j,d_in
                    const float eg = es[g], eg8 = es[g + 8];
                    float pr0 = 0.f, pr1 = 0.f;
#pragma unroll
                    for (int nd = 0; nd < 2; ++nd) {
                        const int din = 16 * r + 8 * nd + 2 * t;
                        const float2 k0 = bf16x2_at(Kt_, g, din), k1 = bf16x2_at(Kt_, g + 8, din);
                        pr0 = fmaf(k0.x, y[nd][0], fmaf(k0.y, y[nd][1], pr0));
                        pr1 = fmaf(k1.x, y[nd][2], fmaf(k1.y, y[nd][3], pr1));
                        k[nd][0] = fmaf(-eg, y[nd][0], k[nd][0]);
                        k[nd][1] = fmaf(-eg, y[nd][1], k[nd][1]);
                        k[nd][2] = fmaf(-eg8, y[nd][2], k[nd][2]);
                        k[nd][3] = fmaf(-eg8, y[nd][3], k[nd][3]);
                    }
                    pr0 += __shfl_xor_sync(0xffffffffu, pr0, 1);
                    pr0 += __shfl_xor_sync(0xffffffffu, pr0, 2);
                    pr1 += __shfl_xor_sync(0xffffffffu, pr1, 1);
                    pr1 += __shfl_xor_sync(0xffffffffu, pr1, 2);
                    if (t == 0) {
                        dep[16 * r + g] = -pr0;
                        dep[16 * r + g + 8] = -pr1;
                    }
                }
                // ---- replica: dW rows [16r, 16r + 16) += Q^T dZ + K^T dE
                {
                    // A fragments of Q^T and K^T (rows d_in 16r .., K = token): transposed loads of the
                    // tiles (tokens 0-7, d_in lo), (tokens 0-7, d_in hi), (tokens 8-15, lo), (8-15, hi)
                    uint32_t qa[4], ka2[4];
                    ldsm_x4_trans(st + QOFF + i * TILE + swz(lr + 8 * (lj >> 1), 16 * r + 8 * (lj & 1)), qa);
                    ldsm_x4_trans(st + KOFF + i * TILE + swz(lr + 8 * (lj >> 1), 16 * r + 8 * (lj & 1)), ka2);
#pragma unroll
                    for (int cc = 0; cc < KS; ++cc) {
                        uint32_t zb[4], eb[4];
                        ldsm_x4_trans(st + ZOFF + i * TILE + off_tk[cc], zb);
                        ldsm_x4_trans(det + off_tk[cc], eb);
                        mma_bf16_16816(rep[2 * cc], qa, zb[0], zb[1]);
                        mma_bf16_16816(rep[2 * cc + 1], qa, zb[2], zb[3]);
                        mma_bf16_16816(rep[2 * cc], ka2, eb[0], eb[1]);
                        mma_bf16_16816(rep[2 * cc + 1], ka2, eb[2], eb[3]);
                    }
                }
                // ---- outputs of block sb: dQ, dK rows (tokens) x d_in [16r, 16r + 16), dV columns [16r, 16r + 16)
                {
                    const size_t row0 = bh * T + size_t(16) * sb;
                    const uint32_t sq = smem_u32(stg), sk = sq + 512;
                    stsm_x4(sq + (st_row * 32) + ((st_col >> 3) << 4), pack_bf16(q[0][0], q[0][1]),
                            pack_bf16(q[0][2], q[0][3]), pack_bf16(q[1][0], q[1][1]), pack_bf16(q[1][2], q[1][3]));
                    stsm_x4(sk + (st_row * 32) + ((st_col >> 3) << 4), pack_bf16(k[0][0], k[0][1]),
                            pack_bf16(k[0][2], k[0][3]), pack_bf16(k[1][0], k[1][1]), pack_bf16(k[1][2], k[1][3]));
                    __syncwarp();
                    const int orow = lane >> 1, ohalf = lane & 1;
                    const uint4 vq = *reinterpret_cast<const uint4*>(stg + orow * 32 + ohalf * 16);
                    const uint4 vk = *reinterpret_cast<const uint4*>(stg + 512 + orow * 32 + ohalf * 16);
                    const size_t o = (row0 + orow) * D + 16 * r + 8 * ohalf;
                    uint4 dv = *reinterpret_cast<const uint4*>(smem + DE_OFF + (s * SPS + i) * TILE +
                                                              swz(orow, 16 * r + 8 * ohalf));
                    dv.x ^= 0x80008000u; dv.y ^= 0x80008000u; dv.z ^= 0x80008000u; dv.w ^= 0x80008000u;
                    if (!PART || 16 * sb + orow < T) {  // rows past T are not stored
                        *reinterpret_cast<uint4*>(dQ + o) = vq;
                        *reinterpret_cast<uint4*>(dK + o) = vk;
                        *reinterpret_cast<uint4*>(dV + o) = dv;
                    }
                    __syncwarp();
                }
            }
            if (err) break;
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&empty_bar[s]));
        }
        // deta of the last block processed (block 0 of the sequence)
        if (!bar_readout_any(err) && p == nsb && r == 0 && lane < 16 && (!PART || lane < T))
            deta[bh * T + lane] = dep[64 + lane] + ((dep[lane] + dep[16 + lane]) + (dep[32 + lane] + dep[48 + lane]));
        cp_async_wait0();
    }
    __syncthreads();
}

template <bool PART>
cudaError_t launch_part(const LinearBwdArgs& a, cudaStream_t s, int* status) {
    const uint64_t heads = uint64_t(a.B) * a.H;
    CUtensorMap mq, mk, mv, mz;
    cudaError_t e;
    if (PART) {  // [heads][T][D]: the boxes of a partial block read zeros past T
        if ((e = make_tma_map_bf16_heads(&mq, a.Q, heads, a.T, D)) != cudaSuccess) return e;
        if ((e = make_tma_map_bf16_heads(&mk, a.K, heads, a.T, D)) != cudaSuccess) return e;
        if ((e = make_tma_map_bf16_heads(&mv, a.V, heads, a.T, D)) != cudaSuccess) return e;
        if ((e = make_tma_map_bf16_heads(&mz, a.dZ, heads, a.T, D)) != cudaSuccess) return e;
    } else {  // [heads * T][D]
        if ((e = make_tma_map_bf16(&mq, a.Q, heads * a.T, D)) != cudaSuccess) return e;
        if ((e = make_tma_map_bf16(&mk, a.K, heads * a.T, D)) != cudaSuccess) return e;
        if ((e = make_tma_map_bf16(&mv, a.V, heads * a.T, D)) != cudaSuccess) return e;
        if ((e = make_tma_map_bf16(&mz, a.dZ, heads * a.T, D)) != cudaSuccess) return e;
    }
    const int bytes = BYTES + 1024;
    auto kern = linear_backward_mma_kernel<PART>;
    if ((e = allow_dynamic_smem(reinterpret_cast<const void*>(kern), bytes)) != cudaSuccess) return e;
    kern<<<unsigned(a.B) * unsigned(a.H), THREADS, bytes, s>>>(
        mq, mk, mv, mz, a.eta, static_cast<const __nv_bfloat16*>(a.W_hist), a.dW_T, static_cast<__nv_bfloat16*>(a.dQ), static_cast<__nv_bfloat16*>(a.dK),
        static_cast<__nv_bfloat16*>(a.dV), a.deta, a.dW0, a.T, status);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_linear_backward_mma(const LinearBwdArgs& a, cudaStream_t s, int* status) {
    // any T: a partial last block weighs its tokens past T by zero
    if (!a.bf16 || a.d != D || a.chunk != 16) return cudaErrorNotSupported;
    if (uint64_t(a.B) * a.H > 0x7fffffffull) return cudaErrorNotSupported;  // TMA head coordinate is int32
    // the 2D maps address rows bh * T + t with an int32 coordinate
    if (a.T % 16 || uint64_t(a.B) * a.H * a.T > 0x7fffffffull) return launch_part<true>(a, s, status);
    return launch_part<false>(a, s, status);
}

}  // namespace ttt
