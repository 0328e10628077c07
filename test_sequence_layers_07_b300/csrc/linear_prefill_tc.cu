// linear_prefill_tc.cu -- TTT-Linear prefill at d = 64 (bf16 Q/K/V/Z, fp32 state): the
// recurrence on warp-level MMAs, the read-out on the 5th-generation tensor cores.
//
// What is computed ("Test-Time Training Layers ...", sections "The Core Mechanism" and
// "Hardware Parallelization"; TTT essay, paragraph on the dual form): per block of b tokens
// with start state W0,
//     E = K W0 - V;  Z = Q W0 - tril(eta . Q K^T) E;  W = W0 - K^T diag(eta) E.
//
// Design (ours, for sm_103a):
//  * Recurrence.  Per 16-token sub-block, with W_b the state at the start of its block:
//    G = -eta . (K W_b - V) and W += K^T G.  A chain of small dependent products, bound by
//    latency: four warps, one per 16-column group, keep W^T in registers in the accumulator
//    layout of the m16n8k16 bf16 MMA (which after an fp32 -> bf16 pack is the A-operand
//    layout), as in the all-warp-MMA kernel.  Each chain warp exports its G rows (and, at
//    every 128-token stage boundary, the bf16 state) to shared memory by stmatrix.
//  * Read-out.  Z does not need the state after every sub-block.  Over a stage of 128
//    tokens with start state W_s, the state before query row q is W_s plus K_j^T G_j over
//    the earlier sub-blocks j, and the sub-block's own term is tril(Q K^T) G; together
//        Z = Q W_s + causal(Q K^T) G       (causal: key k <= query q inside the stage),
//    which is the dual form applied to the stage with the chain's G in place of -eta E.
//    Three dense products per stage run on tcgen05 with fp32 accumulators in TMEM:
//        [S | Z] = Q [K ; W_s^T]^T            M = 128 tokens, N = 128 + 64, K = 64
//        P = bf16(causal(S))  written over S  (epilogue warps, TMEM -> registers -> TMEM)
//        Z += P G                             A = P from TMEM, M = 128, N = 64, K = 128
//    This takes the read-out and the masked scores off the warp-level MMA pipes and the
//    shared-memory load path that the chain warps need.
//  * Warps: 0 TMA producer; 1 issues the [S | Z] product (and owns TMEM); 2..5 the chain;
//    6..9 the epilogue (warp w reads TMEM lanes 32 (w % 4) ..); 10 issues Z += P G.
//    Stage ring of NST slots [Q | K | W_s^T | V | eta]; K and W_s^T are adjacent so that
//    one N = 192 operand covers both.  TMEM: two buffers of 192 columns [S/P | Z].
//  * All waits are bounded; on expiry the kernel records TTT_ERR_TIMEOUT, every role
//    leaves its loop, the producer drains its copies and the issuers wait for their own
//    MMAs before TMEM is released.
#include <cuda.h>

#include "ptx.cuh"
#include "tc.cuh"
#include "ttt_common.cuh"
#include "ttt_internal.h"

namespace ttt {
namespace {

using namespace ptx;

constexpr uint64_t kWaitLimitNs = 4000000000ull;  // 4 s: far beyond any legitimate wait

constexpr int D = 64;
constexpr int CG = 4;     // 16-column groups (chain warps)
constexpr int SPS = 8;    // 16-token sub-blocks per stage
constexpr int BT = 128;   // tokens per stage (the M of the read-out products)
constexpr int NST = 3;    // stage slots
constexpr int KS = D / 16, NT = D / 8;
constexpr int TILE = 16 * D * 2;  // one 16-token [16][64] bf16 sub-tile (one TMA box)
// slot layout (bytes); every operand block 1024-byte aligned
constexpr int QOFF = 0, KOFF = SPS * TILE, WSOFF = 2 * SPS * TILE, VOFF = WSOFF + D * D * 2;
constexpr int EOFF = VOFF + SPS * TILE;
constexpr int STAGE = (EOFF + SPS * 64 + 1023) / 1024 * 1024;
constexpr int GT_OFF = NST * STAGE;  // G^T per slot: [64 columns][128 tokens] bf16 = two SW128 blocks
constexpr int GT_BLK = D * 128;      // one [64][64] bf16 block
constexpr int GT_BYTES = 2 * GT_BLK;
constexpr int BYTES = GT_OFF + NST * GT_BYTES;
// xf barriers per stage index modulo NXF: the [S | Z] issuer waits on the one of the previous
// stage, and the chain's arrive for the last stage does not wait for a refill, so with NST
// barriers one could complete twice before that wait; with 2 NST it cannot.
constexpr int NXF = 2 * NST;
constexpr int NWARPS = 11;
constexpr int THREADS = 32 * NWARPS;
constexpr int TM_COLS = 512;
constexpr int TM_BUF = 192;  // per buffer: S/P columns 0..127, Z columns 128..191
static_assert(BYTES + 1024 <= 232448, "shared memory");

constexpr uint32_t IDESC_SZ = tc::make_idesc(128, 192, 0, 0);  // [S | Z] = Q [K ; W_s^T]^T
constexpr uint32_t IDESC_PG = tc::make_idesc(128, 64, 0, 0);   // Z += P G

// byte offset of (row, col) in a [rows][64] bf16 SW128 block, col % 8 == 0
__device__ __forceinline__ uint32_t swz(int row, int col) {
    return uint32_t((col >> 6) * 2048 + row * 128 + ((((col & 63) >> 3) ^ (row & 7)) << 4));
}

__device__ __forceinline__ void pack_state(const float (&w)[NT][4], uint32_t (&wa)[KS][4]) {
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
        wa[ks][0] = pack_bf16(w[2 * ks][0], w[2 * ks][1]);
        wa[ks][1] = pack_bf16(w[2 * ks][2], w[2 * ks][3]);
        wa[ks][2] = pack_bf16(w[2 * ks + 1][0], w[2 * ks + 1][1]);
        wa[ks][3] = pack_bf16(w[2 * ks + 1][2], w[2 * ks + 1][3]);
    }
}

template <bool SINGLE>
__global__ void __launch_bounds__(THREADS, 1)
linear_prefill_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const float* __restrict__ eta,
                         const float* W0, __nv_bfloat16* __restrict__ Z, float* W_out, int T, int chunk,
                         int* status) {
    extern __shared__ uint8_t smem_dyn[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
    __shared__ __align__(8) uint64_t full_bar[NST];   // TMA data of a slot landed
    __shared__ __align__(8) uint64_t empty_bar[NST];  // every read of a slot done (Z += P G committed)
    __shared__ __align__(8) uint64_t xf_bar[NXF];     // chain: G of the stage and W_s of the next written
    __shared__ __align__(8) uint64_t s_bar[2];        // [S | Z] product of a TMEM buffer committed
    __shared__ __align__(8) uint64_t p_bar[2];        // epilogue wrote P into a TMEM buffer
    __shared__ __align__(8) uint64_t z_bar[2];        // Z += P G of a TMEM buffer committed
    __shared__ __align__(8) uint64_t zr_bar[2];       // epilogue read Z of a TMEM buffer
    __shared__ uint32_t s_tmem;
    __shared__ volatile int s_err;
    __shared__ volatile int s_zero;  // never set: abort flag of the waits that must run to completion

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const size_t bh = blockIdx.x;
    const int nsb = T / 16;                  // 16-token sub-blocks
    const int nstg = (nsb + SPS - 1) / SPS;  // stages
    const int nsub = chunk / 16;             // sub-blocks per block
    const uint32_t sbase = smem_u32(smem);
    const int g = lane >> 2, t = lane & 3;
    const int lj = lane >> 3, lr = lane & 7;
    auto slot = [&](int si) { return sbase + uint32_t((si % NST) * STAGE); };
    auto gt_slot = [&](int si) { return sbase + uint32_t(GT_OFF + (si % NST) * GT_BYTES); };
    auto subs_in = [&](int si) { return nsb - si * SPS < SPS ? nsb - si * SPS : SPS; };

    if (threadIdx.x == 0) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(smem_u32(&full_bar[s]), 1);
            mbar_init(smem_u32(&empty_bar[s]), 1);
        }
        for (int j = 0; j < NXF; ++j) mbar_init(smem_u32(&xf_bar[j]), CG);
        for (int x = 0; x < 2; ++x) {
            mbar_init(smem_u32(&s_bar[x]), 1);
            mbar_init(smem_u32(&p_bar[x]), 4);
            mbar_init(smem_u32(&z_bar[x]), 1);
            mbar_init(smem_u32(&zr_bar[x]), 4);
        }
        s_err = 0;
        s_zero = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(smem_u32(&s_tmem), TM_COLS);
        tc::tmem_relinquish();
    }
    // G^T slots start at zero: in a short last stage the rows past the last sub-block meet
    // only exact zeros of P, and must not hold NaN bit patterns
    for (int i = threadIdx.x; i < NST * GT_BYTES / 16; i += THREADS)
        *reinterpret_cast<uint4*>(smem + GT_OFF + 16 * i) = make_uint4(0, 0, 0, 0);

    // chain warps: initial state into registers and, as bf16 W_s^T, into slot 0
    const bool chain = warp >= 2 && warp < 2 + CG;
    const int cg = warp - 2;
    const int cw0 = 16 * cg;  // first output column of this group
    float w[NT][4];           // W^T[c][d_in], c = g (+8), d_in = 8*nt + 2t (+1)
    // lane l's stmatrix row address: row (l & 7) + 8 ((l >> 3) & 1), column 8 (l >> 4) of a 16 x 16 tile
    const int st_row = cw0 + lr + 8 * (lj & 1), st_col = 8 * (lj >> 1);
    auto store_ws = [&](uint32_t st) {
        uint32_t wa[KS][4];
        pack_state(w, wa);
#pragma unroll
        for (int ks = 0; ks < KS; ++ks)
            stsm_x4(st + WSOFF + swz(st_row, 16 * ks + st_col), wa[ks][0], wa[ks][1], wa[ks][2], wa[ks][3]);
    };
    if (chain) {
        const float* W0h = W0 + bh * D * D;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int r = 8 * nt + 2 * t;
            w[nt][0] = W0h[size_t(r) * D + cw0 + g];
            w[nt][1] = W0h[size_t(r + 1) * D + cw0 + g];
            w[nt][2] = W0h[size_t(r) * D + cw0 + g + 8];
            w[nt][3] = W0h[size_t(r + 1) * D + cw0 + g + 8];
        }
        store_ws(sbase);
    }
    fence_proxy_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tm = s_tmem;

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

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            prefetch_tensormap(&tmQ);
            prefetch_tensormap(&tmK);
            prefetch_tensormap(&tmV);
            int issued = 0;
            for (int si = 0; si < nstg; ++si) {
                const int s = si % NST, n = subs_in(si);
                if (si >= NST && !wait(empty_bar[s], ((si / NST) - 1) & 1)) break;
                const uint32_t fb = smem_u32(&full_bar[s]);
                mbar_arrive_expect_tx(fb, uint32_t(n) * (3 * TILE + 64));
                const uint32_t st = slot(si);
                for (int i = 0; i < n; ++i) {
                    const int y = int(bh * T) + 16 * (si * SPS + i);
                    tma_load_2d(st + QOFF + i * TILE, &tmQ, 0, y, fb);
                    tma_load_2d(st + KOFF + i * TILE, &tmK, 0, y, fb);
                    tma_load_2d(st + VOFF + i * TILE, &tmV, 0, y, fb);
                }
                bulk_load(st + EOFF, eta + bh * T + 16 * si * SPS, uint32_t(n) * 64, fb);
                ++issued;
            }
            // never retire the CTA with copies in flight (this wait ignores the abort flag)
            for (int si = issued > NST ? issued - NST : 0; si < issued; ++si)
                mbar_wait_bounded(smem_u32(&full_bar[si % NST]), (si / NST) & 1, &s_zero, kWaitLimitNs);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ [S | Z] = Q [K ; W_s^T]^T
        if (lane == 0) {
            int last = -1;
            for (int si = 0; si < nstg; ++si) {
                const int s = si % NST, x = si & 1;
                if (!wait(full_bar[s], (si / NST) & 1)) break;
                if (si >= 1 && !wait(xf_bar[(si - 1) % NXF], ((si - 1) / NXF) & 1)) break;  // W_s of this stage
                if (si >= 2 && !wait(zr_bar[x], ((si - 2) >> 1) & 1)) break;  // buffer x drained
                tc::fence_after_sync();
                const uint32_t st = slot(si);
#pragma unroll
                for (int kk = 0; kk < KS; ++kk) {
                    const uint64_t ad = tc::make_desc(st + QOFF + 32 * kk, 16, 1024, tc::kSwizzle128B);
                    const uint64_t bd = tc::make_desc(st + KOFF + 32 * kk, 16, 1024, tc::kSwizzle128B);
                    tc::mma(tm + x * TM_BUF, ad, bd, IDESC_SZ, kk > 0);
                }
                tc::commit(smem_u32(&s_bar[x]));
                last = si;
            }
            // TMEM is released after this CTA's MMAs completed
            if (last >= 0)
                mbar_wait_bounded(smem_u32(&s_bar[last & 1]), (last >> 1) & 1, &s_zero, kWaitLimitNs);
        }
    } else if (warp == NWARPS - 1) {
        // ------------------------------------------------------------ Z += P G
        if (lane == 0) {
            int last = -1;
            for (int si = 0; si < nstg; ++si) {
                const int s = si % NST, x = si & 1;
                if (!wait(xf_bar[si % NXF], (si / NXF) & 1) || !wait(p_bar[x], (si >> 1) & 1)) break;
                tc::fence_after_sync();
                const uint32_t gt = gt_slot(si);
                const uint32_t buf = tm + x * TM_BUF;
#pragma unroll
                for (int kk = 0; kk < BT / 16; ++kk) {
                    const uint64_t bd =
                        tc::make_desc(gt + (kk >> 2) * GT_BLK + 32 * (kk & 3), 16, 1024, tc::kSwizzle128B);
                    tc::mma_ts(buf + 128, buf + 8 * kk, bd, IDESC_PG, 1);
                }
                tc::commit(smem_u32(&z_bar[x]));
                tc::commit(smem_u32(&empty_bar[s]));
                last = si;
            }
            if (last >= 0)
                mbar_wait_bounded(smem_u32(&z_bar[last & 1]), (last >> 1) & 1, &s_zero, kWaitLimitNs);
        }
    } else if (chain) {
        // ------------------------------------------------------------ recurrence
        // P = K W_b, G = -eta (P - V), W += K^T G.  Per stage one wait (the next stage's data)
        // and one arrive; the fragments of the next sub-block load while this one computes.
        const uint32_t off_v = swz(lr + 8 * (lj >> 1), cw0 + 8 * (lj & 1));
        uint32_t off_nk[KS], off_tk[NT / 2];
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) off_nk[ks] = swz(lr + 8 * (lj >> 1), 16 * ks + 8 * (lj & 1));
#pragma unroll
        for (int kk = 0; kk < NT / 2; ++kk) off_tk[kk] = swz(lr + 8 * (lj & 1), 16 * kk + 8 * (lj >> 1));
        uint32_t wa0[KS][4];
        uint32_t kb[KS][4], kt[NT / 2][4];
        float ne0 = 0, ne1 = 0, ne2 = 0, ne3 = 0, nv[8] = {};
        auto load = [&](uint32_t st, int i) {
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) ldsm_x4(st + KOFF + i * TILE + off_nk[ks], kb[ks]);
#pragma unroll
            for (int kk = 0; kk < NT / 2; ++kk) ldsm_x4_trans(st + KOFF + i * TILE + off_tk[kk], kt[kk]);
            uint32_t vv[4];
            ldsm_x4_trans(st + VOFF + i * TILE + off_v, vv);
            const float* es = reinterpret_cast<const float*>(smem + (st - sbase) + EOFF + i * 64);
            const float2 e01 = *reinterpret_cast<const float2*>(es + 2 * t);
            const float2 e23 = *reinterpret_cast<const float2*>(es + 8 + 2 * t);
            ne0 = -e01.x; ne1 = -e01.y; ne2 = -e23.x; ne3 = -e23.y;
            nv[0] = e01.x * bf16_lo(vv[0]); nv[1] = e01.y * bf16_hi(vv[0]);
            nv[2] = e01.x * bf16_lo(vv[1]); nv[3] = e01.y * bf16_hi(vv[1]);
            nv[4] = e23.x * bf16_lo(vv[2]); nv[5] = e23.y * bf16_hi(vv[2]);
            nv[6] = e23.x * bf16_lo(vv[3]); nv[7] = e23.y * bf16_hi(vv[3]);
        };
        bool ok = wait_all(full_bar[0], 0);
        if (ok) load(sbase, 0);
        for (int si = 0; ok && si < nstg; ++si) {
            const int n = subs_in(si);
            const uint32_t st = slot(si), gt = gt_slot(si);
            auto step = [&](int i) {
                const int sb = si * SPS + i;
                if (SINGLE || sb % nsub == 0) pack_state(w, wa0);
                float pa[4][2][4] = {};
#pragma unroll
                for (int ks = 0; ks < KS; ++ks) {
                    mma_bf16_16816(pa[ks & 3][0], wa0[ks], kb[ks][0], kb[ks][1]);
                    mma_bf16_16816(pa[ks & 3][1], wa0[ks], kb[ks][2], kb[ks][3]);
                }
                float p[2][4];
#pragma unroll
                for (int j = 0; j < 2; ++j)
#pragma unroll
                    for (int k = 0; k < 4; ++k) p[j][k] = (pa[0][j][k] + pa[1][j][k]) + (pa[2][j][k] + pa[3][j][k]);
                // G = -eta . (P - V)^T as a bf16 A operand (rows c, cols token j)
                uint32_t ga[4];
                ga[0] = pack_bf16(fmaf(ne0, p[0][0], nv[0]), fmaf(ne1, p[0][1], nv[1]));
                ga[1] = pack_bf16(fmaf(ne0, p[0][2], nv[2]), fmaf(ne1, p[0][3], nv[3]));
                ga[2] = pack_bf16(fmaf(ne2, p[1][0], nv[4]), fmaf(ne3, p[1][1], nv[5]));
                ga[3] = pack_bf16(fmaf(ne2, p[1][2], nv[6]), fmaf(ne3, p[1][3], nv[7]));
                // W^T += G K   (rank-16 update of the running state, fp32 accumulate)
#pragma unroll
                for (int kk = 0; kk < NT / 2; ++kk) {
                    mma_bf16_16816(w[2 * kk], ga, kt[kk][0], kt[kk][1]);
                    mma_bf16_16816(w[2 * kk + 1], ga, kt[kk][2], kt[kk][3]);
                }
                // G^T rows of this group, tokens 16 i .. 16 i + 15 of the stage
                const int tok = 16 * i + st_col;
                stsm_x4(gt + (tok >> 6) * GT_BLK + swz(st_row, tok & 63), ga[0], ga[1], ga[2], ga[3]);
            };
            if (n == SPS) {  // full stage: unrolled, so the compiler schedules across sub-blocks
#pragma unroll
                for (int i = 0; i < SPS; ++i) {
                    step(i);
                    if (i + 1 < SPS) load(st, i + 1);
                }
            } else {
                for (int i = 0; i < n; ++i) {
                    step(i);
                    if (i + 1 < n) load(st, i + 1);
                }
            }
            if (si + 1 < nstg) {
                // the next slot is filled (so its previous stage is fully consumed): load its first
                // fragments and publish its start state
                ok = wait_all(full_bar[(si + 1) % NST], ((si + 1) / NST) & 1);
                if (ok) {
                    load(slot(si + 1), 0);
                    store_ws(slot(si + 1));
                }
            }
            fence_proxy_async_smem();  // stmatrix writes -> tensor-core reads
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&xf_bar[si % NXF]));
        }
        float* Wo = W_out + bh * D * D;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int r = 8 * nt + 2 * t;
            Wo[size_t(r) * D + cw0 + g] = w[nt][0];
            Wo[size_t(r + 1) * D + cw0 + g] = w[nt][1];
            Wo[size_t(r) * D + cw0 + g + 8] = w[nt][2];
            Wo[size_t(r + 1) * D + cw0 + g + 8] = w[nt][3];
        }
    } else {
        // ------------------------------------------------------------ epilogue (warps 6..9)
        const int qd = warp & 3;      // TMEM lane quadrant of this warp
        const int row = 32 * qd + lane;  // token row of the stage
        const uint32_t tl = tm + (uint32_t(32 * qd) << 16);
        for (int si = 0; si < nstg; ++si) {
            const int x = si & 1;
            const uint32_t buf = tl + x * TM_BUF;
            if (!wait_all(s_bar[x], (si >> 1) & 1)) break;
            tc::fence_after_sync();
            // P = bf16(S) with key k > query row zeroed, written over the S columns already read
#pragma unroll
            for (int c = 0; c < BT / 16; ++c) {
                uint32_t pk[8];
                if (16 * c > 32 * qd + 31) {
#pragma unroll
                    for (int j = 0; j < 8; ++j) pk[j] = 0u;
                } else {
                    float v[16];
                    tc::ld16(buf + 16 * c, v);
                    tc::ld_wait();
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        if (16 * c + j > row) v[j] = 0.f;
#pragma unroll
                    for (int j = 0; j < 8; ++j) pk[j] = pack_bf16(v[2 * j], v[2 * j + 1]);
                }
                tc::st8u(buf + 8 * c, pk);
            }
            tc::st_wait();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&p_bar[x]));

            if (!wait_all(z_bar[x], (si >> 1) & 1)) break;
            tc::fence_after_sync();
            float z[64];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                float v[16];
                tc::ld16(buf + 128 + 16 * c, v);
#pragma unroll
                for (int j = 0; j < 16; ++j) z[16 * c + j] = v[j];
            }
            tc::ld_wait();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&zr_bar[x]));
            if (row < 16 * subs_in(si)) {
                uint4* zp = reinterpret_cast<uint4*>(Z + (bh * T + size_t(si) * BT + row) * D);
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    zp[c] = make_uint4(pack_bf16(z[8 * c], z[8 * c + 1]), pack_bf16(z[8 * c + 2], z[8 * c + 3]),
                                       pack_bf16(z[8 * c + 4], z[8 * c + 5]), pack_bf16(z[8 * c + 6], z[8 * c + 7]));
            }
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tm, TM_COLS);
    }
}

template <bool SINGLE>
cudaError_t launch_kernel(const LinearArgs& a, cudaStream_t s, int* status) {
    const uint64_t rows = uint64_t(a.B) * a.H * a.T;
    CUtensorMap mq, mk, mv;
    cudaError_t e;
    if ((e = make_tma_map_bf16(&mq, a.Q, rows, D)) != cudaSuccess) return e;
    if ((e = make_tma_map_bf16(&mk, a.K, rows, D)) != cudaSuccess) return e;
    if ((e = make_tma_map_bf16(&mv, a.V, rows, D)) != cudaSuccess) return e;
    auto kern = linear_prefill_tc_kernel<SINGLE>;
    const int bytes = BYTES + 1024;  // + alignment slack
    if ((e = allow_dynamic_smem(reinterpret_cast<const void*>(kern), bytes)) != cudaSuccess) return e;
    kern<<<unsigned(a.B) * unsigned(a.H), THREADS, bytes, s>>>(mq, mk, mv, a.eta, a.W0,
                                                              static_cast<__nv_bfloat16*>(a.Z), a.W_out, a.T,
                                                              a.chunk, status);
    return cudaGetLastError();
}

}  // namespace

bool linear_prefill_tc_supported(const LinearArgs& a) {
    return a.bf16 && a.d == D && a.chunk % 16 == 0 && a.T % a.chunk == 0 &&
           uint64_t(a.B) * a.H * a.T <= 0x7fffffffull;  // TMA row coordinate is int32
}

// Measured on B300 at B=8 H=12 T=2048: this kernel and the split warp-MMA kernel tie at chunk 16
// (49.7 vs 49.6 us); at chunk 64 this one is faster (53.6 vs 58.9 us), at chunk 512 slower
// (53.5 vs 50.6 us).  Both are bound by the chain warps, which share the SM's tensor cores and
// shared-memory path with the read-out, in either form; the one-warp-per-group kernel
// (linear_prefill_fused.cu) beats both at every chunk, so this one runs only on request.
cudaError_t launch_linear_prefill_tc(const LinearArgs& a, cudaStream_t s, int* status) {
    if (!linear_prefill_tc_supported(a)) return cudaErrorNotSupported;
    return a.chunk == 16 ? launch_kernel<true>(a, s, status) : launch_kernel<false>(a, s, status);
}

}  // namespace ttt
