// linear_prefill_fused.cu -- TTT-Linear prefill, bf16 Q/K/V/Z, fp32 state, d = 64: one warp per
// 16-column group runs the recurrence and the read-out together.
//
// What is computed ("Test-Time Training Layers ...", sections "The Core Mechanism" and
// "Hardware Parallelization"; TTT essay, paragraph on the dual form): per block of b tokens with
// start state W0,
//     E = K W0 - V;  Z = Q W0 - tril(eta . Q K^T) E;  W = W0 - K^T diag(eta) E.
//
// Design (ours, for sm_103a):
//  * Output columns are independent for f = kW, so a head splits into d/16 column groups with no
//    communication.  Each group is ONE warp holding its slice of the running state transposed
//    (W^T, 16 columns x d, fp32) in the accumulator layout of the warp-level m16n8k16 bf16 MMA.
//    After an fp32 -> bf16 pack that layout serves three products without any data movement:
//      - as the A operand of P^T = W^T K^T (the error at the block-start state),
//      - as the B operand of Q W (the read-out), since the accumulator fragment of W^T is the
//        B fragment of W contracted over d,
//      - and the rank-16 update W^T += G K with G = -eta . (K W - V)^T is accumulated straight
//        into it in fp32.
//    G itself, packed as the A operand of that update, is also the B operand of the read-out's
//    correction S G^T (S the masked scores), so the error never leaves the registers either.
//  * Measured on B300: with the same operands in every instruction a warp-level m16n8k16 issues at
//    one per ~8.1 cycles per warp (~2.0 cycles per SM from four warps on); with operands that change
//    every instruction, as here, an SM gets through one per ~6 cycles however many warps share it,
//    so the MMAs per SM bound the time.  Per 16-token
//    sub-block a warp issues 26: 8 for K W, 8 for the update, 8 for Q W and 2 for the correction;
//    the masked scores tril(Q K^T) (8 MMAs per sub-block, the same for every column group) are
//    computed once per CTA: at the start of a stage each warp forms those of every CG-th
//    sub-block and leaves them in shared memory (MMA-fragment order) behind an mbarrier.  There
//    is no second copy of the state and no exchange of G through shared memory.
//  * The recurrence (pack, K W, G, update) is the latency-critical chain; Q W is issued right
//    after K W so the tensor pipe is busy while the chain waits for P, and the Z of a sub-block
//    is stored during the next one (a store waits for its data, so storing at once would stall
//    the chain).  The fragments of sub-block i + 1 (K as both B layouts, Q as A, V, eta) are
//    loaded while sub-block i runs, into a second register set.
//  * A block of b = 16 * nsub tokens runs as nsub sub-blocks: E of every sub-block uses the
//    block-start state (a bf16 copy in registers), the read-out uses the running state, which
//    equals Z = Q W0 - tril(eta . Q K^T) E without forming the b x b matrix.
//  * Warp 0 streams Q/K/V by TMA (16-token boxes, 128-byte swizzle: conflict-free ldmatrix) and
//    eta by a bulk copy into an NST-stage mbarrier ring of SPS sub-blocks per stage.  Each mbarrier
//    wait costs a warp ~230 cycles even when the phase has completed, hence the large stages
//    (two waits per stage and warp: data landed, scores written).
//  * All waits are bounded (by `wait_ns`, normally 4 s); on expiry the kernel records
//    TTT_ERR_TIMEOUT, every warp leaves its loop, and the producer drains its copies (with the
//    4 s bound, whatever `wait_ns` is) before the CTA exits.
#include <cuda.h>
#include <string.h>

#include "ptx.cuh"
#include "ttt_common.cuh"
#include "ttt_internal.h"

namespace ttt {
namespace {

using namespace ptx;

constexpr uint64_t kWaitLimitNs = 4000000000ull;  // 4 s: far beyond any legitimate wait

// byte offset of (row, col) in a [16][D] bf16 tile stored as D/64 TMA boxes of [16][64] with the
// 128-byte swizzle (16-byte chunk index XOR row % 8); col % 8 == 0
__device__ __forceinline__ uint32_t swz(int row, int col) {
    return uint32_t((col >> 6) * 2048 + row * 128 + ((((col & 63) >> 3) ^ (row & 7)) << 4));
}

template <int KS>
__device__ __forceinline__ void pack_state(const float (&w)[2 * KS][4], uint32_t (&wa)[KS][4]) {
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
        wa[ks][0] = pack_bf16(w[2 * ks][0], w[2 * ks][1]);
        wa[ks][1] = pack_bf16(w[2 * ks][2], w[2 * ks][3]);
        wa[ks][2] = pack_bf16(w[2 * ks + 1][0], w[2 * ks + 1][1]);
        wa[ks][3] = pack_bf16(w[2 * ks + 1][2], w[2 * ks + 1][3]);
    }
}

template <int D, int CG, int NST, int SPS, bool HIST = false>
struct FusedCfg {
    static constexpr int KS = D / 16;        // k-steps over the input dimension
    static constexpr int NT = D / 8;         // 8-wide n-tiles of the state over the input dimension
    static constexpr int TILE = 16 * D * 2;  // bytes of one 16-token [16][D] bf16 sub-tile
    // a stage holds SPS sub-blocks: Q sub-tiles, then K, then V, then eta
    static constexpr int QOFF = 0, KOFF = SPS * TILE, VOFF = 2 * SPS * TILE, EOFF = 3 * SPS * TILE;
    static constexpr int STAGE = (EOFF + SPS * 64 + 1023) / 1024 * 1024;
    // masked scores [NST][SPS]: 32 lanes x 16 B; with the recorded states, the three registers of the
    // fragment that can be nonzero, word-major ([3][32 lanes] x 4 B), to make room for a second slice
    static constexpr int SCB = HIST ? 384 : 512;
    static constexpr int SC_OFF = NST * STAGE;
    static constexpr int HS_OFF = SC_OFF + NST * SPS * SCB;  // per warp: [D][16] bf16 state slices (two with HIST)
    static constexpr int BYTES = HS_OFF + CG * D * (HIST ? 64 : 32);
    static constexpr int THREADS = 32 * (CG + 1);
};

// HIST: also write the state at the start of every block to W_hist [B*H][ceil(T/16)][D][D], as bf16
// (the operand the products use, and what the backward reads); instantiated for blocks of 16
// tokens only.
// PART: T is not a multiple of 16 (a partial last sub-block), or the rows of all heads exceed the int32
// coordinate of a 2D tensor map.  Then Q/K/V come through per-head 3D maps (tokens past a head's end
// read as zeros), eta by cp.async where a bulk copy cannot take it, and the rows of Z past T are not
// stored; the instantiation for the common case compiles none of that.
template <int D, int CG, int NST, int SPS, bool SINGLE, bool HIST, bool PART>
__global__ void __launch_bounds__(FusedCfg<D, CG, NST, SPS, HIST>::THREADS, 1)
linear_prefill_fused_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                            const __grid_constant__ CUtensorMap tmV, const float* __restrict__ eta,
                            const float* W0, __nv_bfloat16* __restrict__ Z, float* W_out, int T, int chunk,
                            int* status, const __grid_constant__ CUtensorMap tmH, uint64_t wait_ns) {
    using C = FusedCfg<D, CG, NST, SPS, HIST>;
    constexpr int KS = C::KS, NT = C::NT;

    extern __shared__ uint8_t smem_dyn[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
    __shared__ __align__(8) uint64_t full_bar[NST];
    __shared__ __align__(8) uint64_t empty_bar[NST];
    __shared__ __align__(8) uint64_t sc_bar[NST];  // the stage's masked scores are written
    __shared__ volatile int s_err;
    __shared__ volatile int s_zero;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const size_t bh = blockIdx.x;
    const int nsb = PART ? (T + 15) / 16 : T / 16;  // 16-token sub-blocks (with PART the last may be partial)
    const int nstg = (nsb + SPS - 1) / SPS;  // stages
    const int nsub = chunk / 16;             // sub-blocks per block
    const bool ebulk = (T & 3) == 0;         // a head's eta starts 16-byte aligned (PART)
    const uint32_t sbase = smem_u32(smem);
    const int g = lane >> 2, t = lane & 3;
    const int lj = lane >> 3, lr = lane & 7;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(smem_u32(&full_bar[s]), 1);
            mbar_init(smem_u32(&empty_bar[s]), CG);
            mbar_init(smem_u32(&sc_bar[s]), CG);
        }
        s_err = 0;
        s_zero = 0;
        fence_mbar_init();
    }
    __syncthreads();

    auto wait = [&](uint64_t& bar, uint32_t parity) -> bool {
        if (s_err || !mbar_wait_bounded(smem_u32(&bar), parity, &s_err, wait_ns)) {
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
    auto subs_in = [&](int si) { return nsb - si * SPS < SPS ? nsb - si * SPS : SPS; };

    if (warp == 0) {
        // ---------------------------------------------------------------- TMA producer
        if (lane == 0) {
            prefetch_tensormap(&tmQ);
            prefetch_tensormap(&tmK);
            prefetch_tensormap(&tmV);
            int issued = 0;
            for (int si = 0; si < nstg; ++si) {
                const int s = si % NST, n = subs_in(si);
                if (si >= NST && !wait(empty_bar[s], ((si / NST) - 1) & 1)) break;
                const uint32_t fb = smem_u32(&full_bar[s]);
                const uint32_t st = sbase + s * C::STAGE;
                if constexpr (PART) {
                    // eta: one bulk copy when every token of the stage exists and a head's eta starts
                    // on a 16-byte boundary (4 | T); otherwise 4-byte cp.async copies that the
                    // stage's mbarrier tracks, and zeros past T
                    const int tok = min(16 * n, T - 16 * si * SPS);
                    const bool eb = ebulk && tok == 16 * n;
                    if (!eb) {
                        const float* eg = eta + bh * T + 16 * si * SPS;
                        float* es = reinterpret_cast<float*>(smem + s * C::STAGE + C::EOFF);
                        for (int j = 0; j < 16 * n; ++j) {
                            if (j < tok) cp_async4(st + C::EOFF + 4 * j, eg + j);
                            else es[j] = 0.f;
                        }
                        cp_async_mbar_arrive(fb);  // before this thread's own arrive on the phase
                    }
                    mbar_arrive_expect_tx(fb, uint32_t(n) * 3 * C::TILE + (eb ? uint32_t(n) * 64 : 0u));
                    for (int i = 0; i < n; ++i) {
                        const int y = 16 * (si * SPS + i), z = int(bh);
#pragma unroll
                        for (int box = 0; box < D / 64; ++box) {
                            tma_load_3d(st + C::QOFF + i * C::TILE + box * 2048, &tmQ, 64 * box, y, z, fb);
                            tma_load_3d(st + C::KOFF + i * C::TILE + box * 2048, &tmK, 64 * box, y, z, fb);
                            tma_load_3d(st + C::VOFF + i * C::TILE + box * 2048, &tmV, 64 * box, y, z, fb);
                        }
                    }
                    if (eb) bulk_load(st + C::EOFF, eta + bh * T + 16 * si * SPS, uint32_t(n) * 64, fb);
                } else {
                    mbar_arrive_expect_tx(fb, uint32_t(n) * (3 * C::TILE + 64));
                    for (int i = 0; i < n; ++i) {
                        const int y = int(bh * T) + 16 * (si * SPS + i);
#pragma unroll
                        for (int box = 0; box < D / 64; ++box) {
                            tma_load_2d(st + C::QOFF + i * C::TILE + box * 2048, &tmQ, 64 * box, y, fb);
                            tma_load_2d(st + C::KOFF + i * C::TILE + box * 2048, &tmK, 64 * box, y, fb);
                            tma_load_2d(st + C::VOFF + i * C::TILE + box * 2048, &tmV, 64 * box, y, fb);
                        }
                    }
                    bulk_load(st + C::EOFF, eta + bh * T + 16 * si * SPS, uint32_t(n) * 64, fb);
                }
                ++issued;
            }
            // never retire the CTA with copies in flight (this wait ignores the abort flag)
            for (int si = issued > NST ? issued - NST : 0; si < issued; ++si)
                mbar_wait_bounded(smem_u32(&full_bar[si % NST]), (si / NST) & 1, &s_zero, kWaitLimitNs);
        }
    } else {
        // ---------------------------------------------------------------- one column group
        const int cg = warp - 1;
        const int cw0 = (blockIdx.y * CG + cg) * 16;  // first output column of this group

        // lane-dependent ldmatrix coordinates (byte offsets inside a sub-tile):
        //  off_nk: B fragments with n = token, k = d (plain), used for K in K W and Q K^T;
        //  off_tk: A fragments with m = token, k = d (plain, Q) and B fragments with k = token,
        //          n = d (transposed, K in the update)
        uint32_t off_nk[KS], off_tk[KS];
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            off_nk[ks] = swz(lr + 8 * (lj >> 1), 16 * ks + 8 * (lj & 1));
            off_tk[ks] = swz(lr + 8 * (lj & 1), 16 * ks + 8 * (lj >> 1));
        }
        const uint32_t off_v = swz(lr + 8 * (lj >> 1), cw0 + 8 * (lj & 1));

        float w[NT][4];  // W^T[c][d_in], c = g (+8), d_in = 8*nt + 2t (+1)
        const float* W0h = W0 + bh * D * D;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int r = 8 * nt + 2 * t;
            w[nt][0] = W0h[size_t(r) * D + cw0 + g];
            w[nt][1] = W0h[size_t(r + 1) * D + cw0 + g];
            w[nt][2] = W0h[size_t(r) * D + cw0 + g + 8];
            w[nt][3] = W0h[size_t(r + 1) * D + cw0 + g + 8];
        }

        uint32_t wa0[KS][4];  // bf16 block-start state (A operand of W^T K^T)
        uint32_t wr[KS][4];   // bf16 running state (B operand of Q W); equals wa0 for b = 16
        uint32_t kb[2][KS][4], qa[2][KS][4], kt[KS][4];
        float ne[2][4], nv[2][8];  // -eta of the sub-block's tokens, eta . V in the P^T layout

        auto load_kq = [&](int buf, uint32_t st, int i) {
            const uint32_t k0 = st + C::KOFF + i * C::TILE, q0 = st + C::QOFF + i * C::TILE;
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) ldsm_x4(k0 + off_nk[ks], kb[buf][ks]);
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) ldsm_x4(q0 + off_tk[ks], qa[buf][ks]);
            uint32_t vv[4];
            ldsm_x4_trans(st + C::VOFF + i * C::TILE + off_v, vv);
            const float* es = reinterpret_cast<const float*>(smem + (st - sbase) + C::EOFF + i * 64);
            const float2 e01 = *reinterpret_cast<const float2*>(es + 2 * t);  // zero past T
            const float2 e23 = *reinterpret_cast<const float2*>(es + 8 + 2 * t);
            ne[buf][0] = -e01.x; ne[buf][1] = -e01.y; ne[buf][2] = -e23.x; ne[buf][3] = -e23.y;
            nv[buf][0] = e01.x * bf16_lo(vv[0]); nv[buf][1] = e01.y * bf16_hi(vv[0]);
            nv[buf][2] = e01.x * bf16_lo(vv[1]); nv[buf][3] = e01.y * bf16_hi(vv[1]);
            nv[buf][4] = e23.x * bf16_lo(vv[2]); nv[buf][5] = e23.y * bf16_hi(vv[2]);
            nv[buf][6] = e23.x * bf16_lo(vv[3]); nv[buf][7] = e23.y * bf16_hi(vv[3]);
        };
        auto load_kt = [&](uint32_t st, int i) {
            const uint32_t k0 = st + C::KOFF + i * C::TILE;
#pragma unroll
            for (int kk = 0; kk < KS; ++kk) ldsm_x4_trans(k0 + off_tk[kk], kt[kk]);
        };

        const bool m0 = 2 * t <= g, m1 = 2 * t + 1 <= g;  // causal mask of the scores' A fragment
        __nv_bfloat16* zb = Z + bh * size_t(T) * D + cw0 + 2 * t;
        float zp[2][4] = {};  // Z of the previous sub-block (tokens x columns), stored during the next one
        // chk: rows past T are not stored (only the last sub-block can be partial)
        auto store_z = [&](int sb, bool chk) {
            __nv_bfloat16* zr = zb + size_t(16 * sb + g) * D;  // rows 16 sb + g (+8), columns cw0 + 2t (+8)
            const bool lo = !chk || 16 * sb + g < T, hi = !chk || 16 * sb + g + 8 < T;
            if (lo) *reinterpret_cast<uint32_t*>(zr) = pack_bf16(zp[0][0], zp[0][1]);
            if (hi) *reinterpret_cast<uint32_t*>(zr + 8 * D) = pack_bf16(zp[0][2], zp[0][3]);
            if (lo) *reinterpret_cast<uint32_t*>(zr + 8) = pack_bf16(zp[1][0], zp[1][1]);
            if (hi) *reinterpret_cast<uint32_t*>(zr + 8 * D + 8) = pack_bf16(zp[1][2], zp[1][3]);
        };

        bool ok = true;
        for (int si = 0; ok && si < nstg; ++si) {
            const int s = si % NST, n = subs_in(si);
            const uint32_t par = (si / NST) & 1;
            const uint32_t st = sbase + s * C::STAGE;
            uint8_t* sc = smem + C::SC_OFF + s * SPS * C::SCB;
            if (!(ok = wait_all(full_bar[s], par))) break;
            // this warp's share of the stage's masked scores S = tril(Q K^T), as A fragments
            // (rows query i, cols key j); the second fragment buffers serve as scratch
            for (int i = cg; i < n; i += CG) {
                const uint32_t k0 = st + C::KOFF + i * C::TILE, q0 = st + C::QOFF + i * C::TILE;
#pragma unroll
                for (int ks = 0; ks < KS; ++ks) {
                    ldsm_x4(k0 + off_nk[ks], kb[1][ks]);
                    ldsm_x4(q0 + off_tk[ks], qa[1][ks]);
                }
                float sa[2][4];
                mma_bf16_16816_z(sa[0], qa[1][0], kb[1][0][0], kb[1][0][1]);
                mma_bf16_16816_z(sa[1], qa[1][0], kb[1][0][2], kb[1][0][3]);
#pragma unroll
                for (int ks = 1; ks < KS; ++ks) {
                    mma_bf16_16816(sa[0], qa[1][ks], kb[1][ks][0], kb[1][ks][1]);
                    mma_bf16_16816(sa[1], qa[1][ks], kb[1][ks][2], kb[1][ks][3]);
                }
                uint4 f;
                f.x = pack_bf16(m0 ? sa[0][0] : 0.f, m1 ? sa[0][1] : 0.f);
                f.y = pack_bf16(sa[0][2], sa[0][3]);
                f.z = 0u;
                f.w = pack_bf16(m0 ? sa[1][2] : 0.f, m1 ? sa[1][3] : 0.f);
                if constexpr (HIST) {
                    uint32_t* r = reinterpret_cast<uint32_t*>(sc + i * C::SCB) + lane;
                    r[0] = f.x;
                    r[32] = f.y;
                    r[64] = f.w;
                } else {
                    *reinterpret_cast<uint4*>(sc + i * 512 + lane * 16) = f;
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&sc_bar[s]));
            load_kq(0, st, 0);
            load_kt(st, 0);
            if (!(ok = wait_all(sc_bar[s], par))) break;
            // one 16-token sub-block; n is a compile-time SPS on full stages, so their loop body
            // has no branches and the compiler schedules across sub-blocks
            auto step = [&](const int i, const int n) {
                const int b = i & 1, sb = si * SPS + i;
                if (i > 0) load_kt(st, i);  // used by the update, well after K W and Q W
                if (i + 1 < n) load_kq(b ^ 1, st, i + 1);
                uint4 sf4;
                if constexpr (HIST) {
                    const uint32_t* r = reinterpret_cast<const uint32_t*>(sc + i * C::SCB) + lane;
                    sf4 = make_uint4(r[0], r[32], 0u, r[64]);
                } else {
                    sf4 = *reinterpret_cast<const uint4*>(sc + i * 512 + lane * 16);
                }
                const bool bstart = SINGLE || sb % nsub == 0;
                if (bstart) {
                    pack_state<KS>(w, wa0);
                    if constexpr (HIST) {
                        // the bf16 state at the start of block sb (blocks of 16): the A fragments of
                        // W^T stored transposed (stmatrix) into one of this warp's two [D][16] slices;
                        // a pair of blocks shares one proxy fence, after which two TMA stores write
                        // the slices to W_hist[block][d_in][cw0 ..] and the warp moves on (a plain
                        // store would hold its source registers until the memory system takes them,
                        // stalling the chain)
                        const uint32_t hs = sbase + C::HS_OFF + cg * D * 64;
                        if ((sb & 1) == 0) {
                            if (lane == 0) bulk_wait_read_all();  // the previous pair's stores have read both slices
                            __syncwarp();
                        }
                        const uint32_t slice = hs + (sb & 1) * D * 32;
#pragma unroll
                        for (int ks = 0; ks < KS; ++ks)
                            stsm_x4_trans(slice + (16 * ks + 8 * (lj >> 1) + lr) * 32 + (lj & 1) * 16, wa0[ks][0],
                                          wa0[ks][1], wa0[ks][2], wa0[ks][3]);
                        if ((sb & 1) == 1 || sb == nsb - 1) {  // the pair is complete (or the head ends)
                            fence_proxy_async_smem();
                            __syncwarp();
                            if (lane == 0) {
                                const int first = sb & ~1;
                                tma_store_2d(&tmH, cw0, int((bh * size_t(nsb) + first) * D), hs);
                                if (sb != first) tma_store_2d(&tmH, cw0, int((bh * size_t(nsb) + sb) * D), hs + D * 32);
                                bulk_commit();
                            }
                        }
                    }
                }
                if constexpr (!SINGLE) {
                    if (bstart) {
#pragma unroll
                        for (int ks = 0; ks < KS; ++ks)
#pragma unroll
                            for (int r = 0; r < 4; ++r) wr[ks][r] = wa0[ks][r];
                    } else {
                        pack_state<KS>(w, wr);
                    }
                }
                const uint32_t(&wq)[KS][4] = SINGLE ? wa0 : wr;

                // P^T = W0^T K^T at the block-start state (four independent partial sums)
                float pa[4][2][4];
#pragma unroll
                for (int ks = 0; ks < KS; ++ks) {
                    if (ks < 4) {
                        mma_bf16_16816_z(pa[ks][0], wa0[ks], kb[b][ks][0], kb[b][ks][1]);
                        mma_bf16_16816_z(pa[ks][1], wa0[ks], kb[b][ks][2], kb[b][ks][3]);
                    } else {
                        mma_bf16_16816(pa[ks & 3][0], wa0[ks], kb[b][ks][0], kb[b][ks][1]);
                        mma_bf16_16816(pa[ks & 3][1], wa0[ks], kb[b][ks][2], kb[b][ks][3]);
                    }
                }
                // read-out, first part: Z = Q W (running state), tokens x columns; one chain per
                // n-tile, off the critical path
                float za[2][4];
                mma_bf16_16816_z(za[0], qa[b][0], wq[0][0], wq[0][2]);
                mma_bf16_16816_z(za[1], qa[b][0], wq[0][1], wq[0][3]);
#pragma unroll
                for (int ks = 1; ks < KS; ++ks) {
                    mma_bf16_16816(za[0], qa[b][ks], wq[ks][0], wq[ks][2]);
                    mma_bf16_16816(za[1], qa[b][ks], wq[ks][1], wq[ks][3]);
                }
                if (i > 0) store_z(sb - 1, false);  // a whole sub-block: only the last can be partial
                float p[2][4];
#pragma unroll
                for (int j = 0; j < 2; ++j)
#pragma unroll
                    for (int k = 0; k < 4; ++k) p[j][k] = (pa[0][j][k] + pa[1][j][k]) + (pa[2][j][k] + pa[3][j][k]);
                // G = -eta . (P - V)^T as a bf16 A operand (rows c, cols token j)
                uint32_t ga[4];
                ga[0] = pack_bf16(fmaf(ne[b][0], p[0][0], nv[b][0]), fmaf(ne[b][1], p[0][1], nv[b][1]));
                ga[1] = pack_bf16(fmaf(ne[b][0], p[0][2], nv[b][2]), fmaf(ne[b][1], p[0][3], nv[b][3]));
                ga[2] = pack_bf16(fmaf(ne[b][2], p[1][0], nv[b][4]), fmaf(ne[b][3], p[1][1], nv[b][5]));
                ga[3] = pack_bf16(fmaf(ne[b][2], p[1][2], nv[b][6]), fmaf(ne[b][3], p[1][3], nv[b][7]));
                // W^T += G K   (rank-16 update of the running state, fp32 accumulate)
#pragma unroll
                for (int kk = 0; kk < KS; ++kk) {
                    mma_bf16_16816(w[2 * kk], ga, kt[kk][0], kt[kk][1]);
                    mma_bf16_16816(w[2 * kk + 1], ga, kt[kk][2], kt[kk][3]);
                }
                // read-out, second part: Z += S G^T  (G^T = -eta . E is the B operand held in ga)
                const uint32_t sf[4] = {sf4.x, sf4.y, sf4.z, sf4.w};
#pragma unroll
                for (int j = 0; j < 2; ++j)
#pragma unroll
                    for (int k = 0; k < 4; ++k) zp[j][k] = za[j][k];
                mma_bf16_16816(zp[0], sf, ga[0], ga[2]);
                mma_bf16_16816(zp[1], sf, ga[1], ga[3]);
            };
            if (n == SPS) {
#pragma unroll
                for (int i = 0; i < SPS; ++i) step(i, SPS);
            } else {
#pragma unroll
                for (int i = 0; i < SPS; ++i) {
                    if (i >= n) break;
                    step(i, n);
                }
            }
            store_z(si * SPS + n - 1, PART);  // the last sub-block of the head may be partial
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&empty_bar[s]));  // this warp's reads of the stage are done
        }
        if constexpr (HIST) {
            if (lane == 0) bulk_wait_all();  // the state stores are complete before the CTA retires
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
    }
    __syncthreads();
}

// ---------------------------------------------------------------- host side

template <int D, int CG, int NST, int SPS, bool SINGLE, bool HIST, bool PART>
cudaError_t launch_part(const LinearArgs& a, cudaStream_t s, int* status) {
    using C = FusedCfg<D, CG, NST, SPS, HIST>;
    const uint64_t heads = uint64_t(a.B) * a.H;
    CUtensorMap mq, mk, mv, mh;
    cudaError_t e;
    if (PART) {  // [heads][T][D]: the boxes of a partial sub-block read zeros past T
        if ((e = make_tma_map_bf16_heads(&mq, a.Q, heads, a.T, D)) != cudaSuccess) return e;
        if ((e = make_tma_map_bf16_heads(&mk, a.K, heads, a.T, D)) != cudaSuccess) return e;
        if ((e = make_tma_map_bf16_heads(&mv, a.V, heads, a.T, D)) != cudaSuccess) return e;
    } else {  // [heads * T][D]
        if ((e = make_tma_map_bf16(&mq, a.Q, heads * a.T, D)) != cudaSuccess) return e;
        if ((e = make_tma_map_bf16(&mk, a.K, heads * a.T, D)) != cudaSuccess) return e;
        if ((e = make_tma_map_bf16(&mv, a.V, heads * a.T, D)) != cudaSuccess) return e;
    }
    memset(&mh, 0, sizeof(mh));  // unused without the recorded states
    if (HIST && (e = make_tma_map_bf16_box(&mh, a.W_hist, heads * ((a.T + 15) / 16) * D, D, 16, 64, 0)) != cudaSuccess)
        return e;
    auto kern = linear_prefill_fused_kernel<D, CG, NST, SPS, SINGLE, HIST, PART>;
    const int bytes = C::BYTES + 1024;  // + alignment slack
    if ((e = allow_dynamic_smem(reinterpret_cast<const void*>(kern), bytes)) != cudaSuccess) return e;
    dim3 grid(unsigned(a.B) * unsigned(a.H), D / 16 / CG);
    kern<<<grid, C::THREADS, bytes, s>>>(mq, mk, mv, a.eta, a.W0, static_cast<__nv_bfloat16*>(a.Z), a.W_out, a.T,
                                         a.chunk, status, mh, a.wait_ns ? a.wait_ns : kWaitLimitNs);
    return cudaGetLastError();
}

template <int D, int CG, int NST, int SPS, bool SINGLE, bool HIST>
cudaError_t launch_cfg(const LinearArgs& a, cudaStream_t s, int* status) {
    // the 2D maps address rows bh * T + t with an int32 coordinate
    if (a.T % 16 || uint64_t(a.B) * a.H * a.T > 0x7fffffffull)
        return launch_part<D, CG, NST, SPS, SINGLE, HIST, true>(a, s, status);
    return launch_part<D, CG, NST, SPS, SINGLE, HIST, false>(a, s, status);
}

// stages of 256 tokens, double-buffered: 2 x 97 KB of Q/K/V/eta + 16 KB of scores + 8 KB of state
// staging per CTA (with the recorded states: 12 KB of scores + 16 KB of staging)
constexpr int kSps = 16, kNst = 2;

template <int CG>
cudaError_t launch_cg(const LinearArgs& a, cudaStream_t s, int* status) {
    if (a.W_hist) {
        if (a.chunk != 16) return cudaErrorNotSupported;
        return launch_cfg<64, CG, kNst, kSps, true, true>(a, s, status);
    }
    return a.chunk == 16 ? launch_cfg<64, CG, kNst, kSps, true, false>(a, s, status)
                         : launch_cfg<64, CG, kNst, kSps, false, false>(a, s, status);
}

}  // namespace

bool linear_prefill_fused_supported(const LinearArgs& a) {
    // any T: a ragged last block is fewer sub-blocks, and a partial last sub-block weighs its
    // tokens past T by zero.  TMA coordinates are int32: the head index, and for the recorded
    // states the row of W_hist.
    const uint64_t heads = uint64_t(a.B) * a.H;
    return a.bf16 && a.d == 64 && a.chunk % 16 == 0 && heads <= 0x7fffffffull &&
           (!a.W_hist || heads * ((uint64_t(a.T) + 15) / 16) * 64 <= 0x7fffffffull);
}

cudaError_t launch_linear_prefill_fused(const LinearArgs& a, cudaStream_t s, int* status) {
    if (!linear_prefill_fused_supported(a)) return cudaErrorNotSupported;
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const long long bh = (long long)a.B * a.H;
    // Column groups per CTA: 4 (one CTA per head); fewer when whole-head CTAs would leave more
    // than half of the SMs idle.
    int cg = 4;
    while (cg > 1 && bh * (4 / cg) * 2 <= (long long)sms) cg /= 2;
    switch (cg) {
        case 4: return launch_cg<4>(a, s, status);
        case 2: return launch_cg<2>(a, s, status);
        default: return launch_cg<1>(a, s, status);
    }
}

}  // namespace ttt
