// linear_prefill_mma.cu -- tensor-core TTT-Linear prefill (bf16 Q/K/V/Z, fp32 state).
//
// What is computed ("Test-Time Training Layers ...", sections "The Core
// Mechanism" and "Hardware Parallelization"; TTT essay, paragraph on the dual
// form): per block of b tokens with start state W0,
//     E = K W0 - V;  Z = Q W0 - tril(eta . Q K^T) E;  W = W0 - K^T diag(eta) E.
//
// Design (ours, for sm_103a):
//  * The scan over blocks is a chain of small dependent steps (16 x d x d per
//    16 tokens), bound by the latency of one step, not by FLOPs or bytes.  The
//    state therefore never leaves the register file, held transposed (W^T) in
//    the accumulator layout of the warp-level m16n8k16 bf16 MMA, which after an
//    fp32->bf16 pack is also the A-operand layout: K W0, Q W and the rank-16
//    update K^T diag(eta) E (accumulated straight into W in fp32) need no
//    shared-memory round trip.  (The 5th-generation tcgen05 MMA accepts an
//    N = 16 instruction only every ~40 cycles and needs a commit/mbarrier round
//    trip of several hundred cycles: too slow for a chain of 16 x d x d steps.)
//  * Output columns are independent for f = kW: a column group of 16 owns
//    columns [16c, 16c+16) of W, E and Z, and has two warps.  The chain warp
//    runs only the recurrence (K W0, E, the rank-16 update): the
//    latency-critical path.  Measured on B300, that recurrence alone costs
//    ~180 cycles per 16 tokens at d = 64, while each shared-memory or mbarrier
//    operation on the same warp adds tens of cycles; so the chain warp touches
//    the barriers once per stage of SPS sub-blocks and exports only the 16 x 16
//    error operand G (one 16-byte store per lane).  The read-out warp keeps its
//    own copy of the running state, applying the same bf16 updates in the same
//    order (bitwise the chain's state), and forms Z^T = (Q W)^T + G tril(QK^T)^T.
//  * A block of b = 16*nsub tokens runs as nsub sub-blocks of 16: E of every
//    sub-block uses the block-start state (bf16 copy in registers), the read-out
//    state accumulates the earlier sub-blocks' updates; this equals
//    Z = Q W0 - tril(eta.QK^T) E without forming the b x b matrix.
//  * Warp 0 streams Q/K/V by TMA (16-token boxes, 128-byte swizzle:
//    conflict-free ldmatrix) and eta by a bulk copy into an NST-stage mbarrier
//    ring; a stage holds SPS = 4 sub-blocks (64 tokens).  Warp 1
//    computes the masked 16 x 16 scores tril(Q K^T) of each sub-block once per
//    CTA (they do not depend on the state) and leaves them in shared memory in
//    MMA-fragment order.  Warps 2..2+CG-1 are the chain warps, the rest the
//    read-out warps.
//  * All waits are bounded; on expiry the kernel records TTT_ERR_TIMEOUT, every
//    warp leaves its loop (no warp waits on another without a bound), and the
//    producer drains its copies before the CTA exits.
#include <cuda.h>

#include "ptx.cuh"
#include "ttt_common.cuh"
#include "ttt_internal.h"

namespace ttt {
namespace {

using namespace ptx;

constexpr uint64_t kWaitLimitNs = 4000000000ull;  // 4 s: far beyond any legitimate wait

// byte offset of (row, col) in a [16][D] bf16 tile stored as D/64 TMA boxes of
// [16][64] with the 128-byte swizzle (16-byte chunk index XOR row%8); col % 8 == 0
__device__ __forceinline__ uint32_t swz(int row, int col) {
    return uint32_t((col >> 6) * 2048 + row * 128 + ((((col & 63) >> 3) ^ (row & 7)) << 4));
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

// NX, the depth of the error-operand ring, equals NST: the chain warp can only write the
// operands of stage si after the producer refilled that stage, i.e. after the read-out
// warp released stage si - NST, whose operands used the same slot.
template <int D, int CG, int NST, int SPS, int NX>
struct Cfg {
    static_assert(NX == NST, "error-operand ring must be as deep as the stage ring");
    static constexpr int KS = D / 16;  // k-steps over the input dimension
    static constexpr int NT = D / 8;   // 8-wide n-tiles of the state over the input dimension
    static constexpr int TILE = 16 * D * 2;  // bytes of one 16-token [16][D] bf16 sub-tile
    // a stage holds SPS sub-blocks: Q sub-tiles, then K, then V, then eta
    static constexpr int QOFF = 0, KOFF = SPS * TILE, VOFF = 2 * SPS * TILE, EOFF = 3 * SPS * TILE;
    static constexpr int STAGE = (EOFF + SPS * 64 + 1023) / 1024 * 1024;
    static constexpr int SC_OFF = NST * STAGE;                      // scores [NST][SPS][32 lanes] x 16 B
    static constexpr int G_OFF = SC_OFF + NST * SPS * 512;          // error operands [CG][NX][SPS][32] x 16 B
    static constexpr int ZBUF_OFF = G_OFF + CG * NX * SPS * 512;    // per group [16][16] bf16 Z staging
    static constexpr int BYTES = ZBUF_OFF + CG * 512;
    static constexpr int THREADS = 32 * (2 * CG + 2);
};

// HIST: also write the state at the start of every block to W_hist [B*H][ceil(T/16)][D][D], rounded
// to bf16 (what the backward reads); instantiated for blocks of 16 tokens only.
// PART: T is not a multiple of 16 (a partial last sub-block), or the rows of all heads exceed the int32
// coordinate of a 2D tensor map.  Then Q/K/V come through per-head 3D maps (tokens past a head's end
// read as zeros), eta by cp.async where a bulk copy cannot take it, and the rows of Z past T are not
// stored; the instantiation for the common case compiles none of that.
template <int D, int CG, int NST, int SPS, int NX, bool SINGLE, bool HIST, bool PART>
__global__ void __launch_bounds__(Cfg<D, CG, NST, SPS, NX>::THREADS, 1)
linear_prefill_mma_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                          const __grid_constant__ CUtensorMap tmV, const float* __restrict__ eta,
                          const float* W0, __nv_bfloat16* __restrict__ Z, float* W_out, int T, int chunk,
                          int* status, __nv_bfloat16* __restrict__ W_hist) {
    using C = Cfg<D, CG, NST, SPS, NX>;
    constexpr int KS = C::KS, NT = C::NT;

    extern __shared__ uint8_t smem_dyn[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
    __shared__ __align__(8) uint64_t full_bar[NST];
    __shared__ __align__(8) uint64_t sc_bar[NST];
    __shared__ __align__(8) uint64_t empty_bar[NST];
    __shared__ __align__(8) uint64_t xf_bar[CG][NX];  // error operands of a stage written (chain -> read-out)
    __shared__ volatile int s_err;
    __shared__ volatile int s_zero;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const size_t bh = blockIdx.x;
    const int nsb = PART ? (T + 15) / 16 : T / 16;  // 16-token sub-blocks (with PART the last may be partial)
    const int nstg = (nsb + SPS - 1) / SPS;    // stages
    const int nsub = chunk / 16;               // sub-blocks per block
    const bool ebulk = (T & 3) == 0;           // a head's eta starts 16-byte aligned (PART)
    const uint32_t sbase = smem_u32(smem);
    const int g = lane >> 2, t = lane & 3;
    const int lj = lane >> 3, lr = lane & 7;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(smem_u32(&full_bar[s]), 1);
            mbar_init(smem_u32(&sc_bar[s]), 1);
            mbar_init(smem_u32(&empty_bar[s]), CG + 1);
        }
        for (int c = 0; c < CG; ++c)
            for (int j = 0; j < NX; ++j) mbar_init(smem_u32(&xf_bar[c][j]), 1);
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
    auto subs_in = [&](int si) { return nsb - si * SPS < SPS ? nsb - si * SPS : SPS; };
    // a stage of SPS whole sub-blocks: its loops run without the checks for a partial sub-block
    auto full_stage = [&](int si) { return subs_in(si) == SPS && (!PART || 16 * SPS * (si + 1) <= T); };

    // lane-dependent ldmatrix coordinates (byte offsets inside a sub-tile)
    uint32_t off_nk[KS], off_tk[NT / 2];
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) off_nk[ks] = swz(lr + 8 * (lj >> 1), 16 * ks + 8 * (lj & 1));
#pragma unroll
    for (int kk = 0; kk < NT / 2; ++kk) off_tk[kk] = swz(lr + 8 * (lj & 1), 16 * kk + 8 * (lj >> 1));

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
                const uint32_t st = sbase + s * C::STAGE;
                if constexpr (PART) {
                    // eta: one bulk copy when every token of the stage exists and a head's eta starts
                    // on a 16-byte boundary (4 | T); otherwise 4-byte cp.async copies that the
                    // stage's mbarrier tracks, and zeros past T.  Q/K/V boxes past T read zeros.
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
    } else if (warp == 1) {
        // ------------------------------------------------------------ masked scores
        // S = tril(Q K^T) of every sub-block, as the B fragments of the read-out's
        // correction product G * S_masked (n-tiles: query tokens 0..7 and 8..15).
        const bool m0 = 2 * t <= g, m1 = 2 * t + 1 <= g;
        for (int si = 0; si < nstg; ++si) {
            const int s = si % NST, n = subs_in(si);
            if (!wait_all(full_bar[s], (si / NST) & 1)) break;
            const uint32_t st = sbase + s * C::STAGE;
            for (int i = 0; i < n; ++i) {
                float sc[2][4] = {}, sd[2][4] = {};
#pragma unroll
                for (int ks = 0; ks < KS; ++ks) {
                    uint32_t qb[4], kb[4];
                    ldsm_x4(st + C::QOFF + i * C::TILE + off_nk[ks], qb);
                    ldsm_x4(st + C::KOFF + i * C::TILE + off_nk[ks], kb);
                    const uint32_t qa[4] = {qb[0], qb[2], qb[1], qb[3]};
                    float(&acc)[2][4] = (ks & 1) ? sd : sc;
                    mma_bf16_16816(acc[0], qa, kb[0], kb[1]);
                    mma_bf16_16816(acc[1], qa, kb[2], kb[3]);
                }
#pragma unroll
                for (int j = 0; j < 2; ++j)
#pragma unroll
                    for (int k = 0; k < 4; ++k) sc[j][k] += sd[j][k];
                uint4 f;
                f.x = pack_bf16(m0 ? sc[0][0] : 0.f, m1 ? sc[0][1] : 0.f);
                f.y = pack_bf16(sc[0][2], sc[0][3]);
                f.z = pack_bf16(m0 ? sc[1][2] : 0.f, m1 ? sc[1][3] : 0.f);
                f.w = 0;
                *reinterpret_cast<uint4*>(smem + C::SC_OFF + (s * SPS + i) * 512 + lane * 16) = f;
            }
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(smem_u32(&sc_bar[s]));
                mbar_arrive(smem_u32(&empty_bar[s]));  // this warp's reads of the stage are done
            }
        }
    } else {
        // ------------------------------------------------------------ chain and read-out
        const bool chain = warp < 2 + CG;
        const int cg = chain ? warp - 2 : warp - 2 - CG;
        const int cw0 = (blockIdx.y * CG + cg) * 16;  // first output column of this group

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
        uint8_t* gslots = smem + C::G_OFF + cg * NX * SPS * 512;

        if (chain) {
            // The recurrence only: P = K W0 (block-start state), G = -eta (P - V), W += K^T G.
            // Per stage: one wait, one arrive; the fragments of the next sub-block are loaded
            // while this one's products are in flight.
            const uint32_t off_v = swz(lr + 8 * (lj >> 1), cw0 + 8 * (lj & 1));
            uint32_t wa0[KS][4];
            uint32_t kb[KS][4], kt[NT / 2][4];
            float ne0 = 0, ne1 = 0, ne2 = 0, ne3 = 0, nv[8] = {};
            auto load = [&](uint32_t st, int i) {
#pragma unroll
                for (int ks = 0; ks < KS; ++ks) ldsm_x4(st + C::KOFF + i * C::TILE + off_nk[ks], kb[ks]);
#pragma unroll
                for (int kk = 0; kk < NT / 2; ++kk) ldsm_x4_trans(st + C::KOFF + i * C::TILE + off_tk[kk], kt[kk]);
                uint32_t vv[4];
                ldsm_x4_trans(st + C::VOFF + i * C::TILE + off_v, vv);
                const float* es = reinterpret_cast<const float*>(smem + (st - sbase) + C::EOFF + i * 64);
                const float2 e01 = *reinterpret_cast<const float2*>(es + 2 * t);  // zero past T
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
                const int s = si % NST, n = subs_in(si), x = si % NX;
                const uint32_t st = sbase + s * C::STAGE;
                uint8_t* gout = gslots + x * SPS * 512;
                // one 16-token sub-block of the recurrence
                auto step = [&](int i) {
                    const int sb = si * SPS + i;
                    if (SINGLE || sb % nsub == 0) {
                        if constexpr (HIST) {  // the state at the start of block sb / nsub, as bf16
                            __nv_bfloat16* wh = W_hist + (bh * size_t(nsb) + sb) * D * D;  // chunk 16
#pragma unroll
                            for (int nt = 0; nt < NT; ++nt) {
                                const int r = 8 * nt + 2 * t;
                                wh[size_t(r) * D + cw0 + g] = __float2bfloat16_rn(w[nt][0]);
                                wh[size_t(r + 1) * D + cw0 + g] = __float2bfloat16_rn(w[nt][1]);
                                wh[size_t(r) * D + cw0 + g + 8] = __float2bfloat16_rn(w[nt][2]);
                                wh[size_t(r + 1) * D + cw0 + g + 8] = __float2bfloat16_rn(w[nt][3]);
                            }
                        }
                        pack_state<KS>(w, wa0);
                    }
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
                    *reinterpret_cast<uint4*>(gout + i * 512 + lane * 16) = make_uint4(ga[0], ga[1], ga[2], ga[3]);
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
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&xf_bar[cg][x]));
                if (si + 1 < nstg) {
                    const int s1 = (si + 1) % NST;
                    ok = wait_all(full_bar[s1], ((si + 1) / NST) & 1);
                    if (ok) load(sbase + s1 * C::STAGE, 0);
                }
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
            // Read-out: keeps its own copy of the running state (the same bf16 updates in the
            // same order, so it is bitwise the chain's), and forms Z^T = (Q W_run)^T + G S_masked.
            const uint32_t zst = sbase + C::ZBUF_OFF + cg * 512;
            const uint32_t zst_w = zst + (lr + 8 * (lj >> 1)) * 32 + (((lj & 1) ^ ((lr >> 2) & 1)) << 4);
            const int zrow = lane >> 1, zhalf = lane & 1;
            const uint32_t zst_r = zst + zrow * 32 + ((zhalf ^ ((zrow >> 2) & 1)) << 4);
            __nv_bfloat16* zp = Z + (bh * T + zrow) * D + cw0 + 8 * zhalf;
            for (int si = 0; si < nstg; ++si) {
                const int s = si % NST, n = subs_in(si), x = si % NX;
                const uint32_t par = (si / NST) & 1;
                if (!wait_all(full_bar[s], par) || !wait_all(sc_bar[s], par) || !wait_all(xf_bar[cg][x], (si / NX) & 1))
                    break;
                const uint32_t st = sbase + s * C::STAGE;
                const uint8_t* gin = gslots + x * SPS * 512;
                // chk: rows past T are not stored (only the last sub-block can be partial)
                auto step = [&](int i, bool chk) {
                    uint32_t qb[KS][4], kt[NT / 2][4], wr[KS][4];
#pragma unroll
                    for (int ks = 0; ks < KS; ++ks) ldsm_x4(st + C::QOFF + i * C::TILE + off_nk[ks], qb[ks]);
#pragma unroll
                    for (int kk = 0; kk < NT / 2; ++kk) ldsm_x4_trans(st + C::KOFF + i * C::TILE + off_tk[kk], kt[kk]);
                    const uint4 sz = *reinterpret_cast<const uint4*>(smem + C::SC_OFF + (s * SPS + i) * 512 + lane * 16);
                    const uint4 gf = *reinterpret_cast<const uint4*>(gin + i * 512 + lane * 16);
                    const uint32_t ga[4] = {gf.x, gf.y, gf.z, gf.w};
                    pack_state<KS>(w, wr);
                    float qp[4][2][4] = {};
#pragma unroll
                    for (int ks = 0; ks < KS; ++ks) {
                        mma_bf16_16816(qp[ks & 3][0], wr[ks], qb[ks][0], qb[ks][1]);
                        mma_bf16_16816(qp[ks & 3][1], wr[ks], qb[ks][2], qb[ks][3]);
                    }
#pragma unroll
                    for (int kk = 0; kk < NT / 2; ++kk) {
                        mma_bf16_16816(w[2 * kk], ga, kt[kk][0], kt[kk][1]);
                        mma_bf16_16816(w[2 * kk + 1], ga, kt[kk][2], kt[kk][3]);
                    }
                    float q0[2][4];
#pragma unroll
                    for (int j = 0; j < 2; ++j)
#pragma unroll
                        for (int k = 0; k < 4; ++k) q0[j][k] = (qp[0][j][k] + qp[1][j][k]) + (qp[2][j][k] + qp[3][j][k]);
                    mma_bf16_16816(q0[0], ga, sz.x, 0u);
                    mma_bf16_16816(q0[1], ga, sz.y, sz.z);
                    // Z: stmatrix.trans into the group's staging tile, one 16-byte store per lane
                    stsm_x4_trans(zst_w, pack_bf16(q0[0][0], q0[0][1]), pack_bf16(q0[0][2], q0[0][3]),
                                  pack_bf16(q0[1][0], q0[1][1]), pack_bf16(q0[1][2], q0[1][3]));
                    __syncwarp();
                    uint4 v;
                    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                                 : "r"(zst_r)
                                 : "memory");
                    if (!PART || !chk || 16 * (si * SPS + i) + zrow < T) *reinterpret_cast<uint4*>(zp) = v;
                    zp += 16 * D;
                    __syncwarp();
                                };
                if (full_stage(si)) {
#pragma unroll
                    for (int i = 0; i < SPS; ++i) step(i, false);
                } else {
                    for (int i = 0; i < n; ++i) step(i, true);
                }
                __syncwarp();
                // Q, K, the scores and the error operands of this stage are consumed; the chain
                // warp finished with the stage before it published the error operands
                if (lane == 0) mbar_arrive(smem_u32(&empty_bar[s]));
            }
        }
    }
    __syncthreads();
}

// ---------------------------------------------------------------- host side

template <int D, int CG, int NST, int SPS, int NX, bool SINGLE, bool HIST, bool PART>
cudaError_t launch_part(const LinearArgs& a, cudaStream_t s, int* status) {
    using C = Cfg<D, CG, NST, SPS, NX>;
    const uint64_t heads = uint64_t(a.B) * a.H;
    CUtensorMap mq, mk, mv;
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
    auto kern = linear_prefill_mma_kernel<D, CG, NST, SPS, NX, SINGLE, HIST, PART>;
    const int bytes = C::BYTES + 1024;  // + alignment slack
    if ((e = allow_dynamic_smem(reinterpret_cast<const void*>(kern), bytes)) != cudaSuccess) return e;
    dim3 grid(unsigned(a.B) * unsigned(a.H), D / 16 / CG);
    kern<<<grid, C::THREADS, bytes, s>>>(mq, mk, mv, a.eta, a.W0, static_cast<__nv_bfloat16*>(a.Z), a.W_out, a.T,
                                         a.chunk, status, static_cast<__nv_bfloat16*>(a.W_hist));
    return cudaGetLastError();
}

template <int D, int CG, int NST, int SPS, int NX, bool SINGLE, bool HIST = false>
cudaError_t launch_cfg(const LinearArgs& a, cudaStream_t s, int* status) {
    // the 2D maps address rows bh * T + t with an int32 coordinate
    if (a.T % 16 || uint64_t(a.B) * a.H * a.T > 0x7fffffffull)
        return launch_part<D, CG, NST, SPS, NX, SINGLE, HIST, true>(a, s, status);
    return launch_part<D, CG, NST, SPS, NX, SINGLE, HIST, false>(a, s, status);
}

// Each mbarrier wait costs the waiting warp ~230 cycles on B300 even when the phase has
// already completed, so a stage carries several 16-token sub-blocks (SPS).
template <int D, int CG, int NST, int SPS>
cudaError_t launch_chunk(const LinearArgs& a, cudaStream_t s, int* status) {
    if (a.W_hist) {
        if (a.chunk != 16) return cudaErrorNotSupported;
        return launch_cfg<D, CG, NST, SPS, NST, true, true>(a, s, status);
    }
    return a.chunk == 16 ? launch_cfg<D, CG, NST, SPS, NST, true>(a, s, status)
                         : launch_cfg<D, CG, NST, SPS, NST, false>(a, s, status);
}

}  // namespace

cudaError_t launch_linear_prefill_mma(const LinearArgs& a, cudaStream_t s, int* status) {
    // any T: a ragged last block is fewer sub-blocks, and a partial last sub-block weighs its tokens
    // past T by zero
    if (!a.bf16 || (a.d != 64 && a.d != 128) || a.chunk % 16 != 0) return cudaErrorNotSupported;
    if (uint64_t(a.B) * a.H > 0x7fffffffull) return cudaErrorNotSupported;  // TMA head coordinate is int32
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const long long bh = (long long)a.B * a.H;
    // Column groups per CTA: up to 4 (one CTA per head at d = 64); fewer when whole-head
    // CTAs would leave more than half of the SMs idle.
    int cg = a.d / 16 < 4 ? a.d / 16 : 4;
    if (a.d == 128 && cg > 2) cg = 2;  // shared memory: at most two column groups per CTA at d = 128
    while (cg > 1 && bh * (a.d / 16 / cg) * 2 <= (long long)sms) cg /= 2;
    if (a.d == 64) {
        switch (cg) {
            case 4: return launch_chunk<64, 4, 3, 8>(a, s, status);
            case 2: return launch_chunk<64, 2, 3, 8>(a, s, status);
            default: return launch_chunk<64, 1, 3, 8>(a, s, status);
        }
    }
    switch (cg) {
        case 4:
        case 2: return launch_chunk<128, 2, 4, 4>(a, s, status);
        default: return launch_chunk<128, 1, 4, 4>(a, s, status);
    }
}

}  // namespace ttt
