// linear_segment.cu -- TTT-Linear prefill split along the sequence (bf16 Q/K/V/Z, fp32 state).
//
// What is computed is the chunked scan of "Test-Time Training Layers ..." (sections "The Core
// Mechanism" and "Hardware Parallelization") and of the TTT essay's dual-form paragraph: per block
// of b tokens with start state W,
//     E = K W - V;  Z = Q W - tril(eta . Q K^T) E;  W <- W - K^T diag(eta) E.
//
// Why split: a head's scan is one chain of T / 16 dependent 16-token steps, so with one CTA per
// head the sequence length, not the bytes, sets the time, and heads < SMs leaves SMs idle.
//
// The split (ours): the block update is affine in the block-start state,
//     W <- (I - K^T D K) W + K^T D V      (D = diag(eta)),
// so a segment of whole blocks maps its start state W_s to W_s + Delta_s W_s + B_s, with
//   * Delta_s = (product of the segment's (I - K^T D K)) - I: the same recurrence started from 0
//     with target values -K (x <- x - K^T D (K x + K) is (I + x) <- (I - K^T D K)(I + x)),
//   * B_s: the recurrence started from 0 with the real targets V.
// Keeping Delta (not I + Delta) keeps the bf16 operands of its products at full relative
// precision.  Three launches on the caller's stream:
//   1. map:     (Delta_s, B_s) of every segment but the last, in parallel (the recurrence on the
//               augmented targets [-K | V]: 2d columns, 2d / 16 column groups, no read-out);
//   2. combine: W_{s+1} = W_s + Delta_s W_s + B_s, s = 0 .. S-2, per head and 16-column group
//               (fp32, the only sequential part: S - 1 small products);
//   3. scan:    every segment from its own start state, with the read-out (Z) and, for the last
//               segment, the final state.
// All three are exact algebra: the result equals the one-pass scan up to fp32 rounding.
//
// Workspace (caller-owned, fp32), for P = B*H heads and S segments:
//   maps   [P][S-1][2][d][d]   (Delta_s, B_s)
//   starts [P][S][d][d]        W_s for s = 0 .. S-1 (W_0 a copy of the initial state, so the final
//                              state may overwrite the initial one in place)
// so ttt_linear_prefill_ws can be checked stage by stage.
#include <cuda.h>

#include "mma_tile.cuh"
#include "ptx.cuh"
#include "ttt_common.cuh"
#include "ttt_internal.h"

namespace ttt {
namespace {

using namespace ptx;

constexpr uint64_t kWaitLimitNs = 4000000000ull;  // 4 s: far beyond any legitimate wait

// ============================================================================ 1. segment maps

template <int D, int NG, int NST, int SPS>
struct MapCfg {
    static constexpr int KS = D / 16, NT = D / 8, TILE = 16 * D * 2;
    // a stage holds SPS sub-blocks: K sub-tiles, then V, then eta
    static constexpr int KOFF = 0, VOFF = SPS * TILE, EOFF = 2 * SPS * TILE;
    static constexpr int STAGE = (EOFF + SPS * 64 + 1023) / 1024 * 1024;
    static constexpr int BYTES = NST * STAGE;
    static constexpr int THREADS = 32 * (NG + 1);
};

// Grid: x = head * (S - 1) + segment (every segment but the last), y = set of NG column groups of
// the 2D augmented columns (groups 0 .. D/16-1: Delta with targets -K; the rest: B with targets V).
// Warp 0 streams K, V, eta by TMA / bulk copy; warps 1..NG each run the recurrence of one group.
template <int D, int NG, int NST, int SPS>
__global__ void __launch_bounds__(MapCfg<D, NG, NST, SPS>::THREADS, 1)
linear_segmap_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                     const float* __restrict__ eta, float* __restrict__ maps, int T, int chunk, int seg_len, int nseg,
                     int* status) {
    using C = MapCfg<D, NG, NST, SPS>;
    constexpr int KS = C::KS, NT = C::NT;

    extern __shared__ uint8_t smem_dyn[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
    __shared__ __align__(8) uint64_t full_bar[NST];
    __shared__ __align__(8) uint64_t empty_bar[NST];
    __shared__ volatile int s_err;
    __shared__ volatile int s_zero;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const size_t bh = blockIdx.x / (nseg - 1);
    const int sgi = blockIdx.x % (nseg - 1);
    const int t0 = sgi * seg_len;           // segments before the last have seg_len tokens
    const int nsb = seg_len / 16;
    const int nstg = (nsb + SPS - 1) / SPS;
    const int nsub = chunk / 16;
    const uint32_t sbase = smem_u32(smem);
    const int g = lane >> 2, t = lane & 3;
    const int lj = lane >> 3, lr = lane & 7;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(smem_u32(&full_bar[s]), 1);
            mbar_init(smem_u32(&empty_bar[s]), NG);
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
    auto wait_all = [&](uint64_t& bar, uint32_t parity) -> bool {
        return __all_sync(0xffffffffu, wait(bar, parity));
    };
    auto subs_in = [&](int si) { return nsb - si * SPS < SPS ? nsb - si * SPS : SPS; };

    if (warp == 0) {
        if (lane == 0) {
            prefetch_tensormap(&tmK);
            prefetch_tensormap(&tmV);
            int issued = 0;
            for (int si = 0; si < nstg; ++si) {
                const int s = si % NST, n = subs_in(si);
                if (si >= NST && !wait(empty_bar[s], ((si / NST) - 1) & 1)) break;
                const uint32_t fb = smem_u32(&full_bar[s]);
                mbar_arrive_expect_tx(fb, uint32_t(n) * (2 * C::TILE + 64));
                const uint32_t st = sbase + s * C::STAGE;
                for (int i = 0; i < n; ++i) {
                    const int y = int(bh * T) + t0 + 16 * (si * SPS + i);
#pragma unroll
                    for (int box = 0; box < D / 64; ++box) {
                        tma_load_2d(st + C::KOFF + i * C::TILE + box * 2048, &tmK, 64 * box, y, fb);
                        tma_load_2d(st + C::VOFF + i * C::TILE + box * 2048, &tmV, 64 * box, y, fb);
                    }
                }
                bulk_load(st + C::EOFF, eta + bh * T + t0 + 16 * si * SPS, uint32_t(n) * 64, fb);
                ++issued;
            }
            // never retire the CTA with copies in flight (this wait ignores the abort flag)
            for (int si = issued > NST ? issued - NST : 0; si < issued; ++si)
                mbar_wait_bounded(smem_u32(&full_bar[si % NST]), (si / NST) & 1, &s_zero, kWaitLimitNs);
        }
    } else {
        const int gi = blockIdx.y * NG + warp - 1;  // augmented column group
        const bool is_delta = gi < D / 16;
        const int c0 = 16 * (is_delta ? gi : gi - D / 16);
        uint32_t off_nk[KS], off_tk[NT / 2];
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) off_nk[ks] = swz(lr + 8 * (lj >> 1), 16 * ks + 8 * (lj & 1));
#pragma unroll
        for (int kk = 0; kk < NT / 2; ++kk) off_tk[kk] = swz(lr + 8 * (lj & 1), 16 * kk + 8 * (lj >> 1));
        const uint32_t off_v = swz(lr + 8 * (lj >> 1), c0 + 8 * (lj & 1));
        // the targets: columns c0.. of -K (Delta) or of V (B), read from the stage's K or V tiles
        const uint32_t tgt_off = is_delta ? uint32_t(C::KOFF) : uint32_t(C::VOFF);
        const float tsign = is_delta ? -1.f : 1.f;

        float w[NT][4];  // X^T[c][d_in] of this group, starting from 0
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) w[nt][0] = w[nt][1] = w[nt][2] = w[nt][3] = 0.f;
        uint32_t wa0[KS][4];
        uint32_t kb[KS][4], kt[NT / 2][4];
        float ne0 = 0, ne1 = 0, ne2 = 0, ne3 = 0, nv[8] = {};
        auto load = [&](uint32_t st, int i) {
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) ldsm_x4(st + C::KOFF + i * C::TILE + off_nk[ks], kb[ks]);
#pragma unroll
            for (int kk = 0; kk < NT / 2; ++kk) ldsm_x4_trans(st + C::KOFF + i * C::TILE + off_tk[kk], kt[kk]);
            uint32_t vv[4];
            ldsm_x4_trans(st + tgt_off + i * C::TILE + off_v, vv);
            const float* es = reinterpret_cast<const float*>(smem + (st - sbase) + C::EOFF + i * 64);
            const float2 e01 = *reinterpret_cast<const float2*>(es + 2 * t);
            const float2 e23 = *reinterpret_cast<const float2*>(es + 8 + 2 * t);
            ne0 = -e01.x; ne1 = -e01.y; ne2 = -e23.x; ne3 = -e23.y;
            const float a0 = tsign * e01.x, a1 = tsign * e01.y, a2 = tsign * e23.x, a3 = tsign * e23.y;
            nv[0] = a0 * bf16_lo(vv[0]); nv[1] = a1 * bf16_hi(vv[0]);
            nv[2] = a0 * bf16_lo(vv[1]); nv[3] = a1 * bf16_hi(vv[1]);
            nv[4] = a2 * bf16_lo(vv[2]); nv[5] = a3 * bf16_hi(vv[2]);
            nv[6] = a2 * bf16_lo(vv[3]); nv[7] = a3 * bf16_hi(vv[3]);
        };
        bool ok = wait_all(full_bar[0], 0);
        if (ok) load(sbase, 0);
        for (int si = 0; ok && si < nstg; ++si) {
            const int s = si % NST, n = subs_in(si);
            const uint32_t st = sbase + s * C::STAGE;
            auto step = [&](int i) {
                const int sb = si * SPS + i;  // sub-block inside the segment (t0 is a block boundary)
                if (sb % nsub == 0) pack_state<KS>(w, wa0);
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
                uint32_t ga[4];  // G = -eta . (K X - target)^T
                ga[0] = pack_bf16(fmaf(ne0, p[0][0], nv[0]), fmaf(ne1, p[0][1], nv[1]));
                ga[1] = pack_bf16(fmaf(ne0, p[0][2], nv[2]), fmaf(ne1, p[0][3], nv[3]));
                ga[2] = pack_bf16(fmaf(ne2, p[1][0], nv[4]), fmaf(ne3, p[1][1], nv[5]));
                ga[3] = pack_bf16(fmaf(ne2, p[1][2], nv[6]), fmaf(ne3, p[1][3], nv[7]));
#pragma unroll
                for (int kk = 0; kk < NT / 2; ++kk) {
                    mma_bf16_16816(w[2 * kk], ga, kt[kk][0], kt[kk][1]);
                    mma_bf16_16816(w[2 * kk + 1], ga, kt[kk][2], kt[kk][3]);
                }
            };
            if (n == SPS) {
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
            if (lane == 0) mbar_arrive(smem_u32(&empty_bar[s]));
            if (si + 1 < nstg) {
                ok = wait_all(full_bar[(si + 1) % NST], ((si + 1) / NST) & 1);
                if (ok) load(sbase + ((si + 1) % NST) * C::STAGE, 0);
            }
        }
        float* M = maps + ((bh * (nseg - 1) + sgi) * 2 + (is_delta ? 0 : 1)) * size_t(D) * D;
        store_state<NT>(w, M, D, c0, g, t);
    }
    __syncthreads();
}

// ============================================================================ 2. combine

// Grid (heads, D / CW), D * CW threads (thread: row r = tid / CW, column c0 + tid % CW): W_0 = the
// initial state, then W_{s+1}[:, c0..c0+CW) = W_s + Delta_s W_s + B_s for s = 0..S-2, in fp32.  Only
// W_s is on the chain; Delta_s and B_s are known up front, so they stream NS - 1 hops ahead by
// cp.async into a ring of stages (Delta rows as 16-byte chunks, chunk j of row r at j ^ (r & 7):
// the eight rows a warp reads at once fall in distinct banks).  The state's columns are kept
// transposed (column c as a row of D + 4 words, so the four columns a warp reads sit in distinct
// banks) and double buffered: a hop reads Delta and W in 16-byte pieces and costs one barrier.
template <int D>
struct CombineCfg {
    static constexpr int CW = 4, NT = D * CW, NS = 4;
    static constexpr int DELTA = D * D, BROWS = D * CW, STAGE = DELTA + BROWS;  // floats
    static constexpr int WLD = D + 4;                                           // floats per state column
    static constexpr int BYTES = (NS * STAGE + 2 * CW * WLD) * 4;
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

template <int D>
__global__ void __launch_bounds__(CombineCfg<D>::NT) linear_segcombine_kernel(const float* __restrict__ W0,
                                                                             const float* __restrict__ maps,
                                                                             float* __restrict__ starts, int nseg) {
    using C = CombineCfg<D>;
    constexpr int CW = C::CW, NS = C::NS;
    extern __shared__ __align__(16) float cmb[];
    float* ring = cmb;                   // NS x [Delta (swizzled D x D) | B columns (D x CW)]
    float* Wc = ring + NS * C::STAGE;    // [2][CW][WLD], the current start state's columns
    const size_t bh = blockIdx.x;
    const int c0 = CW * blockIdx.y;
    const int tid = threadIdx.x, cc = tid % CW, r = tid / CW;
    const int hops = nseg - 1;
    const float* mp = maps + bh * size_t(hops) * 2 * D * D;

    auto issue = [&](int hop) {
        float* st = ring + (hop % NS) * C::STAGE;
        const float* Dm = mp + size_t(hop) * 2 * D * D;
        const float* Bm = Dm + size_t(D) * D;
#pragma unroll
        for (int u = 0; u < D * D / 4 / C::NT; ++u) {
            const int i = tid + C::NT * u, row = i / (D / 4), j = i % (D / 4);
            cp_async16(smem_u32(st + row * D + ((j ^ (row & 7)) << 2)), Dm + size_t(row) * D + 4 * j);
        }
        if (tid < D) cp_async16(smem_u32(st + C::DELTA + tid * CW), Bm + size_t(tid) * D + c0);
    };
#pragma unroll
    for (int p = 0; p < NS - 1; ++p) {
        if (p < hops) issue(p);
        cp_async_commit();
    }
    float* Ws0 = starts + bh * nseg * size_t(D) * D;
    float w = W0[bh * D * D + size_t(r) * D + c0 + cc];
    Wc[cc * C::WLD + r] = w;
    Ws0[size_t(r) * D + c0 + cc] = w;
    for (int s = 0; s < hops; ++s) {
        cp_async_wait<NS - 2>();  // this thread's copies of hop s have landed
        __syncthreads();          // everyone's have; W_s is complete; hop s - 1's stage is free
        if (s + NS - 1 < hops) issue(s + NS - 1);
        cp_async_commit();
        const float* st = ring + (s % NS) * C::STAGE;
        const float* Wcur = Wc + (s & 1) * CW * C::WLD + cc * C::WLD;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kc = 0; kc < D / 4; ++kc) {
            const float4 dq = *reinterpret_cast<const float4*>(st + r * D + ((kc ^ (r & 7)) << 2));
            const float4 wq = *reinterpret_cast<const float4*>(Wcur + 4 * kc);
            acc[0] = fmaf(dq.x, wq.x, acc[0]);
            acc[1] = fmaf(dq.y, wq.y, acc[1]);
            acc[2] = fmaf(dq.z, wq.z, acc[2]);
            acc[3] = fmaf(dq.w, wq.w, acc[3]);
        }
        w = w + (((acc[0] + acc[1]) + (acc[2] + acc[3])) + st[C::DELTA + r * CW + cc]);
        Wc[((s + 1) & 1) * CW * C::WLD + cc * C::WLD + r] = w;
        starts[(bh * nseg + s + 1) * size_t(D) * D + size_t(r) * D + c0 + cc] = w;
    }
    cp_async_wait<0>();
}

// ============================================================================ 3. segment scan, d = 64

// Two (head, segment) slots per CTA, four warps each: warp 4 * slot + c runs column group c (16
// output columns) of its slot's segment, recurrence and read-out together in registers, exactly as
// the one-pass d = 64 kernel does (see linear_prefill_fused.cu).  Eight warps and no producer warp,
// so every thread keeps 255 registers (a ninth warp would cut that to 168) and an SM runs two
// segments: the two warps on each SM sub-partition share its MMA pipe, which one warp leaves about
// half idle.  Lane 0 of the slot's first warp issues the TMA copies: stages 0 .. NST-1 up front,
// then stage si + NST - 1 once it has passed the score barrier of stage si, which every warp of the
// slot reaches only after its last read of stage si - 1 (the slot being refilled).
template <int NST, int SPS>
struct SegCfg {
    static constexpr int D = 64, KS = 4, NT = 8, TILE = 16 * D * 2, CG = 4;
    static constexpr int QOFF = 0, KOFF = SPS * TILE, VOFF = 2 * SPS * TILE, EOFF = 3 * SPS * TILE;
    static constexpr int STAGE = (EOFF + SPS * 64 + 1023) / 1024 * 1024;
    static constexpr int SC_OFF = NST * STAGE;          // masked scores [NST][SPS][32 lanes] x 16 B
    static constexpr int SLOT = SC_OFF + NST * SPS * 512;  // bytes per slot (a multiple of 1024)
    static constexpr int BYTES = 2 * SLOT;
    static constexpr int THREADS = 256;
};

template <int NST, int SPS, bool SINGLE>
__global__ void __launch_bounds__(256, 1)
linear_prefill_seg_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                          const __grid_constant__ CUtensorMap tmV, const float* __restrict__ eta,
                          const float* W0, const float* starts, __nv_bfloat16* __restrict__ Z,
                          float* W_out, int T, int chunk, int seg_len, int nseg, int npairs, int* status) {
    using C = SegCfg<NST, SPS>;
    constexpr int D = C::D, KS = C::KS, NT = C::NT, CG = C::CG;
    static_assert(NST >= 2, "the refill scheme needs at least two stages");

    extern __shared__ uint8_t smem_dyn[];
    uint8_t* smem0 = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
    __shared__ __align__(8) uint64_t full_bar[2][NST];
    __shared__ __align__(8) uint64_t sc_bar[2][NST];  // the stage's masked scores are written
    __shared__ volatile int s_err;
    __shared__ volatile int s_zero;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int slot = warp >> 2, cg = warp & 3;
    const int pair = blockIdx.x * 2 + slot;
    const bool active = pair < npairs;
    const size_t bh = size_t(active ? pair : 0) / nseg;
    const int sgi = (active ? pair : 0) % nseg;
    const int t0 = sgi * seg_len;
    const int ntok = T - t0 < seg_len ? T - t0 : seg_len;
    const int nsb = ntok / 16;
    const int nstg = (nsb + SPS - 1) / SPS;
    const int nsub = chunk / 16;
    uint8_t* smem = smem0 + slot * C::SLOT;
    const uint32_t sbase = smem_u32(smem);
    const int g = lane >> 2, t = lane & 3;
    const int lj = lane >> 3, lr = lane & 7;

    if (threadIdx.x == 0) {
        for (int k = 0; k < 2; ++k)
            for (int s = 0; s < NST; ++s) {
                mbar_init(smem_u32(&full_bar[k][s]), 1);
                mbar_init(smem_u32(&sc_bar[k][s]), CG);
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
    auto wait_all = [&](uint64_t& bar, uint32_t parity) -> bool {
        return __all_sync(0xffffffffu, wait(bar, parity));
    };
    auto subs_in = [&](int si) { return nsb - si * SPS < SPS ? nsb - si * SPS : SPS; };

    if (active) {
        const bool issuer = cg == 0 && lane == 0;
        int issued = 0, landed = 0;  // (issuer only) stages issued, stages whose data this warp saw land
        auto issue = [&](int si) {
            const int s = si % NST, n = subs_in(si);
            const uint32_t fb = smem_u32(&full_bar[slot][s]);
            mbar_arrive_expect_tx(fb, uint32_t(n) * (3 * C::TILE + 64));
            const uint32_t st = sbase + s * C::STAGE;
            for (int i = 0; i < n; ++i) {
                const int y = int(bh * T) + t0 + 16 * (si * SPS + i);
                tma_load_2d(st + C::QOFF + i * C::TILE, &tmQ, 0, y, fb);
                tma_load_2d(st + C::KOFF + i * C::TILE, &tmK, 0, y, fb);
                tma_load_2d(st + C::VOFF + i * C::TILE, &tmV, 0, y, fb);
            }
            bulk_load(st + C::EOFF, eta + bh * T + t0 + 16 * si * SPS, uint32_t(n) * 64, fb);
            ++issued;
        };
        if (issuer) {
            prefetch_tensormap(&tmQ);
            prefetch_tensormap(&tmK);
            prefetch_tensormap(&tmV);
            for (int si = 0; si < NST && si < nstg; ++si) issue(si);
        }

        const int cw0 = cg * 16;
        uint32_t off_nk[KS], off_tk[KS];
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            off_nk[ks] = swz(lr + 8 * (lj >> 1), 16 * ks + 8 * (lj & 1));
            off_tk[ks] = swz(lr + 8 * (lj & 1), 16 * ks + 8 * (lj >> 1));
        }
        const uint32_t off_v = swz(lr + 8 * (lj >> 1), cw0 + 8 * (lj & 1));

        float w[NT][4];
        load_state<NT>(w, nseg == 1 ? W0 + bh * D * D : starts + (bh * nseg + sgi) * size_t(D) * D, D, cw0, g, t);
        uint32_t wa0[KS][4];
        uint32_t wr[KS][4];
        uint32_t kb[2][KS][4], qa[2][KS][4], kt[KS][4];
        float ne[2][4], nv[2][8];

        auto load_kq = [&](int buf, uint32_t st, int i) {
            const uint32_t k0 = st + C::KOFF + i * C::TILE, q0 = st + C::QOFF + i * C::TILE;
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) ldsm_x4(k0 + off_nk[ks], kb[buf][ks]);
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) ldsm_x4(q0 + off_tk[ks], qa[buf][ks]);
            uint32_t vv[4];
            ldsm_x4_trans(st + C::VOFF + i * C::TILE + off_v, vv);
            const float* es = reinterpret_cast<const float*>(smem + (st - sbase) + C::EOFF + i * 64);
            const float2 e01 = *reinterpret_cast<const float2*>(es + 2 * t);
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

        const bool m0 = 2 * t <= g, m1 = 2 * t + 1 <= g;
        __nv_bfloat16* zb = Z + (bh * size_t(T) + t0) * D + cw0 + 2 * t;
        float zp[2][4] = {};
        auto store_z = [&](int sb) {
            __nv_bfloat16* zr = zb + size_t(16 * sb + g) * D;
            *reinterpret_cast<uint32_t*>(zr) = pack_bf16(zp[0][0], zp[0][1]);
            *reinterpret_cast<uint32_t*>(zr + 8 * D) = pack_bf16(zp[0][2], zp[0][3]);
            *reinterpret_cast<uint32_t*>(zr + 8) = pack_bf16(zp[1][0], zp[1][1]);
            *reinterpret_cast<uint32_t*>(zr + 8 * D + 8) = pack_bf16(zp[1][2], zp[1][3]);
        };

        bool ok = true;
        for (int si = 0; ok && si < nstg; ++si) {
            const int s = si % NST, n = subs_in(si);
            const uint32_t par = (si / NST) & 1;
            const uint32_t st = sbase + s * C::STAGE;
            uint8_t* sc = smem + C::SC_OFF + s * SPS * 512;
            if (!(ok = wait_all(full_bar[slot][s], par))) break;
            if (issuer) ++landed;
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
                *reinterpret_cast<uint4*>(sc + i * 512 + lane * 16) = f;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&sc_bar[slot][s]));
            load_kq(0, st, 0);
            load_kt(st, 0);
            if (!(ok = wait_all(sc_bar[slot][s], par))) break;
            // every warp of the slot has left stage si - 1: refill its ring slot
            if (issuer && si >= 1 && si + NST - 1 < nstg) issue(si + NST - 1);
            __syncwarp();
            auto step = [&](const int i, const int n) {
                const int b = i & 1, sb = si * SPS + i;
                if (i > 0) load_kt(st, i);
                if (i + 1 < n) load_kq(b ^ 1, st, i + 1);
                const uint4 sf4 = *reinterpret_cast<const uint4*>(sc + i * 512 + lane * 16);
                const bool bstart = SINGLE || sb % nsub == 0;
                if (bstart) pack_state<KS>(w, wa0);
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
                float pa[4][2][4];
#pragma unroll
                for (int ks = 0; ks < KS; ++ks) {
                    mma_bf16_16816_z(pa[ks][0], wa0[ks], kb[b][ks][0], kb[b][ks][1]);
                    mma_bf16_16816_z(pa[ks][1], wa0[ks], kb[b][ks][2], kb[b][ks][3]);
                }
                float za[2][4];
                mma_bf16_16816_z(za[0], qa[b][0], wq[0][0], wq[0][2]);
                mma_bf16_16816_z(za[1], qa[b][0], wq[0][1], wq[0][3]);
#pragma unroll
                for (int ks = 1; ks < KS; ++ks) {
                    mma_bf16_16816(za[0], qa[b][ks], wq[ks][0], wq[ks][2]);
                    mma_bf16_16816(za[1], qa[b][ks], wq[ks][1], wq[ks][3]);
                }
                if (i > 0) store_z(sb - 1);
                float p[2][4];
#pragma unroll
                for (int j = 0; j < 2; ++j)
#pragma unroll
                    for (int k = 0; k < 4; ++k) p[j][k] = (pa[0][j][k] + pa[1][j][k]) + (pa[2][j][k] + pa[3][j][k]);
                uint32_t ga[4];
                ga[0] = pack_bf16(fmaf(ne[b][0], p[0][0], nv[b][0]), fmaf(ne[b][1], p[0][1], nv[b][1]));
                ga[1] = pack_bf16(fmaf(ne[b][0], p[0][2], nv[b][2]), fmaf(ne[b][1], p[0][3], nv[b][3]));
                ga[2] = pack_bf16(fmaf(ne[b][2], p[1][0], nv[b][4]), fmaf(ne[b][3], p[1][1], nv[b][5]));
                ga[3] = pack_bf16(fmaf(ne[b][2], p[1][2], nv[b][6]), fmaf(ne[b][3], p[1][3], nv[b][7]));
#pragma unroll
                for (int kk = 0; kk < KS; ++kk) {
                    mma_bf16_16816(w[2 * kk], ga, kt[kk][0], kt[kk][1]);
                    mma_bf16_16816(w[2 * kk + 1], ga, kt[kk][2], kt[kk][3]);
                }
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
            store_z(si * SPS + n - 1);
        }
        if (sgi == nseg - 1) store_state<NT>(w, W_out + bh * D * D, D, cw0, g, t);
        // never retire the CTA with copies in flight (this wait ignores the abort flag)
        if (issuer)
            for (int si = landed; si < issued; ++si)
                mbar_wait_bounded(smem_u32(&full_bar[slot][si % NST]), (si / NST) & 1, &s_zero, kWaitLimitNs);
    }
    __syncthreads();
}

// ============================================================================ host side

int sm_count() {
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return sms;
}

template <int D, int NG, int NST, int SPS>
cudaError_t launch_maps(const LinearArgs& a, const SegPlan& p, float* maps, cudaStream_t s, int* status) {
    using C = MapCfg<D, NG, NST, SPS>;
    const uint64_t rows = uint64_t(a.B) * a.H * a.T;
    CUtensorMap mk, mv;
    cudaError_t e;
    if ((e = make_tma_map_bf16(&mk, a.K, rows, D)) != cudaSuccess) return e;
    if ((e = make_tma_map_bf16(&mv, a.V, rows, D)) != cudaSuccess) return e;
    auto kern = linear_segmap_kernel<D, NG, NST, SPS>;
    const int bytes = C::BYTES + 1024;
    if ((e = allow_dynamic_smem(reinterpret_cast<const void*>(kern), bytes)) != cudaSuccess) return e;
    dim3 grid(unsigned(a.B) * unsigned(a.H) * unsigned(p.nseg - 1), 2 * D / 16 / NG);
    kern<<<grid, C::THREADS, bytes, s>>>(mk, mv, a.eta, maps, a.T, a.chunk, p.seg_len, p.nseg, status);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_combine(const LinearArgs& a, const SegPlan& p, const float* maps, float* starts, cudaStream_t s) {
    using C = CombineCfg<D>;
    auto kern = linear_segcombine_kernel<D>;
    cudaError_t e;
    if ((e = allow_dynamic_smem(reinterpret_cast<const void*>(kern), C::BYTES)) != cudaSuccess)
        return e;
    kern<<<dim3(unsigned(a.B) * unsigned(a.H), D / C::CW), C::NT, C::BYTES, s>>>(a.W0, maps, starts, p.nseg);
    return cudaGetLastError();
}

constexpr int kSegSps = 8, kSegNst = 2;

cudaError_t launch_scan64(const LinearArgs& a, const SegPlan& p, const float* starts, cudaStream_t s, int* status) {
    using C = SegCfg<kSegNst, kSegSps>;
    const uint64_t rows = uint64_t(a.B) * a.H * a.T;
    CUtensorMap mq, mk, mv;
    cudaError_t e;
    if ((e = make_tma_map_bf16(&mq, a.Q, rows, 64)) != cudaSuccess) return e;
    if ((e = make_tma_map_bf16(&mk, a.K, rows, 64)) != cudaSuccess) return e;
    if ((e = make_tma_map_bf16(&mv, a.V, rows, 64)) != cudaSuccess) return e;
    const int npairs = a.B * a.H * p.nseg;
    const int bytes = C::BYTES + 1024;
    auto run = [&](auto kern) -> cudaError_t {
        cudaError_t e2 = allow_dynamic_smem(reinterpret_cast<const void*>(kern), bytes);
        if (e2 != cudaSuccess) return e2;
        kern<<<unsigned((npairs + 1) / 2), C::THREADS, bytes, s>>>(mq, mk, mv, a.eta, a.W0, starts,
                                                                   static_cast<__nv_bfloat16*>(a.Z), a.W_out, a.T,
                                                                   a.chunk, p.seg_len, p.nseg, npairs, status);
        return cudaGetLastError();
    };
    return a.chunk == 16 ? run(linear_prefill_seg_kernel<kSegNst, kSegSps, true>)
                         : run(linear_prefill_seg_kernel<kSegNst, kSegSps, false>);
}

}  // namespace

bool linear_segmented_supported(const LinearArgs& a) {
    return a.bf16 && a.d == 64 && a.chunk % 16 == 0 && a.T % a.chunk == 0 && a.T > 0 &&
           uint64_t(a.B) * a.H * a.T <= 0x7fffffffull && uint64_t(a.B) * a.H > 0;
}

SegPlan linear_segment_plan(const LinearArgs& a, int force_nseg) {
    SegPlan p{1, a.T};
    if (!linear_segmented_supported(a)) return p;
    const long long heads = (long long)a.B * a.H;
    const int nblk = a.T / a.chunk;
    // The maps cost as much warp-MMA work as the scan of their segments, and the one-pass kernel
    // already saturates the warp-MMA rate of every SM it occupies (measured on B300), so a split
    // pays only where the one-pass scan (one CTA per head, four column groups) leaves at least three
    // quarters of the SMs idle.  Then: two segments per SM (one CTA of two slots), at least 256
    // tokens per segment.
    const int sms = sm_count();
    if (force_nseg <= 0 && heads * 4 > sms) return p;
    long long nseg = force_nseg > 0 ? force_nseg : (2LL * sms) / heads;
    const long long max_by_len = (long long)a.T / 256 > 0 ? (long long)a.T / 256 : 1;
    if (force_nseg <= 0 && nseg > max_by_len) nseg = max_by_len;
    if (nseg > nblk) nseg = nblk;
    if (nseg < 1) nseg = 1;
    const int blk_per_seg = int((nblk + nseg - 1) / nseg);
    p.seg_len = blk_per_seg * a.chunk;
    p.nseg = (nblk + blk_per_seg - 1) / blk_per_seg;  // no empty segment
    return p;
}

size_t linear_segment_workspace_bytes(const LinearArgs& a, const SegPlan& p) {
    if (p.nseg <= 1) return 0;
    return size_t(a.B) * a.H * (3 * size_t(p.nseg) - 2) * size_t(a.d) * a.d * sizeof(float);
}

cudaError_t launch_linear_prefill_segmented(const LinearArgs& a, const SegPlan& p, void* workspace, cudaStream_t s,
                                            int* status) {
    if (!linear_segmented_supported(a)) return cudaErrorNotSupported;
    float* maps = static_cast<float*>(workspace);
    float* starts = maps ? maps + size_t(a.B) * a.H * (p.nseg - 1) * 2 * a.d * a.d : nullptr;
    cudaError_t e;
    if (p.nseg > 1) {
        if ((e = launch_maps<64, 8, 3, 8>(a, p, maps, s, status)) != cudaSuccess) return e;
        if ((e = launch_combine<64>(a, p, maps, starts, s)) != cudaSuccess) return e;
    }
    return launch_scan64(a, p, starts, s, status);
}

}  // namespace ttt
