// mlp_prefill_mma.cu -- TTT-MLP prefill for d = 64, hidden = 256, blocks of 16 tokens, bf16
// Q/K/V/Z, fp32 state, on warp-level tensor-core MMAs with the whole state in registers.
//
// What is computed ("Test-Time Training (TTT) Layers for Sequence Modeling", section
// "Variants: TTT-Linear vs. TTT-MLP"; loss, step and readout of "Test-Time Training Layers
// ...", section "The Core Mechanism"; gradients at the block start as in the TTT essay's
// dual-form paragraph).  Per block of 16 tokens with start state (W1 [64][256], W2 [256][64]):
//   Zk = K W1, Hk = GELU(Zk), E2 = Hk W2 - V, E1 = (E2 W2^T) . GELU'(Zk)
//   Hq = GELU(Q W1 - tril(Q K^T) diag(eta) E1)
//   Z  = Hq W2 - tril(Hq Hk^T) diag(eta) E2
//   W1 <- W1 - K^T diag(eta) E1,   W2 <- W2 - Hk^T diag(eta) E2
//
// Design (ours, for sm_103a):
//  * The scan is a chain of dependent products per 16 tokens (Zk, E2, E1, the updates).  As
//    tcgen05 products each link costs an MMA -> commit -> mbarrier -> TMEM-load round trip of
//    several hundred cycles; here every link is a handful of warp-level m16n8k16 MMAs on
//    register operands.
//  * Eight compute warps; warp w owns hidden units [32w, 32w + 32): its slices of W1^T
//    (32 x 64) and W2^T (64 x 32), fp32, in the MMA accumulator layout.  An accumulator
//    fragment of a matrix X, read as bf16 pairs, is the A fragment of X and the B fragment of
//    X^T, both contracting over X's column index.  Every product is arranged so that it
//    contracts over the column index of its register operand, or takes the operand from
//    shared memory, or transposes it in registers (movmatrix):
//      Zk = K W1                   A: K tile           B: W1^T fragments        (over d)
//      E2^T (partial) = W2^T Hk^T  A: W2^T fragments   B: Zk-layout Hk           (over the slice)
//      E1 = E2 W2^T . GELU'(Zk)    A: E2 (shared)      B: bf16 copy of W2 (shared, per slice)
//      W1^T += (-eta E1)^T K       A: movmatrix(-eta E1)   B: K tile
//      W2^T += (-eta E2)^T Hk      A: (shared)         B: movmatrix(Hk)
//      read-out: Zq1 = Q W1 + tril(Q K^T)(-eta E1), Hq = GELU(Zq1),
//                Z = Hq W2 + tril(Hq Hk^T)(-eta E2)   (start-of-block W1, W2)
//  * Contractions over the hidden dimension (E2, Hq W2, Hq Hk^T) are split over the eight
//    warps and summed in shared memory between two named barriers per block; the read-out's
//    sums of block n are taken inside block n + 1's barriers, so it adds none.
//  * K/Q/V tiles arrive by TMA and eta by bulk copy in a 4-slot ring; thread 0 refills a slot
//    right after the first barrier of the block that no longer reads it.  No producer warp:
//    with eight warps the compiler may give each thread the 255 registers the state needs.
//    Each warp forms the masked scores tril(Q K^T) itself from fragments it already loads.
//  * Waits on mbarriers are bounded.  The warps meet only at reducing barriers (bar.red.or of
//    the per-thread error flag), so after an expired wait they all leave the loop at the same
//    barrier; thread 0 drains the copies in flight before the CTA exits.
#include <cuda.h>
#include <string.h>

#include "ptx.cuh"
#include "ttt_common.cuh"
#include "ttt_internal.h"

namespace ttt {
namespace {

using namespace ptx;

constexpr uint64_t kWaitLimitNs = 4000000000ull;  // 4 s: far beyond any legitimate wait
constexpr int D = 64, HID = 256, BT = 16;
constexpr int NCW = 8;         // warps
constexpr int HS = HID / NCW;  // hidden units per warp
constexpr int NST = 4;         // ring slots
constexpr int THREADS = 32 * NCW;
constexpr int TILE = BT * D * 2;  // [16][64] bf16, one TMA box

// shared memory (offsets from a 1024-byte aligned base)
constexpr int SLOT = 8192;  // K | Q | V | eta (64 B)
constexpr int S_K = 0, S_Q = TILE, S_V = 2 * TILE, S_ETA = 3 * TILE;
constexpr int OFF_W2C = NST * SLOT;              // bf16 W2 [256 hidden][64], 128-byte swizzled rows
constexpr int OFF_E2P = OFF_W2C + HID * 128;     // E2^T partials [8 warps][256 fragments] float4
constexpr int OFF_ZP = OFF_E2P + NCW * 4096;     // Hq W2 partials [8 warps][8 n-tiles][32 lanes] float4
constexpr int OFF_SP = OFF_ZP + NCW * 4096;      // Hq Hk^T partials [8 warps][2 n-tiles][32 lanes] float4
constexpr int OFF_E2T = OFF_SP + NCW * 1024;     // E2^T bf16 [64][16]
constexpr int OFF_NE2T = OFF_E2T + 2048;         // (-eta E2)^T bf16 [2 blocks][64][16]
constexpr int OFF_S2 = OFF_NE2T + 2 * 2048;      // tril(Hq Hk^T) bf16 [16][16]
constexpr int SMEM_BYTES = OFF_S2 + 512;
// the recording variant: per warp a [64 d][32 hidden] bf16 staging slice of W1 (64-byte rows, 64-byte
// swizzle), written out by a TMA store; W2 goes out straight from its bf16 copy
constexpr int OFF_H1S = (SMEM_BYTES + 1023) / 1024 * 1024;
constexpr int SMEM_BYTES_HIST = OFF_H1S + NCW * 4096;
static_assert(SMEM_BYTES_HIST + 1024 <= 232448, "shared memory");
// byte offset of (row, col) in a [rows][32] bf16 block with 64-byte rows and the 64-byte swizzle (16-byte
// chunk index XOR (row / 2) % 4, the pattern a TMA store with that mode reads); col % 8 == 0
__device__ __forceinline__ uint32_t sw64(int row, int col) {
    return uint32_t(row * 64 + ((((col >> 3) ^ (row >> 1)) & 3) << 4));
}

// byte offset of (row, col) in a [rows][64] bf16 block with 128-byte rows, 16-byte chunk index
// XOR row % 8 (the layout a TMA box with the 128-byte swizzle writes); col % 8 == 0
__device__ __forceinline__ uint32_t swz(int row, int col) {
    return uint32_t(row * 128 + ((((col >> 3) ^ row) & 7) << 4));
}
// byte offset of (row, col) in a [rows][16] bf16 block with 32-byte rows, chunk XOR (row / 4) % 2
// (rows 0..7 of an 8 x 8 ldmatrix tile then fall in distinct banks)
__device__ __forceinline__ uint32_t sw16(int row, int col) {
    return uint32_t(row * 32 + ((((col >> 3) ^ (row >> 2)) & 1) << 4) + (col & 7) * 2);
}

__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t& r0, uint32_t& r1) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr) : "memory");
}
// transpose of an 8 x 8 bf16 tile held one row pair per thread (thread (g, t): row g, cols 2t, 2t + 1)
__device__ __forceinline__ uint32_t movt(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

__device__ __forceinline__ float tanh_fast(float x) {
    float y;
    asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
// GELU, tanh form, and its exact derivative (of the tanh form)
__device__ __forceinline__ float gelu(float x) {
    const float c = 0.7978845608028654f, a = 0.044715f;
    const float t = tanh_fast(c * fmaf(a * x, x * x, x));
    return 0.5f * x * (1.f + t);
}
__device__ __forceinline__ float gelu_and_prime(float x, float& gp) {
    const float c = 0.7978845608028654f, a = 0.044715f;
    const float t = tanh_fast(c * fmaf(a * x, x * x, x));
    gp = 0.5f * (1.f + t) + 0.5f * x * (1.f - t * t) * c * fmaf(3.f * a, x * x, 1.f);
    return 0.5f * x * (1.f + t);
}

// barrier over the compute warps that also ORs a per-thread flag: every thread gets the same answer
__device__ __forceinline__ bool bar_compute_any(bool c) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, 1, %2, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(uint32_t(c)), "n"(32 * NCW)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ float bf16_at(const uint8_t* tile, int row, int col) {
    return __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(tile + swz(row, col & ~7) + (col & 7) * 2));
}

// HIST: also write the state at the start of every block to W1_hist / W2_hist (bf16).
// PART: T is not a multiple of 16 (a partial last block), or the rows of all heads exceed the int32
// coordinate of a 2D tensor map.  Then Q/K/V come through per-head 3D maps (tokens past a head's end
// read as zeros), eta by cp.async where a bulk copy cannot take it, and the rows of Z past T are not
// stored; the instantiation for the common case compiles none of that.
template <bool HIST, bool PART>
__global__ void __launch_bounds__(THREADS, 1)
mlp_prefill_mma_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const float* __restrict__ eta, const float* W1_0,
                       const float* W2_0, __nv_bfloat16* __restrict__ Z, float* W1_out, float* W2_out, int T,
                       const __grid_constant__ CUtensorMap tmH1, const __grid_constant__ CUtensorMap tmH2,
                       int* status) {
    extern __shared__ uint8_t smem_dyn[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
    __shared__ __align__(8) uint64_t full_bar[NST];  // TMA data of a slot landed
    __shared__ volatile int s_err;
    __shared__ volatile int s_zero;  // never set: abort flag of the waits that must run to completion

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const size_t bh = blockIdx.x;
    const int nblk = PART ? (T + BT - 1) / BT : T / BT;  // with PART the last block may be partial
    const uint32_t sb = smem_u32(smem);
    const int g = lane >> 2, t = lane & 3;
    const int lr = lane & 7, lm = lane >> 3;  // ldmatrix: row inside a tile, tile index

    if (threadIdx.x == 0) {
        for (int s = 0; s < NST; ++s) mbar_init(smem_u32(&full_bar[s]), 1);
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

    // ldmatrix row offsets inside a [16][64] tile, k-step ks (columns 16 ks ..):
    //  off_a: tiles (rows 0-7, k lo), (rows 8-15, k lo), (rows 0-7, k hi), (rows 8-15, k hi) -- the
    //         A fragment of the tile; with .trans, the B fragments of the tile (K = rows) for the
    //         column n-tiles 2 ks and 2 ks + 1
    //  off_b: tiles (rows 0-7, k lo), (rows 0-7, k hi), (rows 8-15, k lo), (rows 8-15, k hi) -- the
    //         B fragments (N = rows) for the row n-tiles 0 and 1
    uint32_t off_a[4], off_b[4];
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
        off_a[ks] = swz(lr + 8 * (lm & 1), 16 * ks + 8 * (lm >> 1));
        off_b[ks] = swz(lr + 8 * (lm >> 1), 16 * ks + 8 * (lm & 1));
    }

    auto issue = [&](int m) {  // thread 0: TMA copies of block m into slot m % NST
        const int s = m % NST;
        const uint32_t fb = smem_u32(&full_bar[s]);
        const uint32_t st = sb + s * SLOT;
        if constexpr (PART) {
            // eta by bulk copy when the block's 16 values exist and start on a 16-byte boundary
            // (4 | T); otherwise by 4-byte cp.async copies that the slot's mbarrier tracks, and
            // zeros past T (every read of the slot's previous block is done by now)
            const bool ebulk = (T & 3) == 0 && BT * (m + 1) <= T;
            if (!ebulk) {
                float* es = reinterpret_cast<float*>(smem + s * SLOT + S_ETA);
                const float* eg = eta + bh * T + BT * m;
                for (int j = 0; j < BT; ++j) {
                    if (BT * m + j < T) cp_async4(st + S_ETA + 4 * j, eg + j);
                    else es[j] = 0.f;
                }
                cp_async_mbar_arrive(fb);  // before this thread's own arrive on the phase
            }
            mbar_arrive_expect_tx(fb, 3 * TILE + (ebulk ? 64 : 0));
            const int y = BT * m, z = int(bh);
            tma_load_3d(st + S_K, &tmK, 0, y, z, fb);
            tma_load_3d(st + S_Q, &tmQ, 0, y, z, fb);
            tma_load_3d(st + S_V, &tmV, 0, y, z, fb);
            if (ebulk) bulk_load(st + S_ETA, eta + bh * T + BT * m, 64, fb);
        } else {
            mbar_arrive_expect_tx(fb, 3 * TILE + 64);
            const int y = int(bh * T) + BT * m;
            tma_load_2d(st + S_K, &tmK, 0, y, fb);
            tma_load_2d(st + S_Q, &tmQ, 0, y, fb);
            tma_load_2d(st + S_V, &tmV, 0, y, fb);
            bulk_load(st + S_ETA, eta + bh * T + BT * m, 64, fb);
        }
    };
    int issued = 0;  // thread 0's count of blocks whose copies it issued
    if (threadIdx.x == 0) {
        prefetch_tensormap(&tmQ);
        prefetch_tensormap(&tmK);
        prefetch_tensormap(&tmV);
        for (; issued < NST && issued < nblk; ++issued) issue(issued);
    }
    {
        const int h0 = HS * warp;  // first hidden unit of this warp
        // W1^T slice: w1[mh][nd] = rows (hidden) 16 mh + g (+8), columns (d) 8 nd + 2t (+1)
        // W2^T slice: w2[mo][nh] = rows (d) 16 mo + g (+8), columns (hidden) 8 nh + 2t (+1)
        float w1[2][8][4], w2[4][4][4];
        {
            const float* W1h = W1_0 + bh * D * HID;
            const float* W2h = W2_0 + bh * HID * D;
#pragma unroll
            for (int mh = 0; mh < 2; ++mh)
#pragma unroll
                for (int nd = 0; nd < 8; ++nd)
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        w1[mh][nd][k] = W1h[size_t(8 * nd + 2 * t + (k & 1)) * HID + h0 + 16 * mh + g + 8 * (k >> 1)];
#pragma unroll
            for (int mo = 0; mo < 4; ++mo)
#pragma unroll
                for (int nh = 0; nh < 4; ++nh)
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        w2[mo][nh][k] = W2h[size_t(h0 + 8 * nh + 2 * t + (k & 1)) * D + 16 * mo + g + 8 * (k >> 1)];
        }
        // bf16 copy of this warp's rows of W2 ([hidden][d]) for the E1 product: transposing stores
        auto store_w2c = [&]() {
#pragma unroll
            for (int nh = 0; nh < 4; ++nh)
#pragma unroll
                for (int mp = 0; mp < 2; ++mp)
                    stsm_x4_trans(sb + OFF_W2C + swz(h0 + 8 * nh + lr, 32 * mp + 8 * lm),
                                  pack_bf16(w2[2 * mp][nh][0], w2[2 * mp][nh][1]),
                                  pack_bf16(w2[2 * mp][nh][2], w2[2 * mp][nh][3]),
                                  pack_bf16(w2[2 * mp + 1][nh][0], w2[2 * mp + 1][nh][1]),
                                  pack_bf16(w2[2 * mp + 1][nh][2], w2[2 * mp + 1][nh][3]));
        };
        store_w2c();
        if constexpr (HIST) fence_proxy_async_smem();  // the first block's TMA store reads the copy
        __syncwarp();

        const bool m0 = 2 * t <= g, m1 = 2 * t + 1 <= g;  // causal mask of the score fragment
        const float4* e2p_all = reinterpret_cast<const float4*>(smem + OFF_E2P);
        const float4* zp_all = reinterpret_cast<const float4*>(smem + OFF_ZP);
        const float4* sp_all = reinterpret_cast<const float4*>(smem + OFF_SP);
        bool err = false;
        float zq[4][4], gp[4][4];
        uint32_t sca[4];     // tril(Q K^T) of the block as an A fragment (rows query, K = key)
        uint32_t hkp[4][2];  // Hk as bf16 pairs: [n-tile j (hidden 8j..)][token rows 0-7 / 8-15]
        float4 zsum = make_float4(0.f, 0.f, 0.f, 0.f);

        for (int n = 0; n <= nblk; ++n) {
            const bool have = n < nblk;
            const int s = n % NST;
            const uint32_t par = (n / NST) & 1;
            const uint32_t st = sb + s * SLOT;
            if (have) {
                if (!err && !wait(full_bar[s], par)) err = true;
                if constexpr (HIST) {
                    // the state at the start of block n (this warp's hidden slice), rounded to bf16: the
                    // operand the block's products use and what the backward reads.  W1^T is staged
                    // transposed into [d][32 hidden] (stmatrix.trans), W2 is already in its bf16 copy
                    // (rows [hidden][d], 128-byte swizzle); one TMA store each, and the warp moves on
                    // (scalar stores would hold their source registers on the chain)
                    const uint32_t s1 = sb + OFF_H1S + warp * 4096;
                    if (lane == 0) bulk_wait_read_all();  // the previous block's stores have read the staging
                    __syncwarp();
#pragma unroll
                    for (int mh = 0; mh < 2; ++mh)
#pragma unroll
                        for (int nd = 0; nd < 8; nd += 2)
                            stsm_x4_trans(s1 + sw64(8 * nd + 8 * (lm >> 1) + lr, 16 * mh + 8 * (lm & 1)),
                                          pack_bf16(w1[mh][nd][0], w1[mh][nd][1]),
                                          pack_bf16(w1[mh][nd][2], w1[mh][nd][3]),
                                          pack_bf16(w1[mh][nd + 1][0], w1[mh][nd + 1][1]),
                                          pack_bf16(w1[mh][nd + 1][2], w1[mh][nd + 1][3]));
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&tmH1, h0, int((bh * size_t(nblk) + n) * D), s1);
                        tma_store_2d(&tmH2, 0, int((bh * size_t(nblk) + n) * HID + h0), sb + OFF_W2C + h0 * 128);
                        bulk_commit();
                    }
                }
                // ---- Zk = K W1 and Zq = Q W1 (start-of-block W1)
                float zk[4][4], sc[2][4] = {};
#pragma unroll
                for (int j = 0; j < 4; ++j)
#pragma unroll
                    for (int k = 0; k < 4; ++k) zk[j][k] = zq[j][k] = 0.f;
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    uint32_t ka[4], qa[4], kb[4];
                    ldsm_x4(st + S_K + off_a[ks], ka);
                    ldsm_x4(st + S_Q + off_a[ks], qa);
                    ldsm_x4(st + S_K + off_b[ks], kb);
                    mma_bf16_16816(sc[0], qa, kb[0], kb[1]);  // S = Q K^T, keys 0-7
                    mma_bf16_16816(sc[1], qa, kb[2], kb[3]);  //              keys 8-15
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int mh = j >> 1, hf = 2 * (j & 1);
                        const uint32_t b0 = pack_bf16(w1[mh][2 * ks][hf], w1[mh][2 * ks][hf + 1]);
                        const uint32_t b1 = pack_bf16(w1[mh][2 * ks + 1][hf], w1[mh][2 * ks + 1][hf + 1]);
                        mma_bf16_16816(zk[j], ka, b0, b1);
                        mma_bf16_16816(zq[j], qa, b0, b1);
                    }
                }
                // tril (key j <= query i) as the A fragment of tril(Q K^T)(-eta E1)
                sca[0] = pack_bf16(m0 ? sc[0][0] : 0.f, m1 ? sc[0][1] : 0.f);  // (i = g,     j = 2t, 2t + 1)
                sca[1] = pack_bf16(sc[0][2], sc[0][3]);                        // (i = g + 8, j = 2t, 2t + 1)
                sca[2] = 0u;                                                   // (i = g,     j = 8 + 2t ..)
                sca[3] = pack_bf16(m0 ? sc[1][2] : 0.f, m1 ? sc[1][3] : 0.f);  // (i = g + 8, j = 8 + 2t ..)
                // ---- Hk = GELU(Zk), GELU'(Zk); E2^T partial = W2^T Hk^T over this warp's slice
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    hkp[j][0] = pack_bf16(gelu_and_prime(zk[j][0], gp[j][0]), gelu_and_prime(zk[j][1], gp[j][1]));
                    hkp[j][1] = pack_bf16(gelu_and_prime(zk[j][2], gp[j][2]), gelu_and_prime(zk[j][3], gp[j][3]));
                }
                float4* e2p_mine = reinterpret_cast<float4*>(smem + OFF_E2P + warp * 4096);
#pragma unroll
                for (int mo = 0; mo < 4; ++mo) {
                    float e[2][4] = {};
#pragma unroll
                    for (int kh = 0; kh < 2; ++kh) {
                        const uint32_t a[4] = {pack_bf16(w2[mo][2 * kh][0], w2[mo][2 * kh][1]),
                                               pack_bf16(w2[mo][2 * kh][2], w2[mo][2 * kh][3]),
                                               pack_bf16(w2[mo][2 * kh + 1][0], w2[mo][2 * kh + 1][1]),
                                               pack_bf16(w2[mo][2 * kh + 1][2], w2[mo][2 * kh + 1][3])};
                        mma_bf16_16816(e[0], a, hkp[2 * kh][0], hkp[2 * kh + 1][0]);
                        mma_bf16_16816(e[1], a, hkp[2 * kh][1], hkp[2 * kh + 1][1]);
                    }
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt)
                        e2p_mine[(2 * mo + nt) * 32 + lane] = make_float4(e[nt][0], e[nt][1], e[nt][2], e[nt][3]);
                }
            }
            // ---- barrier 1: E2^T partials of this block and read-out partials of the last are written;
            // every read of block n - 1's slot is done, so it takes block n - 1 + NST
            if (bar_compute_any(err)) break;
            if (threadIdx.x == 0 && n >= 1 && issued < nblk) issue(issued++);
            if (have) {
                // E2 = sum of the partials - V; thread f owns accumulator fragment f of the E2^T tile
                const int f = threadIdx.x;
                const int mo = f >> 6, nt = (f >> 5) & 1, l2 = f & 31;
                const int o0 = 16 * mo + (l2 >> 2), k0 = 8 * nt + 2 * (l2 & 3);  // d row, first token
                float4 acc = e2p_all[f];
#pragma unroll
                for (int w = 1; w < NCW; ++w) {
                    const float4 p = e2p_all[w * 256 + f];
                    acc.x += p.x; acc.y += p.y; acc.z += p.z; acc.w += p.w;
                }
                const uint8_t* vt = smem + s * SLOT + S_V;
                const float* et = reinterpret_cast<const float*>(smem + s * SLOT + S_ETA);
                const float e00 = acc.x - bf16_at(vt, k0, o0), e01 = acc.y - bf16_at(vt, k0 + 1, o0);
                const float e10 = acc.z - bf16_at(vt, k0, o0 + 8), e11 = acc.w - bf16_at(vt, k0 + 1, o0 + 8);
                const float n0 = -et[k0], n1 = -et[k0 + 1];
                *reinterpret_cast<uint32_t*>(smem + OFF_E2T + sw16(o0, k0)) = pack_bf16(e00, e01);
                *reinterpret_cast<uint32_t*>(smem + OFF_E2T + sw16(o0 + 8, k0)) = pack_bf16(e10, e11);
                uint8_t* ne = smem + OFF_NE2T + (n & 1) * 2048;
                *reinterpret_cast<uint32_t*>(ne + sw16(o0, k0)) = pack_bf16(n0 * e00, n1 * e01);
                *reinterpret_cast<uint32_t*>(ne + sw16(o0 + 8, k0)) = pack_bf16(n0 * e10, n1 * e11);
            }
            if (n >= 1) {
                // read-out sums of block n - 1: this thread's Z fragment (n-tile = warp) and the scores
                float4 z = zp_all[warp * 32 + lane];
#pragma unroll
                for (int w = 1; w < NCW; ++w) {
                    const float4 p = zp_all[(w * 8 + warp) * 32 + lane];
                    z.x += p.x; z.y += p.y; z.z += p.z; z.w += p.w;
                }
                zsum = z;
                if (threadIdx.x < 64) {
                    const int f = threadIdx.x, nt = f >> 5, l2 = f & 31;
                    const int i0 = l2 >> 2, j0 = 8 * nt + 2 * (l2 & 3);
                    float4 c = sp_all[f];
#pragma unroll
                    for (int w = 1; w < NCW; ++w) {
                        const float4 p = sp_all[w * 64 + f];
                        c.x += p.x; c.y += p.y; c.z += p.z; c.w += p.w;
                    }
                    *reinterpret_cast<uint32_t*>(smem + OFF_S2 + sw16(i0, j0)) =
                        pack_bf16(j0 <= i0 ? c.x : 0.f, j0 + 1 <= i0 ? c.y : 0.f);
                    *reinterpret_cast<uint32_t*>(smem + OFF_S2 + sw16(i0 + 8, j0)) =
                        pack_bf16(j0 <= i0 + 8 ? c.z : 0.f, j0 + 1 <= i0 + 8 ? c.w : 0.f);
                }
            }
            // ---- barrier 2: E2 of this block and the read-out scores of the last are complete
            if (bar_compute_any(err)) break;
            if (n >= 1) {
                // Z of block n - 1 = Hq W2 + tril(Hq Hk^T)(-eta E2), d columns 8 warp .. 8 warp + 7
                uint32_t sa[4], nb0, nb1;
                ldsm_x4(sb + OFF_S2 + sw16(lr + 8 * (lm & 1), 8 * (lm >> 1)), sa);
                ldsm_x2(sb + OFF_NE2T + ((n - 1) & 1) * 2048 + sw16(8 * warp + lr, 8 * (lm & 1)), nb0, nb1);
                float c[4] = {zsum.x, zsum.y, zsum.z, zsum.w};
                mma_bf16_16816(c, sa, nb0, nb1);
                uint32_t* zr = reinterpret_cast<uint32_t*>(Z + (bh * T + size_t(BT) * (n - 1) + g) * D + 8 * warp + 2 * t);
                if (!PART || BT * (n - 1) + g < T) zr[0] = pack_bf16(c[0], c[1]);  // rows past T: not stored
                if (!PART || BT * (n - 1) + g + 8 < T) zr[8 * D / 2] = pack_bf16(c[2], c[3]);
            }
            if (!have) break;

            // ---- E1 = (E2 W2^T) . GELU'(Zk) over this warp's slice, then -eta . E1
            float e1[4][4] = {};
#pragma unroll
            for (int ko = 0; ko < 4; ++ko) {
                uint32_t ea[4];
                ldsm_x4_trans(sb + OFF_E2T + sw16(16 * ko + lr + 8 * (lm >> 1), 8 * (lm & 1)), ea);
#pragma unroll
                for (int jp = 0; jp < 2; ++jp) {
                    uint32_t wb[4];
                    ldsm_x4(sb + OFF_W2C + swz(h0 + 16 * jp + lr + 8 * (lm >> 1), 16 * ko + 8 * (lm & 1)), wb);
                    mma_bf16_16816(e1[2 * jp], ea, wb[0], wb[1]);
                    mma_bf16_16816(e1[2 * jp + 1], ea, wb[2], wb[3]);
                }
            }
            const float* et = reinterpret_cast<const float*>(smem + s * SLOT + S_ETA);
            const float ng = -et[g], ng8 = -et[g + 8];
            uint32_t tr[4][2];  // (-eta E1)^T blocks: [n-tile j][token rows 0-7 / 8-15], transposed
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                tr[j][0] = movt(pack_bf16(ng * e1[j][0] * gp[j][0], ng * e1[j][1] * gp[j][1]));
                tr[j][1] = movt(pack_bf16(ng8 * e1[j][2] * gp[j][2], ng8 * e1[j][3] * gp[j][3]));
            }
            // ---- W1^T += (-eta E1)^T K
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                uint32_t kt[4];
                ldsm_x4_trans(st + S_K + off_a[kk], kt);
#pragma unroll
                for (int mh = 0; mh < 2; ++mh) {
                    const uint32_t a[4] = {tr[2 * mh][0], tr[2 * mh + 1][0], tr[2 * mh][1], tr[2 * mh + 1][1]};
                    mma_bf16_16816(w1[mh][2 * kk], a, kt[0], kt[1]);
                    mma_bf16_16816(w1[mh][2 * kk + 1], a, kt[2], kt[3]);
                }
            }
            // ---- read-out: Zq1 = Q W1 + tril(Q K^T)(-eta E1); Hq = GELU(Zq1)
#pragma unroll
            for (int j = 0; j < 4; ++j) mma_bf16_16816(zq[j], sca, tr[j][0], tr[j][1]);
            uint32_t hq[4][2];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                hq[j][0] = pack_bf16(gelu(zq[j][0]), gelu(zq[j][1]));
                hq[j][1] = pack_bf16(gelu(zq[j][2]), gelu(zq[j][3]));
            }
            // ---- partials over this slice: Hq W2 (start-of-block W2) and Hq Hk^T
            {
                float4* zp_mine = reinterpret_cast<float4*>(smem + OFF_ZP + warp * 4096);
#pragma unroll
                for (int no = 0; no < 8; ++no) {
                    const int mo = no >> 1, hf = 2 * (no & 1);
                    float c[4] = {};
#pragma unroll
                    for (int kh = 0; kh < 2; ++kh) {
                        const uint32_t a[4] = {hq[2 * kh][0], hq[2 * kh][1], hq[2 * kh + 1][0], hq[2 * kh + 1][1]};
                        mma_bf16_16816(c, a, pack_bf16(w2[mo][2 * kh][hf], w2[mo][2 * kh][hf + 1]),
                                       pack_bf16(w2[mo][2 * kh + 1][hf], w2[mo][2 * kh + 1][hf + 1]));
                    }
                    zp_mine[no * 32 + lane] = make_float4(c[0], c[1], c[2], c[3]);
                }
                float4* sp_mine = reinterpret_cast<float4*>(smem + OFF_SP + warp * 1024);
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    float c[4] = {};
#pragma unroll
                    for (int kh = 0; kh < 2; ++kh) {
                        const uint32_t a[4] = {hq[2 * kh][0], hq[2 * kh][1], hq[2 * kh + 1][0], hq[2 * kh + 1][1]};
                        mma_bf16_16816(c, a, hkp[2 * kh][nt], hkp[2 * kh + 1][nt]);
                    }
                    sp_mine[nt * 32 + lane] = make_float4(c[0], c[1], c[2], c[3]);
                }
            }
            // ---- W2^T += (-eta E2)^T Hk, then the bf16 copy of W2 for the next block's E1
            {
                uint32_t ht[4][2];
#pragma unroll
                for (int nh = 0; nh < 4; ++nh) {
                    ht[nh][0] = movt(hkp[nh][0]);
                    ht[nh][1] = movt(hkp[nh][1]);
                }
                const uint32_t ne = sb + OFF_NE2T + (n & 1) * 2048;
#pragma unroll
                for (int mo = 0; mo < 4; ++mo) {
                    uint32_t na[4];
                    ldsm_x4(ne + sw16(16 * mo + lr + 8 * (lm & 1), 8 * (lm >> 1)), na);
#pragma unroll
                    for (int nh = 0; nh < 4; ++nh) mma_bf16_16816(w2[mo][nh], na, ht[nh][0], ht[nh][1]);
                }
            }
            __syncwarp();
            if constexpr (HIST) {  // the block's W2 store has read the bf16 copy before it is rewritten
                if (lane == 0) bulk_wait_read_all();
                __syncwarp();
            }
            store_w2c();
            if constexpr (HIST) fence_proxy_async_smem();  // the next block's TMA store reads the copy
            __syncwarp();
        }
        if constexpr (HIST) {
            if (lane == 0) bulk_wait_all();  // the state stores are complete before the CTA retires
        }

        // final state (fp32)
        float* W1h = W1_out + bh * D * HID;
        float* W2h = W2_out + bh * HID * D;
#pragma unroll
        for (int mh = 0; mh < 2; ++mh)
#pragma unroll
            for (int nd = 0; nd < 8; ++nd)
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    W1h[size_t(8 * nd + 2 * t + (k & 1)) * HID + h0 + 16 * mh + g + 8 * (k >> 1)] = w1[mh][nd][k];
#pragma unroll
        for (int mo = 0; mo < 4; ++mo)
#pragma unroll
            for (int nh = 0; nh < 4; ++nh)
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    W2h[size_t(h0 + 8 * nh + 2 * t + (k & 1)) * D + 16 * mo + g + 8 * (k >> 1)] = w2[mo][nh][k];
    }
    // never retire the CTA with copies in flight (after an early exit; this wait ignores the abort flag)
    if (threadIdx.x == 0)
        for (int m = issued > NST ? issued - NST : 0; m < issued; ++m)
            mbar_wait_bounded(smem_u32(&full_bar[m % NST]), (m / NST) & 1, &s_zero, kWaitLimitNs);
    __syncthreads();
}

}  // namespace

bool mlp_prefill_mma_supported(const MlpArgs& a) {
    // any T (a partial last block weighs its tokens past T by zero); TMA coordinates are int32: the
    // head index, and for the recorded states the rows of W2_hist
    const uint64_t heads = uint64_t(a.B) * a.H;
    return a.bf16 && a.d == D && a.hidden == HID && a.chunk == BT && heads <= 0x7fffffffull &&
           (!a.W1_hist || heads * ((uint64_t(a.T) + BT - 1) / BT) * HID <= 0x7fffffffull);
}

cudaError_t launch_mlp_prefill_mma(const MlpArgs& a, cudaStream_t s, int* status) {
    if (!mlp_prefill_mma_supported(a)) return cudaErrorNotSupported;
    const uint64_t heads = uint64_t(a.B) * a.H;
    CUtensorMap mq, mk, mv, h1, h2;
    cudaError_t e;
    // the 2D maps address rows bh * T + t with an int32 coordinate
    const bool part = a.T % BT || heads * a.T > 0x7fffffffull;
    if (part) {  // [heads][T][D]: the boxes of a partial block read zeros past T
        if ((e = make_tma_map_bf16_heads(&mq, a.Q, heads, a.T, D)) != cudaSuccess) return e;
        if ((e = make_tma_map_bf16_heads(&mk, a.K, heads, a.T, D)) != cudaSuccess) return e;
        if ((e = make_tma_map_bf16_heads(&mv, a.V, heads, a.T, D)) != cudaSuccess) return e;
    } else {  // [heads * T][D]
        if ((e = make_tma_map_bf16(&mq, a.Q, heads * a.T, D)) != cudaSuccess) return e;
        if ((e = make_tma_map_bf16(&mk, a.K, heads * a.T, D)) != cudaSuccess) return e;
        if ((e = make_tma_map_bf16(&mv, a.V, heads * a.T, D)) != cudaSuccess) return e;
    }
    memset(&h1, 0, sizeof(h1));  // unused without the recorded states
    memset(&h2, 0, sizeof(h2));
    if (a.W1_hist) {  // W1_hist as [blocks * d][hidden], W2_hist as [blocks * hidden][d]
        const uint64_t blocks = heads * ((a.T + BT - 1) / BT);
        if ((e = make_tma_map_bf16_box(&h1, a.W1_hist, blocks * D, HID, HS, D, 64)) != cudaSuccess) return e;
        if ((e = make_tma_map_bf16_box(&h2, a.W2_hist, blocks * HID, D, D, HS, 128)) != cudaSuccess) return e;
    }
    auto run = [&](auto kern, int bytes) -> cudaError_t {
        cudaError_t e2 = allow_dynamic_smem(reinterpret_cast<const void*>(kern), bytes);
        if (e2 != cudaSuccess) return e2;
        kern<<<unsigned(a.B) * unsigned(a.H), THREADS, bytes, s>>>(mq, mk, mv, a.eta, a.W1_0, a.W2_0,
                                                                  static_cast<__nv_bfloat16*>(a.Z), a.W1_out,
                                                                  a.W2_out, a.T, h1, h2, status);
        return cudaGetLastError();
    };
    // + 1024 bytes of alignment slack
    if (a.W1_hist)
        return part ? run(mlp_prefill_mma_kernel<true, true>, SMEM_BYTES_HIST + 1024)
                    : run(mlp_prefill_mma_kernel<true, false>, SMEM_BYTES_HIST + 1024);
    return part ? run(mlp_prefill_mma_kernel<false, true>, SMEM_BYTES + 1024)
                : run(mlp_prefill_mma_kernel<false, false>, SMEM_BYTES + 1024);
}

}  // namespace ttt
