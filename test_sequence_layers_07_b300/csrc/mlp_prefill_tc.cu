// mlp_prefill_tc.cu -- tensor-core (tcgen05) TTT-MLP prefill for d = 64, hidden = 256,
// blocks of 16 tokens, bf16 Q/K/V/Z, fp32 state.
//
// What is computed ("Test-Time Training (TTT) Layers for Sequence Modeling",
// section "Variants: TTT-Linear vs. TTT-MLP"; loss, step and readout of
// "Test-Time Training Layers ...", section "The Core Mechanism"; gradients at
// the block start as in the TTT essay's dual-form paragraph).  Per block of 16
// tokens with start state (W1 [64][256], W2 [256][64]):
//   Zk = K W1, Hk = GELU(Zk), E2 = Hk W2 - V, E1 = (E2 W2^T) . GELU'(Zk)
//   Hq = GELU(Q W1 - tril(Q K^T) diag(eta) E1)
//   Z  = Hq W2 - tril(Hq Hk^T) diag(eta) E2
//   W1 <- W1 - K^T diag(eta) E1,   W2 <- W2 - Hk^T diag(eta) E2
//
// Design (ours, for sm_103a):
//  * One CTA per (batch, head).  The fp32 state lives in tensor memory for the
//    whole scan, as the accumulators of the two rank-16 update products
//    (W1^T: 256 lanes x 64 columns as two 128-lane halves; W2: likewise), so
//    the updates are single tcgen05.mma instructions with accumulate on.
//  * Every product runs on tcgen05 with M = 128 (the hidden dimension, or the
//    head dimension stacked over other rows): bf16 operands in shared memory
//    in the 128-byte-swizzled layout TMA writes, fp32 accumulators in TMEM.
//    One operand buffer [W2^T | Hk | pad] serves four products: read K-major
//    it gives Hk W2 (and Hq W2 with the scores Hk Hq^T in rows 64..79 of the
//    same accumulator); read MN-major it gives E2 W2^T and the W2 update.
//  * eta is folded into the error operands (eta.E1, eta.E2), so the causal
//    score operands are plain tril(Q K^T) and tril(Hq Hk^T), and the update
//    products read the TMA tile of K directly (negate bit of the instruction).
//  * The bf16 copies of the state are refreshed from TMEM once per block:
//    W1 as soon as its update has landed (overlapping the Z half of the block),
//    W2 after its last reader.
//  * Eight compute warps: warp w reads TMEM lanes 32(w%4)..+31 of half w/4.
//    Lane 0 of warps 0..3 issue the MMAs (split four ways: one thread issues a
//    tcgen05.mma only every ~85 cycles) and commit to one mbarrier; a ninth warp
//    streams Q/K/V tiles by TMA and eta by a bulk copy into a 4-stage ring.
//  * All waits are bounded; on expiry the kernel records TTT_ERR_TIMEOUT,
//    leaves the loop on every thread at the next barrier, drains its copies
//    and frees its tensor memory.
#include <cuda.h>

#include "ptx.cuh"
#include "tc.cuh"
#include "ttt_common.cuh"
#include "ttt_internal.h"

namespace ttt {
namespace {

using namespace ptx;

constexpr int D = 64, HID = 256, BT = 16;
constexpr int NST = 4;
constexpr int NCW = 8;  // compute warps
constexpr int THREADS = 32 * (NCW + 1);
constexpr uint64_t kWaitLimitNs = 4000000000ull;

// shared memory map (offsets from a 1024-byte aligned base)
constexpr int TILE = BT * D * 2;                 // one [16][64] bf16 tile
constexpr int STAGE = 3 * TILE;                  // K | Q | V
constexpr int OFF_RING = 0;
constexpr int OFF_W2S = NST * STAGE;             // 4 blocks of [128 rows][64]: W2^T rows 0..63, Hk 64..79
constexpr int W2S_BLK = 128 * 128;
constexpr int OFF_W1T = OFF_W2S + 4 * W2S_BLK;   // W1^T [256][64]
constexpr int OFF_E1P = OFF_W1T + HID * 128;     // eta.E1 [16][256] as 4 tiles [16][64]
constexpr int OFF_HQ = OFF_E1P + 4 * TILE;       // Hq [16][256]
constexpr int OFF_E2P = OFF_HQ + 4 * TILE;       // eta.E2 [16][64]
constexpr int OFF_E2 = OFF_E2P + TILE;           // E2 [16][64]
constexpr int OFF_B1 = OFF_E2 + TILE;            // tril(Q K^T)^T, 16 x 16, core-matrix layout
constexpr int OFF_B2 = OFF_B1 + 512;             // tril(Hq Hk^T)^T
constexpr int OFF_ETA = OFF_B2 + 512;            // NST x 16 fp32
constexpr int SMEM_BYTES = OFF_ETA + NST * 64;
static_assert(OFF_W2S % 1024 == 0 && OFF_W1T % 1024 == 0 && OFF_E1P % 1024 == 0 && OFF_HQ % 1024 == 0 &&
                  OFF_E2P % 1024 == 0 && OFF_E2 % 1024 == 0,
              "swizzled operand blocks must be 1024-byte aligned");
// the stacked score product reads 128 rows (16 KB) from any stage base: stay inside the buffer
static_assert((NST - 1) * STAGE + 128 * 128 <= SMEM_BYTES, "score operand overrun");

// tensor-memory columns
constexpr uint32_t TM_W1T = 0;   // W1^T, half h at +64h (lane = hidden % 128, column = d)
constexpr uint32_t TM_W2 = 128;  // W2,   half h at +64h
constexpr uint32_t TM_ZKQ = 256;  // half h at +32h: (K W1)^T in columns 0..15, (Q W1)^T in 16..31 (then the
                                  // layer-1 pre-activation of the read-out)
constexpr uint32_t TM_S1 = 320;  // rows 0..15: K Q^T
constexpr uint32_t TM_P = 336;   // rows 0..63: (Hk W2)^T as four partial sums at +16j
constexpr uint32_t TM_G = 400;   // (E2 W2^T)^T, half h at +16h
constexpr uint32_t TM_ZO = 432;  // rows 0..63: Z^T; rows 64..79: Hk Hq^T; four partial sums at +16j
constexpr uint32_t TM_COLS = 512;

constexpr uint32_t ID_KK16 = tc::make_idesc(128, 16, 0, 0);         // A, B K-major
constexpr uint32_t ID_KK32 = tc::make_idesc(128, 32, 0, 0);         // A, B K-major, N = 32
constexpr uint32_t ID_MK16 = tc::make_idesc(128, 16, 1, 0);         // A MN-major, B K-major
constexpr uint32_t ID_MM64N = tc::make_idesc(128, 64, 1, 1, 0, 1);  // both MN-major, -B
constexpr uint32_t ID_MM16N = tc::make_idesc(128, 16, 1, 1, 0, 1);  // both MN-major, -B

__device__ __forceinline__ uint64_t sw_desc(uint32_t addr, uint32_t lbo) {
    return tc::make_desc(addr, lbo, 1024, tc::kSwizzle128B);
}
// 16 x 16 MN-major core-matrix operand: K groups of 8 rows 256 bytes apart, N groups 128 bytes apart
__device__ __forceinline__ uint64_t core16_desc(uint32_t addr) { return tc::make_desc(addr, 256, 128, tc::kSwizzleNone); }

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

__device__ __forceinline__ void st_bf16(uint8_t* p, float v) {
    *reinterpret_cast<__nv_bfloat16*>(p) = __float2bfloat16_rn(v);
}

// row j (0..15) of a 16 x 16 MN-major core-matrix operand: 16 bf16 values (N index i)
__device__ __forceinline__ void st_core_row(uint8_t* base, int j, const float (&v)[16]) {
    uint4 a, b;
    a.x = pack_bf16(v[0], v[1]); a.y = pack_bf16(v[2], v[3]); a.z = pack_bf16(v[4], v[5]); a.w = pack_bf16(v[6], v[7]);
    b.x = pack_bf16(v[8], v[9]); b.y = pack_bf16(v[10], v[11]); b.z = pack_bf16(v[12], v[13]);
    b.w = pack_bf16(v[14], v[15]);
    uint8_t* r = base + (j >> 3) * 256 + (j & 7) * 16;
    *reinterpret_cast<uint4*>(r) = a;
    *reinterpret_cast<uint4*>(r + 128) = b;
}

__device__ __forceinline__ void bar_compute() { asm volatile("bar.sync 1, %0;" ::"n"(32 * NCW) : "memory"); }

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

__global__ void __launch_bounds__(THREADS, 1)
mlp_prefill_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, const float* __restrict__ eta, const float* W1_0,
                      const float* W2_0, __nv_bfloat16* __restrict__ Z, float* W1_out, float* W2_out, int T,
                      int* status) {
    extern __shared__ uint8_t smem_dyn[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
    __shared__ __align__(8) uint64_t full_bar[NST];
    __shared__ __align__(8) uint64_t empty_bar[NST];
    __shared__ __align__(8) uint64_t mma_bar;
    __shared__ uint32_t s_tmem;
    __shared__ volatile int s_err;   // set by any thread that saw a wait expire: speeds up the others' aborts
    __shared__ volatile int s_zero;  // never set: abort flag of the waits that must run to completion

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const size_t bh = blockIdx.x;
    const int nblk = T / BT;
    const uint32_t sb = smem_u32(smem);

    if (tid == 0) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(smem_u32(&full_bar[s]), 1);
            mbar_init(smem_u32(&empty_bar[s]), 1);
        }
        mbar_init(smem_u32(&mma_bar), 4);  // one commit per MMA issuer
        s_err = 0;
        s_zero = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tc::tmem_alloc(smem_u32(&s_tmem), TM_COLS);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tm = s_tmem;

    if (warp == NCW) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            prefetch_tensormap(&tmQ);
            prefetch_tensormap(&tmK);
            prefetch_tensormap(&tmV);
            int issued = 0;
            for (int n = 0; n < nblk; ++n) {
                const int s = n % NST;
                if (n >= NST) {
                    if (s_err ||
                        !mbar_wait_bounded(smem_u32(&empty_bar[s]), ((n / NST) - 1) & 1, &s_err, kWaitLimitNs)) {
                        if (!s_err) record_status(status, kStatusTimeout);
                        s_err = 1;
                        break;
                    }
                }
                const uint32_t fb = smem_u32(&full_bar[s]);
                mbar_arrive_expect_tx(fb, STAGE + 64);
                const uint32_t st = sb + OFF_RING + s * STAGE;
                const int y = int(bh * T) + BT * n;
                tma_load_2d(st, &tmK, 0, y, fb);
                tma_load_2d(st + TILE, &tmQ, 0, y, fb);
                tma_load_2d(st + 2 * TILE, &tmV, 0, y, fb);
                bulk_load(sb + OFF_ETA + s * 64, eta + bh * T + BT * n, 64, fb);
                ++issued;
            }
            // never retire with copies in flight (this wait ignores the abort flag)
            for (int n = issued > NST ? issued - NST : 0; n < issued; ++n)
                mbar_wait_bounded(smem_u32(&full_bar[n % NST]), (n / NST) & 1, &s_zero, kWaitLimitNs);
        }
    } else {
        // ------------------------------------------------------------ compute warps
        const int h = warp >> 2, q = warp & 3;
        const int hid = 128 * h + 32 * q + lane;  // hidden unit of this thread's TMEM lane
        const uint32_t tl = tm + (uint32_t(32 * q) << 16);  // this warp's lane quadrant
        const int hb = hid >> 6, hc = hid & 63;

        // initial state -> TMEM (fp32) and the bf16 operand copies
        {
            const float* w1 = W1_0 + bh * D * HID;
            const float* w2 = W2_0 + bh * HID * D;
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 16) {
                float v[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) v[i] = w1[(c0 + i) * HID + hid];
                tc::st16(tl + TM_W1T + 64 * h + c0, v);
                uint4 a, b;
                a.x = pack_bf16(v[0], v[1]); a.y = pack_bf16(v[2], v[3]);
                a.z = pack_bf16(v[4], v[5]); a.w = pack_bf16(v[6], v[7]);
                b.x = pack_bf16(v[8], v[9]); b.y = pack_bf16(v[10], v[11]);
                b.z = pack_bf16(v[12], v[13]); b.w = pack_bf16(v[14], v[15]);
                *reinterpret_cast<uint4*>(smem + OFF_W1T + tc::sw128(hid, c0)) = a;
                *reinterpret_cast<uint4*>(smem + OFF_W1T + tc::sw128(hid, c0 + 8)) = b;
#pragma unroll
                for (int i = 0; i < 16; i += 4) {
                    const float4 f = *reinterpret_cast<const float4*>(w2 + size_t(hid) * D + c0 + i);
                    v[i] = f.x; v[i + 1] = f.y; v[i + 2] = f.z; v[i + 3] = f.w;
                }
                tc::st16(tl + TM_W2 + 64 * h + c0, v);
#pragma unroll
                for (int i = 0; i < 16; ++i) st_bf16(smem + OFF_W2S + hb * W2S_BLK + tc::sw128(c0 + i, hc), v[i]);
            }
            // rows 64..127 of the stacked W2 operand (Hk and padding) start at zero
            for (int i = tid; i < 4 * 64 * 8; i += 32 * NCW) {
                const int blk = i >> 9, r = 64 + ((i >> 3) & 63), ch = i & 7;
                *reinterpret_cast<uint4*>(smem + OFF_W2S + blk * W2S_BLK + r * 128 + ch * 16) = make_uint4(0, 0, 0, 0);
            }
            tc::st_wait();
        }
        tc::fence_async_smem();
        tc::fence_before_sync();
        bar_compute();

        // Error protocol: `err` is this thread's own view; the loop is left only on the
        // OR of every compute thread's view, taken by a reducing barrier, so all
        // compute threads leave at the same barrier.
        uint32_t mph = 0;
        bool err = false;
        auto fail = [&]() {
            if (!s_err) record_status(status, kStatusTimeout);
            s_err = 1;
            err = true;
        };
        auto wait_mma = [&]() -> bool {
            const bool ok = !err && mbar_wait_bounded(smem_u32(&mma_bar), mph, &s_err, kWaitLimitNs);
            mph ^= 1;
            if (!ok) fail();
            tc::fence_after_sync();
            return __all_sync(0xffffffffu, ok);  // warp-uniform: the TMEM loads that follow are warp-wide
        };
        auto end_stage = [&]() -> bool {
            tc::fence_async_smem();
            tc::fence_before_sync();
            return bar_compute_any(err);
        };

        const uint32_t w2s = sb + OFF_W2S, w1t = sb + OFF_W1T;
        // Four MMA issuers (lane 0 of warps 0..3, one per SM sub-partition): one thread
        // issues a tcgen05.mma only every ~85 cycles, so each stage's products are split
        // over four threads, with the long contractions (K = 256) cut into four partial
        // accumulators that the epilogue adds in a fixed order (deterministic).
        const bool issuer = lane == 0 && warp < 4;
        const int r = warp;  // issuer index

        // per-thread 16-byte chunk offsets of the swizzled layout for this thread's column
        // (hidden unit hc of a 64-wide block): element (row, hc) lives at row*128 + xo[row & 7]
        uint32_t xo[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) xo[i] = uint32_t((((hc >> 3) ^ i) << 4) + ((hc & 7) << 1));
        // the head-dimension column of the epilogues over d (warps 0,1 of either half)
        const int dd = 32 * (q & 1) + lane;
        uint32_t xd[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) xd[i] = uint32_t((((dd >> 3) ^ i) << 4) + ((dd & 7) << 1));
        const bool dwarp = q < 2;  // warps 0, 1, 4, 5 read TMEM lanes 0..63 (the head dimension)
        const int t0 = 8 * h;      // ...and split the 16 token columns between the halves

        for (int n = 0; n < nblk; ++n) {
            const int s = n % NST;
            const uint32_t st = sb + OFF_RING + s * STAGE;
            const uint8_t* stp = smem + OFF_RING + s * STAGE;
            if (!mbar_wait_bounded(smem_u32(&full_bar[s]), (n / NST) & 1, &s_err, kWaitLimitNs)) fail();
            float et[16];
#pragma unroll
            for (int i = 0; i < 16; i += 4) {
                const float4 f = *reinterpret_cast<const float4*>(smem + OFF_ETA + s * 64 + 4 * i);
                et[i] = f.x; et[i + 1] = f.y; et[i + 2] = f.z; et[i + 3] = f.w;
            }

            // ---- S1: (K W1)^T | (Q W1)^T per half (the K and Q tiles are adjacent: N = 32), K Q^T
            if (issuer && !err) {
                tc::fence_after_sync();
                if (r < 2) {
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        tc::mma(tm + TM_ZKQ + 32 * r, sw_desc(w1t + r * 128 * 128 + ks * 32, 16),
                                sw_desc(st + ks * 32, 16), ID_KK32, ks > 0);
                } else if (r == 2) {
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        tc::mma(tm + TM_S1, sw_desc(st + ks * 32, 16), sw_desc(st + TILE + ks * 32, 16), ID_KK16,
                                ks > 0);
                }
                tc::commit(smem_u32(&mma_bar));
            }
            __syncwarp();
            float gp[16];
            if (wait_mma()) {
                float zk[16], s1[16];
                tc::ld16(tl + TM_ZKQ + 32 * h, zk);
                if (warp == 0) tc::ld16(tl + TM_S1, s1);
                tc::ld_wait();
                uint8_t* hk = smem + OFF_W2S + hb * W2S_BLK + 64 * 128;
#pragma unroll
                for (int t = 0; t < 16; ++t) st_bf16(hk + t * 128 + xo[t & 7], gelu_and_prime(zk[t], gp[t]));
                if (warp == 0 && lane < 16) {
                    float rr[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) rr[i] = i >= lane ? s1[i] : 0.f;
                    st_core_row(smem + OFF_B1, lane, rr);
                }
            }
            if (end_stage()) break;

            // ---- S2: (Hk W2)^T, K = 256 split into four partial accumulators
            if (issuer) {
                tc::fence_after_sync();
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint32_t o = r * W2S_BLK + kk * 32;
                    tc::mma(tm + TM_P + 16 * r, sw_desc(w2s + o, 16), sw_desc(w2s + o + 64 * 128, 16), ID_KK16, kk > 0);
                }
                tc::commit(smem_u32(&mma_bar));
            }
            __syncwarp();
            if (wait_mma() && dwarp) {
                float p[8], pp[8];
                tc::ld8(tl + TM_P + t0, p);
#pragma unroll
                for (int j = 1; j < 4; ++j) {
                    tc::ld8(tl + TM_P + 16 * j + t0, pp);
                    tc::ld_wait();
#pragma unroll
                    for (int i = 0; i < 8; ++i) p[i] += pp[i];
                }
                float v[8];
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    v[i] = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(stp + 2 * TILE + (t0 + i) * 128 +
                                                                                    xd[(t0 + i) & 7]));
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int t = t0 + i;
                    const float e = p[i] - v[i];
                    st_bf16(smem + OFF_E2 + t * 128 + xd[t & 7], e);
                    st_bf16(smem + OFF_E2P + t * 128 + xd[t & 7], et[t] * e);
                }
            }
            if (end_stage()) break;

            // ---- S3: (E2 W2^T)^T per half (issuers 0, 1) and the W2 update W2 += Hk^T (-eta.E2) (issuers 2, 3)
            if (issuer) {
                tc::fence_after_sync();
                if (r < 2) {
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        tc::mma(tm + TM_G + 16 * r, sw_desc(w2s + 2 * r * W2S_BLK + ks * 2048, W2S_BLK),
                                sw_desc(sb + OFF_E2 + ks * 32, 16), ID_MK16, ks > 0);
                } else {
                    const int hh = r - 2;
                    tc::mma(tm + TM_W2 + 64 * hh, sw_desc(w2s + 2 * hh * W2S_BLK + 64 * 128, W2S_BLK),
                            sw_desc(sb + OFF_E2P, TILE), ID_MM64N, 1);
                }
                tc::commit(smem_u32(&mma_bar));
            }
            __syncwarp();
            if (wait_mma()) {
                float g[16];
                tc::ld16(tl + TM_G + 16 * h, g);
                tc::ld_wait();
                uint8_t* e1 = smem + OFF_E1P + hb * TILE;
#pragma unroll
                for (int t = 0; t < 16; ++t) st_bf16(e1 + t * 128 + xo[t & 7], et[t] * g[t] * gp[t]);
            }
            if (end_stage()) break;

            // ---- S4: read-out layer 1 with the causal delta (issuers 0, 1) and the W1 update
            //      W1^T += (eta.E1)^T (-K) (issuers 2, 3)
            if (issuer) {
                tc::fence_after_sync();
                const int hh = r & 1;
                const uint64_t a = sw_desc(sb + OFF_E1P + 2 * hh * TILE, TILE);
                if (r < 2)
                    tc::mma(tm + TM_ZKQ + 32 * hh + 16, a, core16_desc(sb + OFF_B1), ID_MM16N, 1);
                else
                    tc::mma(tm + TM_W1T + 64 * hh, a, sw_desc(st, TILE), ID_MM64N, 1);
                tc::commit(smem_u32(&mma_bar));
            }
            __syncwarp();
            if (wait_mma()) {
                float zq[16];
                tc::ld16(tl + TM_ZKQ + 32 * h + 16, zq);
                tc::ld_wait();
                uint8_t* hq = smem + OFF_HQ + hb * TILE;
#pragma unroll
                for (int t = 0; t < 16; ++t) st_bf16(hq + t * 128 + xo[t & 7], gelu(zq[t]));
                // the W1 update has landed: refresh its bf16 copy (row hid) for the next block
                uint8_t* w1row = smem + OFF_W1T + hid * 128;
#pragma unroll
                for (int c0 = 0; c0 < D; c0 += 16) {
                    float w[16];
                    tc::ld16(tl + TM_W1T + 64 * h + c0, w);
                    tc::ld_wait();
                    uint4 a, b;
                    a.x = pack_bf16(w[0], w[1]); a.y = pack_bf16(w[2], w[3]);
                    a.z = pack_bf16(w[4], w[5]); a.w = pack_bf16(w[6], w[7]);
                    b.x = pack_bf16(w[8], w[9]); b.y = pack_bf16(w[10], w[11]);
                    b.z = pack_bf16(w[12], w[13]); b.w = pack_bf16(w[14], w[15]);
                    *reinterpret_cast<uint4*>(w1row + ((((c0 >> 3) ^ hid) & 7) << 4)) = a;
                    *reinterpret_cast<uint4*>(w1row + (((((c0 >> 3) + 1) ^ hid) & 7) << 4)) = b;
                }
            }
            if (end_stage()) break;

            // ---- S5: (Hq W2)^T in rows 0..63 and Hk Hq^T in rows 64..79, K = 256 in four partials
            if (issuer) {
                tc::fence_after_sync();
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    tc::mma(tm + TM_ZO + 16 * r, sw_desc(w2s + r * W2S_BLK + kk * 32, 16),
                            sw_desc(sb + OFF_HQ + r * TILE + kk * 32, 16), ID_KK16, kk > 0);
                tc::commit(smem_u32(&mma_bar));
            }
            __syncwarp();
            if (wait_mma()) {
                if (warp == 2) {
                    float s2[16], sp[16];
                    tc::ld16(tl + TM_ZO, s2);
#pragma unroll
                    for (int j = 1; j < 4; ++j) {
                        tc::ld16(tl + TM_ZO + 16 * j, sp);
                        tc::ld_wait();
#pragma unroll
                        for (int i = 0; i < 16; ++i) s2[i] += sp[i];
                    }
                    if (lane < 16) {
                        float rr[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) rr[i] = i >= lane ? s2[i] : 0.f;
                        st_core_row(smem + OFF_B2, lane, rr);
                    }
                }
                // W2's last reader of this block has finished: refresh its bf16 copy (column hc of W2^T)
                uint8_t* w2c = smem + OFF_W2S + hb * W2S_BLK;
#pragma unroll
                for (int c0 = 0; c0 < D; c0 += 16) {
                    float w[16];
                    tc::ld16(tl + TM_W2 + 64 * h + c0, w);
                    tc::ld_wait();
#pragma unroll
                    for (int i = 0; i < 16; ++i) st_bf16(w2c + (c0 + i) * 128 + xo[i & 7], w[i]);
                }
            }
            if (end_stage()) break;

            // ---- S6: Z^T += (eta.E2)^T (-tril(Hq Hk^T)^T), into partial 0
            if (issuer) {
                tc::fence_after_sync();
                if (r == 0) tc::mma(tm + TM_ZO, sw_desc(sb + OFF_E2P, TILE), core16_desc(sb + OFF_B2), ID_MM16N, 1);
                tc::commit(smem_u32(&mma_bar));
            }
            __syncwarp();
            if (wait_mma() && dwarp) {
                float z[8], zp[8];
                tc::ld8(tl + TM_ZO + t0, z);
#pragma unroll
                for (int j = 1; j < 4; ++j) {
                    tc::ld8(tl + TM_ZO + 16 * j + t0, zp);
                    tc::ld_wait();
#pragma unroll
                    for (int i = 0; i < 8; ++i) z[i] += zp[i];
                }
                __nv_bfloat16* zo = Z + (bh * T + size_t(BT) * n + t0) * D + dd;
#pragma unroll
                for (int i = 0; i < 8; ++i) zo[i * D] = __float2bfloat16_rn(z[i]);
            }
            const bool stop = end_stage();
            if (tid == 0) mbar_arrive(smem_u32(&empty_bar[s]));
            if (stop) break;
        }

        // every MMA this CTA issued has completed before the state is read and TMEM freed
        if (issuer) {
            tc::commit(smem_u32(&mma_bar));
        }
        if (tid == 0) mbar_wait_bounded(smem_u32(&mma_bar), mph, &s_zero, kWaitLimitNs);
        bar_compute();
        tc::fence_after_sync();

        // final state
        {
            float* w1 = W1_out + bh * D * HID;
            float* w2 = W2_out + bh * HID * D;
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 16) {
                float v[16];
                tc::ld16(tl + TM_W1T + 64 * h + c0, v);
                tc::ld_wait();
#pragma unroll
                for (int i = 0; i < 16; ++i) w1[(c0 + i) * HID + hid] = v[i];
                tc::ld16(tl + TM_W2 + 64 * h + c0, v);
                tc::ld_wait();
#pragma unroll
                for (int i = 0; i < 16; i += 4)
                    *reinterpret_cast<float4*>(w2 + size_t(hid) * D + c0 + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
            }
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tm, TM_COLS);
    }
}

}  // namespace

bool mlp_prefill_tc_supported(const MlpArgs& a) {
    return a.bf16 && a.d == D && a.hidden == HID && a.chunk == BT && a.T % BT == 0 &&
           uint64_t(a.B) * a.H * a.T <= 0x7fffffffull;
}

cudaError_t launch_mlp_prefill_tc(const MlpArgs& a, cudaStream_t s, int* status) {
    if (!mlp_prefill_tc_supported(a)) return cudaErrorNotSupported;
    const uint64_t rows = uint64_t(a.B) * a.H * a.T;
    CUtensorMap mq, mk, mv;
    cudaError_t e;
    if ((e = make_tma_map_bf16(&mq, a.Q, rows, D)) != cudaSuccess) return e;
    if ((e = make_tma_map_bf16(&mk, a.K, rows, D)) != cudaSuccess) return e;
    if ((e = make_tma_map_bf16(&mv, a.V, rows, D)) != cudaSuccess) return e;
    const int bytes = SMEM_BYTES + 1024;
    if ((e = allow_dynamic_smem(reinterpret_cast<const void*>(mlp_prefill_tc_kernel), bytes)) !=
        cudaSuccess)
        return e;
    mlp_prefill_tc_kernel<<<unsigned(a.B) * unsigned(a.H), THREADS, bytes, s>>>(
        mq, mk, mv, a.eta, a.W1_0, a.W2_0, static_cast<__nv_bfloat16*>(a.Z), a.W1_out, a.W2_out, a.T, status);
    return cudaGetLastError();
}

}  // namespace ttt
