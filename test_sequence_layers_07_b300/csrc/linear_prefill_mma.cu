// linear_prefill_mma.cu -- tensor-core TTT-Linear prefill (bf16 Q/K/V/Z, fp32 state).
//
// What is computed ("Test-Time Training Layers ...", sections "The Core
// Mechanism" and "Hardware Parallelization"; TTT essay, paragraph on the dual
// form): per block of b tokens with start state W0,
//     E = K W0 - V;  Z = Q W0 - tril(eta . Q K^T) E;  W = W0 - K^T diag(eta) E.
//
// Design (ours, for sm_103a):
//  * The scan over blocks is a chain of small dependent steps (16 x d x d per
//    16 tokens), so it is latency-bound, not FLOP- or byte-bound.  The state
//    therefore never leaves the register file: each consumer warp owns 16
//    output columns of W, held transposed (W^T, 16 x d, fp32) in the
//    accumulator layout of the warp-level m16n8k16 bf16 MMA.  That layout is
//    also the A-operand layout after an fp32->bf16 pack, so every product with
//    the state (K W0, Q W, and the rank-16 update K^T diag(eta) E accumulated
//    straight into W) runs with no shared-memory round trip.
//  * For f = kW the output columns of W, E and Z depend only on the same
//    columns of W0 and V, so column groups run independently (CG warps per
//    CTA, D/16/CG CTAs per head); each warp recomputes the 16x16 Q K^T tile.
//  * A block of b = 16*nsub tokens is processed as nsub sub-blocks of 16:
//    E of every sub-block uses the block-start state (bf16 copy kept in
//    registers), while the read-out state W_run accumulates the updates of the
//    earlier sub-blocks, which gives exactly Z = Q W0 - tril(eta.QK^T) E
//    without ever forming the b x b matrix.
//  * Everything of a sub-block that does not depend on the state (operand
//    fragments, the masked Q K^T scores, -eta and eta*V) is prepared one
//    sub-block ahead, under the MMA latency of the current one.
//  * One producer warp streams 16-token Q/K/V tiles with TMA tensor copies
//    (128-byte swizzle, so ldmatrix reads are bank-conflict free) and eta with
//    a bulk copy, into an NST-stage ring guarded by mbarriers.  All waits are
//    bounded; on expiry the kernel records TTT_ERR_TIMEOUT and drains.
//  * Z leaves through stmatrix.trans into a small per-warp staging tile and
//    16-byte stores (32-byte row segments), with no CTA-wide barrier.
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

template <int D>
__device__ __forceinline__ void pack_state(const float (&w)[D / 8][4], uint32_t (&wa)[D / 16][4]) {
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
        wa[ks][0] = pack_bf16(w[2 * ks][0], w[2 * ks][1]);
        wa[ks][1] = pack_bf16(w[2 * ks][2], w[2 * ks][3]);
        wa[ks][2] = pack_bf16(w[2 * ks + 1][0], w[2 * ks + 1][1]);
        wa[ks][3] = pack_bf16(w[2 * ks + 1][2], w[2 * ks + 1][3]);
    }
}

template <int D, int CG, int NST>
struct MmaCfg {
    static constexpr int TILE = 16 * D * 2;  // bytes of a [16][D] bf16 tile
    static constexpr int STAGE = 3 * TILE;   // Q, K, V
    static constexpr int ZBUF_OFF = NST * STAGE;
    static constexpr int ETA_OFF = ZBUF_OFF + CG * 512;  // per-warp [16][16] Z staging
    static constexpr int BYTES = ETA_OFF + NST * 64;
    static constexpr int THREADS = 32 * (CG + 1);
};

template <int D, int CG, int NST, bool SINGLE>
__global__ void __launch_bounds__(32 * (CG + 1), 1)
linear_prefill_mma_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                          const __grid_constant__ CUtensorMap tmV, const float* __restrict__ eta,
                          const float* W0, __nv_bfloat16* __restrict__ Z, float* W_out, int T, int chunk,
                          int* status) {
    using C = MmaCfg<D, CG, NST>;
    constexpr int KS = D / 16;  // k-steps over the input dimension
    constexpr int NT = D / 8;   // 8-wide n-tiles of the state over the input dimension

    extern __shared__ uint8_t smem_dyn[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
    __shared__ __align__(8) uint64_t full_bar[NST];
    __shared__ __align__(8) uint64_t empty_bar[NST];
    __shared__ volatile int s_err;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const size_t bh = blockIdx.x;
    const int nsb = T / 16;       // 16-token sub-blocks
    const int nsub = chunk / 16;  // sub-blocks per block
    const uint32_t sbase = smem_u32(smem);

    if (threadIdx.x == 0) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(smem_u32(&full_bar[s]), 1);
            mbar_init(smem_u32(&empty_bar[s]), CG);
        }
        s_err = 0;
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            prefetch_tensormap(&tmQ);
            prefetch_tensormap(&tmK);
            prefetch_tensormap(&tmV);
            int issued = 0;
            for (int sb = 0; sb < nsb; ++sb) {
                const int s = sb % NST;
                if (sb >= NST) {
                    if (s_err ||
                        !mbar_wait_bounded(smem_u32(&empty_bar[s]), ((sb / NST) - 1) & 1, &s_err, kWaitLimitNs)) {
                        if (!s_err) record_status(status, kStatusTimeout);
                        s_err = 1;
                        break;
                    }
                }
                const uint32_t fb = smem_u32(&full_bar[s]);
                mbar_arrive_expect_tx(fb, 3 * C::TILE + 64);
                const uint32_t st = sbase + s * C::STAGE;
                const int y = int(bh * T) + 16 * sb;
#pragma unroll
                for (int box = 0; box < D / 64; ++box) {
                    tma_load_2d(st + box * 2048, &tmQ, 64 * box, y, fb);
                    tma_load_2d(st + C::TILE + box * 2048, &tmK, 64 * box, y, fb);
                    tma_load_2d(st + 2 * C::TILE + box * 2048, &tmV, 64 * box, y, fb);
                }
                bulk_load(sbase + C::ETA_OFF + s * 64, eta + bh * T + 16 * sb, 64, fb);
                ++issued;
            }
            // never retire the CTA with copies in flight: wait (bounded) for the last stages
            for (int sb = issued > NST ? issued - NST : 0; sb < issued; ++sb)
                mbar_wait_bounded(smem_u32(&full_bar[sb % NST]), (sb / NST) & 1, &s_err, kWaitLimitNs);
        }
    } else {
        // ------------------------------------------------------------ consumers
        const int cw0 = (blockIdx.y * CG + (warp - 1)) * 16;  // first output column of this warp
        const int g = lane >> 2, t = lane & 3;
        const int lj = lane >> 3, lr = lane & 7;

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
        uint32_t wa0[KS][4];                  // bf16 copy of the block-start state (A operand)
        constexpr bool kHoistKt = (D <= 64);  // keep register pressure in check for D = 128

        // lane-dependent ldmatrix coordinates (byte offsets inside a stage tile)
        uint32_t off_nk[KS], off_tk[NT / 2];
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) off_nk[ks] = swz(lr + 8 * (lj >> 1), 16 * ks + 8 * (lj & 1));
#pragma unroll
        for (int kk = 0; kk < NT / 2; ++kk) off_tk[kk] = swz(lr + 8 * (lj & 1), 16 * kk + 8 * (lj >> 1));
        const uint32_t off_v = swz(lr + 8 * (lj >> 1), cw0 + 8 * (lj & 1));
        // per-warp Z staging tile [16 tokens][16 columns] bf16 (rows of 32 bytes, halves swapped
        // on rows 4..7 mod 8 to spread banks) and this lane's store coordinates
        const uint32_t zst = sbase + C::ZBUF_OFF + (warp - 1) * 512;
        const uint32_t zst_w = zst + (lr + 8 * (lj >> 1)) * 32 + (((lj & 1) ^ ((lr >> 2) & 1)) << 4);
        const int zrow = lane >> 1, zhalf = lane & 1;
        const uint32_t zst_r = zst + zrow * 32 + ((zhalf ^ ((zrow >> 2) & 1)) << 4);
        __nv_bfloat16* zp = Z + (bh * T + zrow) * D + cw0 + 8 * zhalf;
        const bool m0 = 2 * t <= g, m1 = 2 * t + 1 <= g;  // causal mask of the diagonal 8x8 blocks

        // State-independent work of a sub-block, prepared one sub-block ahead:
        // operand fragments, the masked scores, -eta and eta*v.
        uint32_t kb[KS][4], qb[KS][4], kt[kHoistKt ? NT / 2 : 1][4];
        uint32_t sz00 = 0, sz10 = 0, sz11 = 0;  // masked S as B operands of the Z product
        float ne0 = 0, ne1 = 0, ne2 = 0, ne3 = 0, nv[8] = {};
        auto prepare = [&](int sb, uint32_t st) -> bool {
            const int s = sb % NST;
            if (!mbar_wait_bounded(smem_u32(&full_bar[s]), (sb / NST) & 1, &s_err, kWaitLimitNs)) return false;
            const uint32_t kb_ = st + C::TILE, vb_ = st + 2 * C::TILE;
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                ldsm_x4(kb_ + off_nk[ks], kb[ks]);
                ldsm_x4(st + off_nk[ks], qb[ks]);
            }
            uint32_t vv[4];
            ldsm_x4_trans(vb_ + off_v, vv);
            if constexpr (kHoistKt) {
#pragma unroll
                for (int kk = 0; kk < NT / 2; ++kk) ldsm_x4_trans(kb_ + off_tk[kk], kt[kk]);
            }
            const float* es = reinterpret_cast<const float*>(smem + C::ETA_OFF + s * 64);
            const float2 e01 = *reinterpret_cast<const float2*>(es + 2 * t);
            const float2 e23 = *reinterpret_cast<const float2*>(es + 8 + 2 * t);
            float sc[2][4] = {};
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                const uint32_t qa[4] = {qb[ks][0], qb[ks][2], qb[ks][1], qb[ks][3]};
                mma_bf16_16816(sc[0], qa, kb[ks][0], kb[ks][1]);
                mma_bf16_16816(sc[1], qa, kb[ks][2], kb[ks][3]);
            }
            sz00 = pack_bf16(m0 ? sc[0][0] : 0.f, m1 ? sc[0][1] : 0.f);
            sz10 = pack_bf16(sc[0][2], sc[0][3]);
            sz11 = pack_bf16(m0 ? sc[1][2] : 0.f, m1 ? sc[1][3] : 0.f);
            ne0 = -e01.x; ne1 = -e01.y; ne2 = -e23.x; ne3 = -e23.y;
            nv[0] = e01.x * bf16_lo(vv[0]); nv[1] = e01.y * bf16_hi(vv[0]);
            nv[2] = e01.x * bf16_lo(vv[1]); nv[3] = e01.y * bf16_hi(vv[1]);
            nv[4] = e23.x * bf16_lo(vv[2]); nv[5] = e23.y * bf16_hi(vv[2]);
            nv[6] = e23.x * bf16_lo(vv[3]); nv[7] = e23.y * bf16_hi(vv[3]);
            return true;
        };

        bool ok = !s_err && prepare(0, sbase);
        int sub = 0;  // sub-block index inside the current block
        for (int sb = 0; ok && sb < nsb; ++sb) {
            const int s = sb % NST;
            const uint32_t st = sbase + s * C::STAGE;

            if (SINGLE || sub == 0) pack_state<D>(w, wa0);
            uint32_t war[SINGLE ? 1 : KS][4];
            if constexpr (!SINGLE) pack_state<D>(w, war);

            // P^T = W0^T K^T (two accumulators per n-tile halve the dependent chain), QW^T = W^T Q^T
            float pe[2][4] = {}, po[2][4] = {}, qw[2][4] = {};
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                float(&pa)[2][4] = (ks & 1) ? po : pe;
                mma_bf16_16816(pa[0], wa0[ks], kb[ks][0], kb[ks][1]);
                mma_bf16_16816(pa[1], wa0[ks], kb[ks][2], kb[ks][3]);
                const uint32_t(&wq)[4] = SINGLE ? wa0[ks] : war[SINGLE ? 0 : ks];
                mma_bf16_16816(qw[0], wq, qb[ks][0], qb[ks][1]);
                mma_bf16_16816(qw[1], wq, qb[ks][2], qb[ks][3]);
            }
            // G = -eta . (P - V)^T  as a bf16 A operand (rows c, cols token j)
            uint32_t ga[4];
            ga[0] = pack_bf16(fmaf(ne0, pe[0][0] + po[0][0], nv[0]), fmaf(ne1, pe[0][1] + po[0][1], nv[1]));
            ga[1] = pack_bf16(fmaf(ne0, pe[0][2] + po[0][2], nv[2]), fmaf(ne1, pe[0][3] + po[0][3], nv[3]));
            ga[2] = pack_bf16(fmaf(ne2, pe[1][0] + po[1][0], nv[4]), fmaf(ne3, pe[1][1] + po[1][1], nv[5]));
            ga[3] = pack_bf16(fmaf(ne2, pe[1][2] + po[1][2], nv[6]), fmaf(ne3, pe[1][3] + po[1][3], nv[7]));

            // W^T += G K   (rank-16 update of the running state, fp32 accumulate)
#pragma unroll
            for (int kk = 0; kk < NT / 2; ++kk) {
                if constexpr (kHoistKt) {
                    mma_bf16_16816(w[2 * kk], ga, kt[kk][0], kt[kk][1]);
                    mma_bf16_16816(w[2 * kk + 1], ga, kt[kk][2], kt[kk][3]);
                } else {
                    uint32_t k2[4];
                    ldsm_x4_trans(st + C::TILE + off_tk[kk], k2);
                    mma_bf16_16816(w[2 * kk], ga, k2[0], k2[1]);
                    mma_bf16_16816(w[2 * kk + 1], ga, k2[2], k2[3]);
                }
            }
            // Z^T = QW^T + G * S_masked
            mma_bf16_16816(qw[0], ga, sz00, 0u);
            mma_bf16_16816(qw[1], ga, sz10, sz11);
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&empty_bar[s]));  // stage fully read

            if (!SINGLE) sub = (sub + 1 == nsub) ? 0 : sub + 1;
            // next sub-block's state-independent work overlaps this one's MMA latency
            if (sb + 1 < nsb) {
                if (s_err) {
                    ok = false;
                } else if (!prepare(sb + 1, sbase + ((sb + 1) % NST) * C::STAGE)) {
                    if (!s_err) record_status(status, kStatusTimeout);
                    s_err = 1;
                    ok = false;
                }
            }
            // Z: stmatrix.trans into the warp's staging tile, one 16-byte store per lane
            stsm_x4_trans(zst_w, pack_bf16(qw[0][0], qw[0][1]), pack_bf16(qw[0][2], qw[0][3]),
                          pack_bf16(qw[1][0], qw[1][1]), pack_bf16(qw[1][2], qw[1][3]));
            __syncwarp();
            uint4 v;
            asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                         : "r"(zst_r)
                         : "memory");
            *reinterpret_cast<uint4*>(zp) = v;
            zp += 16 * D;
            __syncwarp();
        }
        if (!ok && !s_err) {
            record_status(status, kStatusTimeout);
            s_err = 1;
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

template <int D, int CG, int NST, bool SINGLE>
cudaError_t launch_cfg(const LinearArgs& a, cudaStream_t s, int* status) {
    using C = MmaCfg<D, CG, NST>;
    const uint64_t rows = uint64_t(a.B) * a.H * a.T;
    CUtensorMap mq, mk, mv;
    cudaError_t e;
    if ((e = make_tma_map_bf16(&mq, a.Q, rows, D)) != cudaSuccess) return e;
    if ((e = make_tma_map_bf16(&mk, a.K, rows, D)) != cudaSuccess) return e;
    if ((e = make_tma_map_bf16(&mv, a.V, rows, D)) != cudaSuccess) return e;
    auto kern = linear_prefill_mma_kernel<D, CG, NST, SINGLE>;
    const int bytes = C::BYTES + 1024;  // + alignment slack
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes)) != cudaSuccess) return e;
    dim3 grid(unsigned(a.B) * unsigned(a.H), D / 16 / CG);
    kern<<<grid, C::THREADS, bytes, s>>>(mq, mk, mv, a.eta, a.W0, static_cast<__nv_bfloat16*>(a.Z), a.W_out, a.T,
                                         a.chunk, status);
    return cudaGetLastError();
}

int pick_cg(int d, long long bh, int sms) {
#ifdef TTT_LINEAR_CG
    (void)bh;
    (void)sms;
    return TTT_LINEAR_CG > d / 16 ? d / 16 : TTT_LINEAR_CG;
#else
    // up to 4 consumer warps per CTA (one per SM sub-partition); narrower CTAs only
    // when whole-head CTAs would leave more than half of the SMs idle
    int cg = d / 16 < 4 ? d / 16 : 4;
    while (cg > 1 && bh * (d / 16 / cg) * 2 <= (long long)sms) cg /= 2;
    return cg;
#endif
}

}  // namespace

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static cudaError_t get_encoder(EncodeTiledFn* fn) {
    static EncodeTiledFn cached = nullptr;
    if (!cached) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q);
        if (e != cudaSuccess) return e;
        if (q != cudaDriverEntryPointSuccess || !p) return cudaErrorSymbolNotFound;
        cached = reinterpret_cast<EncodeTiledFn>(p);
    }
    *fn = cached;
    return cudaSuccess;
}

// [rows][D] bf16 viewed as a 2D tensor; box = 16 rows x 64 columns, 128-byte swizzle.
cudaError_t make_tma_map_bf16(CUtensorMap* m, const void* base, uint64_t rows, int D) {
    EncodeTiledFn enc;
    cudaError_t e = get_encoder(&enc);
    if (e != cudaSuccess) return e;
    cuuint64_t dims[2] = {cuuint64_t(D), cuuint64_t(rows)};
    cuuint64_t strides[1] = {cuuint64_t(D) * 2};
    cuuint32_t box[2] = {64, 16};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t launch_linear_prefill_mma(const LinearArgs& a, cudaStream_t s, int* status) {
    if (!a.bf16 || (a.d != 64 && a.d != 128) || a.chunk % 16 != 0 || a.T % a.chunk != 0) return cudaErrorNotSupported;
    if (uint64_t(a.B) * a.H * a.T > 0x7fffffffull) return cudaErrorNotSupported;  // TMA row coordinate is int32
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int cg = pick_cg(a.d, (long long)a.B * a.H, sms);
    const bool single = a.chunk == 16;
#define TTT_LAUNCH(D_, CG_, NST_) \
    return single ? launch_cfg<D_, CG_, NST_, true>(a, s, status) : launch_cfg<D_, CG_, NST_, false>(a, s, status)
    if (a.d == 64) {
        switch (cg) {
            case 4: TTT_LAUNCH(64, 4, 16);
            case 2: TTT_LAUNCH(64, 2, 16);
            default: TTT_LAUNCH(64, 1, 16);
        }
    }
    switch (cg) {
        case 4: TTT_LAUNCH(128, 4, 8);
        case 2: TTT_LAUNCH(128, 2, 8);
        default: TTT_LAUNCH(128, 1, 8);
    }
#undef TTT_LAUNCH
}

}  // namespace ttt
