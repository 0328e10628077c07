// decode.cu -- TTT-Linear online decode step (a block of one token), in place:
//     e = k W - v;   W <- W - eta k^T e;   z = q W_new = q W - eta (q.k) e
// ("Test-Time Training Layers ...", section "The Core Mechanism", and the
// per-token forward step of its PyTorch listing section).
//
// Bandwidth-bound: every step streams the fp32 state (d*d*4 bytes per head)
// in and out exactly once.  Per head, 2*d threads each own D/8 rows x 4
// columns of W in registers (one float4 per row): the loads of a warp cover
// whole 16-byte-aligned row segments (coalesced, all issued before the first
// use), the partial products k W and q W are reduced across the 8 row groups
// through shared memory, and the same registers are updated and stored back,
// so W is read once and written once.
#include "ttt_common.cuh"
#include "ttt_internal.h"

namespace ttt {
namespace {

constexpr int kThreads = 256;

template <typename TI, int D>
__global__ void __launch_bounds__(kThreads)
linear_decode_kernel(const TI* __restrict__ q, const TI* __restrict__ k, const TI* __restrict__ v,
                     const float* __restrict__ eta, float* __restrict__ W, TI* __restrict__ z, int BH) {
    constexpr int NT = 2 * D;            // threads per head
    constexpr int HPC = kThreads / NT;   // heads per CTA
    constexpr int CQ = D / 4;            // column quads
    constexpr int RG = NT / CQ;          // row groups (= 8)
    constexpr int RPT = D / RG;          // rows per thread
    static_assert(RG == 8, "layout assumes 8 row groups");

    __shared__ float4 red_k[HPC][RG][CQ];
    __shared__ float4 red_q[HPC][RG][CQ];
    __shared__ float red_qk[HPC][RG];

    const int hl = threadIdx.x / NT;
    const int lt = threadIdx.x % NT;
    const int cq = lt % CQ, rg = lt / CQ;
    const int head = blockIdx.x * HPC + hl;
    const bool live = head < BH;

    float4 w[RPT];
    float kr[RPT], qr[RPT];
    float4* Wh = reinterpret_cast<float4*>(W + size_t(live ? head : 0) * D * D);
    if (live) {
#pragma unroll
        for (int m = 0; m < RPT; ++m) w[m] = __ldcs(Wh + (rg + RG * m) * CQ + cq);
        const TI* kh = k + size_t(head) * D;
        const TI* qh = q + size_t(head) * D;
#pragma unroll
        for (int m = 0; m < RPT; ++m) {
            kr[m] = to_f32(kh[rg + RG * m]);
            qr[m] = to_f32(qh[rg + RG * m]);
        }
        float4 pk = make_float4(0.f, 0.f, 0.f, 0.f), pq = pk;
        float qk = 0.f;
#pragma unroll
        for (int m = 0; m < RPT; ++m) {
            pk.x += kr[m] * w[m].x; pk.y += kr[m] * w[m].y; pk.z += kr[m] * w[m].z; pk.w += kr[m] * w[m].w;
            pq.x += qr[m] * w[m].x; pq.y += qr[m] * w[m].y; pq.z += qr[m] * w[m].z; pq.w += qr[m] * w[m].w;
            qk += qr[m] * kr[m];
        }
        red_k[hl][rg][cq] = pk;
        red_q[hl][rg][cq] = pq;
        if (cq == 0) red_qk[hl][rg] = qk;
    }
    __syncthreads();
    if (!live) return;

    float4 kw = make_float4(0.f, 0.f, 0.f, 0.f), qw = kw;
    float qk = 0.f;
#pragma unroll
    for (int g = 0; g < RG; ++g) {
        float4 a = red_k[hl][g][cq], b = red_q[hl][g][cq];
        kw.x += a.x; kw.y += a.y; kw.z += a.z; kw.w += a.w;
        qw.x += b.x; qw.y += b.y; qw.z += b.z; qw.w += b.w;
        qk += red_qk[hl][g];
    }
    const TI* vh = v + size_t(head) * D + 4 * cq;
    const float et = eta[head];
    float4 e = make_float4(kw.x - to_f32(vh[0]), kw.y - to_f32(vh[1]), kw.z - to_f32(vh[2]), kw.w - to_f32(vh[3]));

    if (rg == 0) {
        const float s = et * qk;
        TI* zh = z + size_t(head) * D + 4 * cq;
        zh[0] = from_f32<TI>(qw.x - s * e.x);
        zh[1] = from_f32<TI>(qw.y - s * e.y);
        zh[2] = from_f32<TI>(qw.z - s * e.z);
        zh[3] = from_f32<TI>(qw.w - s * e.w);
    }
#pragma unroll
    for (int m = 0; m < RPT; ++m) {
        const float a = et * kr[m];
        float4 o = w[m];
        o.x -= a * e.x; o.y -= a * e.y; o.z -= a * e.z; o.w -= a * e.w;
        __stcs(Wh + (rg + RG * m) * CQ + cq, o);
    }
}

template <typename TI, int D>
cudaError_t launch_d(const DecodeArgs& a, cudaStream_t s) {
    constexpr int HPC = kThreads / (2 * D);
    const int BH = a.B * a.H;
    const unsigned grid = unsigned((BH + HPC - 1) / HPC);
    linear_decode_kernel<TI, D><<<grid, kThreads, 0, s>>>(
        static_cast<const TI*>(a.q), static_cast<const TI*>(a.k), static_cast<const TI*>(a.v), a.eta, a.W,
        static_cast<TI*>(a.z), BH);
    return cudaGetLastError();
}

template <typename TI>
cudaError_t launch_t(const DecodeArgs& a, cudaStream_t s) {
    switch (a.d) {
        case 16: return launch_d<TI, 16>(a, s);
        case 32: return launch_d<TI, 32>(a, s);
        case 64: return launch_d<TI, 64>(a, s);
        case 128: return launch_d<TI, 128>(a, s);
        default: return cudaErrorNotSupported;
    }
}

}  // namespace

cudaError_t launch_linear_decode(const DecodeArgs& a, cudaStream_t s) {
    return a.bf16 ? launch_t<__nv_bfloat16>(a, s) : launch_t<float>(a, s);
}

}  // namespace ttt
