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
//
// For d in {64, 128} a streaming kernel is used instead: each CTA runs GPC
// groups of d threads (thread c owns column c of W, so k W and q W need no
// reduction across threads), and each group works through a fixed, equal
// share of the heads.  The 16 or 64 KB state of a head arrives by one bulk
// copy (cp.async.bulk, with q, k, v) into an NSTG-stage shared-memory ring,
// is updated in place, and leaves by one bulk store; the next heads' copies
// are in flight meanwhile.
#include "ptx.cuh"
#include "ttt_common.cuh"
#include "ttt_internal.h"

namespace ttt {
namespace {

constexpr int kThreads = 256;
constexpr uint64_t kWaitLimitNs = 4000000000ull;

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

template <typename TI, int D, int GPC, int NSTG>
struct StreamCfg {
    static constexpr int WB = D * D * 4;              // fp32 state of a head
    static constexpr int IO = D * int(sizeof(TI));    // one of q, k, v
    static constexpr int STG = (WB + 3 * IO + 127) / 128 * 128;
    static constexpr int BYTES = GPC * NSTG * STG;
    static constexpr int THREADS = GPC * D;
};

__device__ __forceinline__ void group_bar(int id, int n) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory"); }

__device__ __forceinline__ bool group_any(int id, int n, bool c) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(uint32_t(c)), "r"(id), "r"(n)
        : "memory");
    return r != 0;
}

// 8 consecutive elements of q, k or v in shared memory, as fp32
__device__ __forceinline__ void ld8(const float* p, float (&o)[8]) {
    const float4 a = reinterpret_cast<const float4*>(p)[0], b = reinterpret_cast<const float4*>(p)[1];
    o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w; o[4] = b.x; o[5] = b.y; o[6] = b.z; o[7] = b.w;
}
__device__ __forceinline__ void ld8(const __nv_bfloat16* p, float (&o)[8]) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    o[0] = ptx::bf16_lo(u.x); o[1] = ptx::bf16_hi(u.x); o[2] = ptx::bf16_lo(u.y); o[3] = ptx::bf16_hi(u.y);
    o[4] = ptx::bf16_lo(u.z); o[5] = ptx::bf16_hi(u.z); o[6] = ptx::bf16_lo(u.w); o[7] = ptx::bf16_hi(u.w);
}

template <typename TI, int D, int GPC, int NSTG>
__global__ void __launch_bounds__(GPC * D, 1)
linear_decode_stream_kernel(const TI* __restrict__ q, const TI* __restrict__ k, const TI* __restrict__ v,
                            const float* __restrict__ eta, float* W, TI* __restrict__ z, int BH, int per,
                            int* status) {
    using C = StreamCfg<TI, D, GPC, NSTG>;
    extern __shared__ __align__(128) uint8_t smem_s[];
    __shared__ __align__(8) uint64_t full[GPC][NSTG];
    __shared__ volatile int s_err;
    __shared__ volatile int s_zero;
    const int g = threadIdx.x / D, c = threadIdx.x % D;  // group, column
    const int h0 = (blockIdx.x * GPC + g) * per;         // first head of this group
    const int nh = BH - h0 < per ? (BH - h0 > 0 ? BH - h0 : 0) : per;
    const int bar_id = 1 + g;
    if (threadIdx.x == 0) {
        for (int gg = 0; gg < GPC; ++gg)
            for (int st = 0; st < NSTG; ++st) ptx::mbar_init(ptx::smem_u32(&full[gg][st]), 1);
        s_err = 0;
        s_zero = 0;
        ptx::fence_mbar_init();
    }
    __syncthreads();
    uint8_t* gbase = smem_s + g * NSTG * C::STG;
    const uint32_t gb = ptx::smem_u32(gbase);
    const bool prod = c == 0;
    auto issue = [&](int i) {  // the group's i-th head into stage i % NSTG
        const int st = i % NSTG;
        const size_t h = size_t(h0) + i;
        const uint32_t dst = gb + st * C::STG;
        const uint32_t fb = ptx::smem_u32(&full[g][st]);
        ptx::mbar_arrive_expect_tx(fb, C::WB + 3 * C::IO);
        ptx::bulk_load(dst, W + h * D * D, C::WB, fb);
        ptx::bulk_load(dst + C::WB, q + h * D, C::IO, fb);
        ptx::bulk_load(dst + C::WB + C::IO, k + h * D, C::IO, fb);
        ptx::bulk_load(dst + C::WB + 2 * C::IO, v + h * D, C::IO, fb);
    };
    // NSTG - 1 heads are in flight ahead of the one being updated; the last stage is refilled
    // one head late, so that the refill never waits for a store that was just issued
    int issued = 0;
    if (prod)
        for (; issued < NSTG && issued < nh; ++issued) issue(issued);
    int done = 0;
    for (int i = 0; i < nh; ++i) {
        const int st = i % NSTG;
        const size_t h = size_t(h0) + i;
        const bool ok = ptx::mbar_wait_bounded(ptx::smem_u32(&full[g][st]), (i / NSTG) & 1, &s_err, kWaitLimitNs);
        if (group_any(bar_id, D, !ok)) {
            if (!s_err) record_status(status, kStatusTimeout);
            s_err = 1;
            break;
        }
        float* Ws = reinterpret_cast<float*>(gbase + st * C::STG);
        const TI* qs = reinterpret_cast<const TI*>(gbase + st * C::STG + C::WB);
        const TI* ks = qs + D;
        const TI* vs = ks + D;
        const float et = eta[h];
        float w[D <= 64 ? D : 1];
        float kw = 0.f, qw = 0.f, qk = 0.f;
#pragma unroll(D <= 64 ? D / 8 : 2)
        for (int r0 = 0; r0 < D; r0 += 8) {
            float kr[8], qr[8];
            ld8(ks + r0, kr);
            ld8(qs + r0, qr);
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const float wv = Ws[(r0 + u) * D + c];
                if constexpr (D <= 64) w[r0 + u] = wv;
                kw = fmaf(kr[u], wv, kw);
                qw = fmaf(qr[u], wv, qw);
                qk = fmaf(qr[u], kr[u], qk);
            }
        }
        const float e = kw - to_f32(vs[c]);
        z[h * D + c] = from_f32<TI>(fmaf(-et * qk, e, qw));  // q W_new = q W - eta (q.k) e
        const float ne = -et * e;
#pragma unroll(D <= 64 ? D / 8 : 2)
        for (int r0 = 0; r0 < D; r0 += 8) {
            float kr[8];
            ld8(ks + r0, kr);
#pragma unroll
            for (int u = 0; u < 8; ++u)  // registers hold the column at d = 64; re-read it at d = 128
                Ws[(r0 + u) * D + c] = fmaf(ne, kr[u], D <= 64 ? w[r0 + u] : Ws[(r0 + u) * D + c]);
        }
        ptx::fence_proxy_async_smem();  // the stage's new state is visible to the bulk store
        group_bar(bar_id, D);
        if (prod) {
            ptx::bulk_store(W + h * D * D, ptx::smem_u32(Ws), C::WB);
            ptx::bulk_commit();
            // refill the previous head's stage, whose store was issued one head ago
            if (i >= 1 && issued < nh) {
                ptx::bulk_wait_read_1();
                issue(issued);
                ++issued;
            }
        }
        done = i + 1;
    }
    if (prod) {
        ptx::bulk_wait_all();
        // never retire with copies in flight (after an expired wait only)
        for (int i = done; i < issued; ++i)
            ptx::mbar_wait_bounded(ptx::smem_u32(&full[g][i % NSTG]), (i / NSTG) & 1, &s_zero, kWaitLimitNs);
    }
}

template <typename TI, int D, int GPC, int NSTG>
cudaError_t launch_stream(const DecodeArgs& a, cudaStream_t s, int* status) {
    using C = StreamCfg<TI, D, GPC, NSTG>;
    const int BH = a.B * a.H;
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    // an equal share of heads per group, one CTA per SM at most
    const int groups0 = sms * GPC;
    const int per = (BH + groups0 - 1) / groups0;
    const int groups = (BH + per - 1) / per;
    const unsigned grid = unsigned((groups + GPC - 1) / GPC);
    auto kern = linear_decode_stream_kernel<TI, D, GPC, NSTG>;
    cudaError_t e = allow_dynamic_smem(reinterpret_cast<const void*>(kern), C::BYTES);
    if (e != cudaSuccess) return e;
    kern<<<grid, C::THREADS, C::BYTES, s>>>(static_cast<const TI*>(a.q), static_cast<const TI*>(a.k),
                                           static_cast<const TI*>(a.v), a.eta, a.W, static_cast<TI*>(a.z), BH, per,
                                           status);
    return cudaGetLastError();
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
cudaError_t launch_t(const DecodeArgs& a, cudaStream_t s, int* status) {
    switch (a.d) {
        case 16: return launch_d<TI, 16>(a, s);
        case 32: return launch_d<TI, 32>(a, s);
        case 64: return launch_stream<TI, 64, 4, 3>(a, s, status);
        case 128: return launch_stream<TI, 128, 1, 3>(a, s, status);
        default: return cudaErrorNotSupported;
    }
}

}  // namespace

cudaError_t launch_linear_decode(const DecodeArgs& a, cudaStream_t s, int* status) {
    return a.bf16 ? launch_t<__nv_bfloat16>(a, s, status) : launch_t<float>(a, s, status);
}

}  // namespace ttt
