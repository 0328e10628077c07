// mlp_decode.cu -- TTT-MLP online decode step (a block of one token), in place.
//
// Inner model f(x; W1, W2) = GELU(x W1) W2, tanh form of GELU, no biases
// ("Test-Time Training (TTT) Layers for Sequence Modeling", section "Variants:
// TTT-Linear vs. TTT-MLP"); one gradient step on 1/2 ||f(k) - v||^2 and the
// read-out through the updated weights ("Test-Time Training Layers ...",
// section "The Core Mechanism"):
//   u = k W1, a = GELU(u), e2 = a W2 - v, e1 = (e2 W2^T) . GELU'(u)
//   W1 <- W1 - eta k^T e1,  W2 <- W2 - eta a^T e2
//   z  = GELU(q W1_new) W2_new
// The read-out needs no second pass over the updated weights:
//   q W1_new = q W1 - eta (q.k) e1   and   hq W2_new = hq W2 - eta (hq.a) e2.
//
// Bandwidth-bound: each step reads and writes the 2*d*hidden fp32 state of a
// head exactly once.  One CTA per (batch, head), one thread per hidden unit j:
// the thread keeps column j of W1 in registers (coalesced loads and stores
// across the warp); W2 is copied into shared memory by 16-byte cp.async, so
// u = k W1 runs while it lands and no register holds it on the way.  Its rows
// are unpadded with the 16-byte chunks of row r permuted by an XOR of r: the
// row walk (e2 W2^T, 16-byte reads) and the column walks (a W2, hq W2) are
// bank-conflict free.  Column sums over the hidden units are split over
// hidden/d thread groups and finished through shared memory.  At hidden = 256
// two CTAs share an SM (up to 128 registers a thread); three, at 80 registers,
// spill and measured slower.
#include "ttt_common.cuh"
#include "ttt_internal.h"

namespace ttt {
namespace {

__device__ __forceinline__ float tanh_fast(float x) {
    float y;
    asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// GELU (tanh form) and its exact derivative
__device__ __forceinline__ float gelu_d(float x, float& gp) {
    const float c = 0.7978845608028654f, a = 0.044715f;
    const float t = tanh_fast(c * fmaf(a * x, x * x, x));
    gp = 0.5f * (1.f + t) + 0.5f * x * (1.f - t * t) * c * fmaf(3.f * a, x * x, 1.f);
    return 0.5f * x * (1.f + t);
}
__device__ __forceinline__ float gelu_f(float x) {
    const float c = 0.7978845608028654f, a = 0.044715f;
    const float t = tanh_fast(c * fmaf(a * x, x * x, x));
    return 0.5f * x * (1.f + t);
}

// word offset of W2[r][c] in shared memory: chunk c/4 of row r at position (c/4) XOR f(r), f(r) chosen so
// that eight consecutive rows put a given chunk in eight distinct 16-byte bank groups
template <int D>
__device__ __forceinline__ int w2_chunk(int r, int x) {
    constexpr int NCH = D / 4;
    const int f = NCH >= 8 ? (r & 7) : ((r >> 1) & (NCH - 1));
    return r * D + ((x ^ f) << 2);
}
template <int D>
__device__ __forceinline__ int w2_off(int r, int c) {
    return w2_chunk<D>(r, c >> 2) + (c & 3);
}

__device__ __forceinline__ void cp_async16(float* dst, const float* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
                 "l"(src)
                 : "memory");
}

template <int HID>
__device__ __forceinline__ float block_sum(float v, float* red) {
    v = warp_sum(v);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    if (l == 0) red[w] = v;
    __syncthreads();
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < HID / 32; ++i) s += red[i];
    __syncthreads();
    return s;
}

template <typename TI, int D, int HID>
__global__ void __launch_bounds__(HID, HID == 256 ? 2 : 1)
mlp_decode_kernel(const TI* __restrict__ q, const TI* __restrict__ k, const TI* __restrict__ v,
                  const float* __restrict__ eta, float* __restrict__ W1, float* __restrict__ W2, TI* __restrict__ z) {
    constexpr int NCH = D / 4;      // 16-byte chunks of a row of W2
    constexpr int PARTS = HID / D;  // thread groups of a column sum
    extern __shared__ __align__(16) float sm[];
    float* w2s = sm;                          // [HID][D], chunks permuted (w2_off)
    float* ks = w2s + HID * D;                // [D]
    float* qs = ks + D;                       // [D]
    float* vs = qs + D;                       // [D]
    float* av = vs + D;                       // [HID]  GELU(k W1)
    float* hqv = av + HID;                    // [HID]  GELU(q W1_new)
    float* part = hqv + HID;                  // [PARTS][D]
    float* e2s = part + PARTS * D;            // [D]
    float* red = e2s + D;                     // [HID / 32]

    const int j = threadIdx.x;
    const size_t bh = blockIdx.x;
    float* W1h = W1 + bh * D * HID;
    float* W2h = W2 + bh * HID * D;

    // column j of W1 into registers, then W2 into shared memory by cp.async (coalesced 16-byte pieces):
    // W1's loads go first, so that u = k W1 can run while W2 is still landing
    float w1[D];
#pragma unroll
    for (int i = 0; i < D; ++i) w1[i] = W1h[i * HID + j];
#pragma unroll 4
    for (int idx = j; idx < HID * NCH; idx += HID) cp_async16(w2s + w2_chunk<D>(idx / NCH, idx % NCH), W2h + 4 * idx);
    asm volatile("cp.async.commit_group;" ::: "memory");
    if (j < D) {
        ks[j] = to_f32(k[bh * D + j]);
        qs[j] = to_f32(q[bh * D + j]);
        vs[j] = to_f32(v[bh * D + j]);
    }
    const float et = eta[bh];
    __syncthreads();

    // u = k W1 and k-free q W1 for this hidden unit; q.k
    float u = 0.f, uq = 0.f, qk = 0.f;
#pragma unroll
    for (int i = 0; i < D; ++i) {
        u = fmaf(ks[i], w1[i], u);
        uq = fmaf(qs[i], w1[i], uq);
        qk = fmaf(qs[i], ks[i], qk);
    }
    float gp;
    const float aj = gelu_d(u, gp);
    av[j] = aj;
    asm volatile("cp.async.wait_group 0;" ::: "memory");  // this thread's pieces of W2 have landed
    __syncthreads();                                       // everyone's have

    // p = a W2: column c of W2 summed over this thread's share of the hidden units
    const int c = j % D, pi = j / D;
    {
        float s = 0.f;
#pragma unroll 8
        for (int r = pi * (HID / PARTS); r < (pi + 1) * (HID / PARTS); ++r) s = fmaf(av[r], w2s[w2_off<D>(r, c)], s);
        part[pi * D + c] = s;
    }
    __syncthreads();
    if (j < D) {
        float p = 0.f;
#pragma unroll
        for (int i = 0; i < PARTS; ++i) p += part[i * D + j];
        e2s[j] = p - vs[j];
    }
    __syncthreads();

    // e1 = (e2 W2^T) . GELU'(u): row j of W2, 16 bytes at a time
    float g0 = 0.f, g1 = 0.f;
#pragma unroll
    for (int x = 0; x < NCH; ++x) {
        const float4 w = *reinterpret_cast<const float4*>(w2s + w2_chunk<D>(j, x));
        const float4 e = *reinterpret_cast<const float4*>(e2s + 4 * x);
        g0 = fmaf(e.x, w.x, fmaf(e.y, w.y, g0));
        g1 = fmaf(e.z, w.z, fmaf(e.w, w.w, g1));
    }
    const float e1 = (g0 + g1) * gp;

    // W1 <- W1 - eta k^T e1 (column j, in registers), written back
#pragma unroll
    for (int i = 0; i < D; ++i) W1h[i * HID + j] = fmaf(-et * ks[i], e1, w1[i]);
    // read-out layer 1 through the updated W1: q W1_new = q W1 - eta (q.k) e1
    const float hq = gelu_f(fmaf(-et * qk, e1, uq));
    hqv[j] = hq;
    const float hqa = block_sum<HID>(hq * aj, red);  // also orders hqv before its readers

    // z = hq W2_new = hq W2 - eta (hq.a) e2
    {
        float s = 0.f;
#pragma unroll 8
        for (int r = pi * (HID / PARTS); r < (pi + 1) * (HID / PARTS); ++r) s = fmaf(hqv[r], w2s[w2_off<D>(r, c)], s);
        part[pi * D + c] = s;
    }
    __syncthreads();
    if (j < D) {
        float r = 0.f;
#pragma unroll
        for (int i = 0; i < PARTS; ++i) r += part[i * D + j];
        z[bh * D + j] = from_f32<TI>(fmaf(-et * hqa, e2s[j], r));
    }

    // W2 <- W2 - eta a^T e2, written back (coalesced)
#pragma unroll 4
    for (int idx = j; idx < HID * NCH; idx += HID) {
        const int r = idx / NCH, cc = 4 * (idx % NCH);
        const float4 w = *reinterpret_cast<const float4*>(w2s + w2_chunk<D>(r, idx % NCH));
        const float4 e = *reinterpret_cast<const float4*>(e2s + cc);
        const float s = -et * av[r];
        reinterpret_cast<float4*>(W2h)[idx] = make_float4(fmaf(s, e.x, w.x), fmaf(s, e.y, w.y), fmaf(s, e.z, w.z),
                                                          fmaf(s, e.w, w.w));
    }
}

template <int D, int HID>
constexpr size_t smem_bytes() {
    return sizeof(float) * (size_t(HID) * D + 3 * D + 2 * HID + (HID / D) * D + D + HID / 32);
}

template <typename TI, int D, int HID>
cudaError_t launch_dh(const MlpDecodeArgs& a, cudaStream_t s) {
    auto kern = mlp_decode_kernel<TI, D, HID>;
    constexpr size_t bytes = smem_bytes<D, HID>();
    cudaError_t e = allow_dynamic_smem(reinterpret_cast<const void*>(kern), int(bytes));
    if (e != cudaSuccess) return e;
    kern<<<unsigned(a.B) * unsigned(a.H), HID, bytes, s>>>(static_cast<const TI*>(a.q), static_cast<const TI*>(a.k),
                                                          static_cast<const TI*>(a.v), a.eta, a.W1, a.W2,
                                                          static_cast<TI*>(a.z));
    return cudaGetLastError();
}

template <typename TI, int D>
cudaError_t launch_d(const MlpDecodeArgs& a, cudaStream_t s) {
    switch (a.hidden) {
        case 64: return launch_dh<TI, D, 64>(a, s);
        case 128: return launch_dh<TI, D, 128>(a, s);
        case 256: return launch_dh<TI, D, 256>(a, s);
        default: return cudaErrorNotSupported;
    }
}

template <typename TI>
cudaError_t launch_t(const MlpDecodeArgs& a, cudaStream_t s) {
    switch (a.d) {
        case 16: return launch_d<TI, 16>(a, s);
        case 32: return launch_d<TI, 32>(a, s);
        case 64: return launch_d<TI, 64>(a, s);
        default: return cudaErrorNotSupported;
    }
}

}  // namespace

cudaError_t launch_mlp_decode(const MlpDecodeArgs& a, cudaStream_t s) {
    return a.bf16 ? launch_t<__nv_bfloat16>(a, s) : launch_t<float>(a, s);
}

}  // namespace ttt
