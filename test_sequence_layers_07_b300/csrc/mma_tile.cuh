// mma_tile.cuh -- tile addressing and state packing shared by the warp-MMA TTT-Linear kernels.
#pragma once

#include <stdint.h>

#include "ptx.cuh"

namespace ttt {

// byte offset of (row, col) in a [16][D] bf16 tile stored as D/64 TMA boxes of [16][64] with the
// 128-byte swizzle (16-byte chunk index XOR row % 8); col % 8 == 0
__device__ __forceinline__ uint32_t swz(int row, int col) {
    return uint32_t((col >> 6) * 2048 + row * 128 + ((((col & 63) >> 3) ^ (row & 7)) << 4));
}

// The fp32 state W^T of a 16-column group (accumulator layout of m16n8k16: w[nt] holds columns
// g (+8) of input rows 8 nt + 2t (+1)) packed to bf16 A fragments over the input dimension.
template <int KS>
__device__ __forceinline__ void pack_state(const float (&w)[2 * KS][4], uint32_t (&wa)[KS][4]) {
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
        wa[ks][0] = ptx::pack_bf16(w[2 * ks][0], w[2 * ks][1]);
        wa[ks][1] = ptx::pack_bf16(w[2 * ks][2], w[2 * ks][3]);
        wa[ks][2] = ptx::pack_bf16(w[2 * ks + 1][0], w[2 * ks + 1][1]);
        wa[ks][3] = ptx::pack_bf16(w[2 * ks + 1][2], w[2 * ks + 1][3]);
    }
}

// Loads / stores the 16 columns [c0, c0 + 16) of a row-major [D][D] fp32 matrix in the state
// layout above (lane (g, t) of the warp).
template <int NT>
__device__ __forceinline__ void load_state(float (&w)[NT][4], const float* M, int D, int c0, int g, int t) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int r = 8 * nt + 2 * t;
        w[nt][0] = M[size_t(r) * D + c0 + g];
        w[nt][1] = M[size_t(r + 1) * D + c0 + g];
        w[nt][2] = M[size_t(r) * D + c0 + g + 8];
        w[nt][3] = M[size_t(r + 1) * D + c0 + g + 8];
    }
}

template <int NT>
__device__ __forceinline__ void store_state(const float (&w)[NT][4], float* M, int D, int c0, int g, int t) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int r = 8 * nt + 2 * t;
        M[size_t(r) * D + c0 + g] = w[nt][0];
        M[size_t(r + 1) * D + c0 + g] = w[nt][1];
        M[size_t(r) * D + c0 + g + 8] = w[nt][2];
        M[size_t(r + 1) * D + c0 + g + 8] = w[nt][3];
    }
}

}  // namespace ttt
