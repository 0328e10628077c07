// ttt_common.cuh -- small device helpers shared by the kernel translation units.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ttt {

// Element loads/stores with conversion to and from fp32.
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Device status codes (same values as ttt_status in include/ttt.h).
enum : int { kStatusOk = 0, kStatusTimeout = 4 };

// Records the first error a kernel observed; later errors do not overwrite it.
__device__ __forceinline__ void record_status(int* status, int code) {
    if (status) atomicCAS(status, kStatusOk, code);
}

}  // namespace ttt
