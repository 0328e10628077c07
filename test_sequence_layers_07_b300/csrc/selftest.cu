// selftest.cu -- exercise of the bounded-wait failure path on the device.
//
// One CTA waits on an mbarrier that no thread ever arrives on, with the same
// bounded wait the prefill kernels use; when the limit expires it records
// TTT_ERR_TIMEOUT in the device status word and returns.  Nothing traps,
// faults or hangs: the context stays usable and the host reads the status
// with ttt_get_device_status().
#include "ptx.cuh"
#include "ttt_common.cuh"
#include "ttt_internal.h"

namespace ttt {
namespace {

__global__ void wait_timeout_kernel(unsigned long long limit_ns, int* status) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ volatile int never;
    if (threadIdx.x == 0) {
        ptx::mbar_init(ptx::smem_u32(&bar), 1);
        ptx::fence_mbar_init();
        never = 0;
    }
    __syncthreads();
    // phase 0 never completes: the only way out is the bound
    const bool ok = ptx::mbar_wait_bounded(ptx::smem_u32(&bar), 0, &never, limit_ns);
    if (!ok && threadIdx.x == 0) record_status(status, kStatusTimeout);
}

}  // namespace

cudaError_t launch_wait_timeout_selftest(unsigned long long limit_ns, cudaStream_t s, int* status) {
    wait_timeout_kernel<<<1, 32, 0, s>>>(limit_ns, status);
    return cudaGetLastError();
}

}  // namespace ttt
