// attn_selftest_bounded_wait: checks, on the device, the bounded wait that
// every kernel of the library uses for its mbarriers.
//
// One warp initialises a shared-memory mbarrier that expects one arrival and
// then waits on it through ptx::mbar_wait, the same helper the decode and
// prefill kernels call.  Nothing ever arrives, so the wait must give up after
// its wall-time limit and report failure; the kernel then records the timeout
// bit and the time it waited, and returns.  Nothing is loaded asynchronously
// and nothing is allocated, so there is nothing else to wind down.
#include <cuda_runtime.h>

#include "attn_internal.h"
#include "ptx.cuh"

namespace attn {
namespace {

__global__ void __launch_bounds__(32) selftest_bounded_wait_kernel(int64_t* result) {
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = ptx::smem_u32(&bar);
    if (threadIdx.x == 0) {
        ptx::mbar_init(b, 1);
        ptx::fence_mbar_init();
    }
    __syncwarp();
    const uint64_t t0 = ptx::globaltimer_ns();
    const bool completed = __all_sync(0xffffffffu, ptx::mbar_wait(b, 0));
    const uint64_t t1 = ptx::globaltimer_ns();
    if (threadIdx.x == 0) {
        result[0] = completed ? 0 : ATTN_DEVICE_ERR_TIMEOUT;
        result[1] = (int64_t)(t1 - t0);
    }
}

}  // namespace
}  // namespace attn

extern "C" attn_status attn_selftest_bounded_wait(int64_t* result, void* stream) {
    if (!result) return ATTN_ERR_INVALID_ARG;
    attn::selftest_bounded_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(result);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}
