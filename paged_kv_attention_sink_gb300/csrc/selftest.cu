// attn_selftest_bounded_wait: checks, on the device, the bounded wait that
// every kernel of the library uses for its mbarriers.
//
// One warp initialises a shared-memory mbarrier that expects one arrival and
// then waits on it through ptx::mbar_wait, the same helper the decode and
// prefill kernels call.  Nothing ever arrives, so the wait must give up after
// its wall-time limit and report failure; the kernel then records the timeout
// bit and the time it waited, and returns.  Nothing is loaded asynchronously
// and nothing is allocated, so there is nothing else to wind down.
//
// attn_selftest_exp2: evaluates the prefill softmax's FMA-pipe exponential
// (exp2_poly.cuh, the same inline function and the same argument set-up the
// kernel uses) next to the MUFU's ex2.approx on the same scores, so a test
// can bound the polynomial's error on the GPU itself.
#include <cuda_runtime.h>

#include "attn_internal.h"
#include "exp2_poly.cuh"
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

// Thread k handles scores 2k and 2k + 1 (the polynomial works on pairs).
__global__ void selftest_exp2_kernel(const float* x, float* y_poly, float* y_mufu, int64_t n, float scale_log2,
                                     float m) {
    const int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (2 * k >= n) return;
    const bool two = 2 * k + 1 < n;
    const float s0 = x[2 * k], s1 = two ? x[2 * k + 1] : s0;
    // As in the prefill softmax: a = scale_log2 / R, b = 1/2 - m / R.
    const float a = scale_log2 * exp2poly::kInvRange;
    const float b = fmaf(-m, exp2poly::kInvRange, 0.5f);
    const float2 p = exp2poly::exp2_pair(s0, s1, a, b);
    y_poly[2 * k] = p.x;
    y_mufu[2 * k] = ptx::ex2(fmaf(s0, scale_log2, -m));
    if (two) {
        y_poly[2 * k + 1] = p.y;
        y_mufu[2 * k + 1] = ptx::ex2(fmaf(s1, scale_log2, -m));
    }
}

}  // namespace
}  // namespace attn

extern "C" attn_status attn_selftest_exp2(const float* x, float* y_poly, float* y_mufu, int64_t n,
                                          float scale_log2, float m, void* stream) {
    if (n < 0 || (n > 0 && (!x || !y_poly || !y_mufu))) return ATTN_ERR_INVALID_ARG;
    if (n == 0) return ATTN_OK;
    const int64_t pairs = (n + 1) / 2;
    const int threads = 256;
    const int64_t blocks = (pairs + threads - 1) / threads;
    if (blocks > 0x7fffffff) return ATTN_ERR_INVALID_ARG;
    attn::selftest_exp2_kernel<<<(unsigned)blocks, threads, 0, static_cast<cudaStream_t>(stream)>>>(
        x, y_poly, y_mufu, n, scale_log2, m);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

extern "C" attn_status attn_selftest_bounded_wait(int64_t* result, void* stream) {
    if (!result) return ATTN_ERR_INVALID_ARG;
    attn::selftest_bounded_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(result);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}
