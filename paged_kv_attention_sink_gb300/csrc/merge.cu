// attn_merge_states: combine two attention states over disjoint key sets.
//
// The split of attention along the KV length in "GPT-OSS on day 0"
// (Perplexity), section "Sink Attention", implies this log-sum-exp merge
// (the page does not print it): with L = max(lse_a, lse_b) and
// w = exp(lse - L), v = (w_a v_a + w_b v_b) / (w_a + w_b) and
// lse = L + ln(w_a + w_b).  HBM-bound elementwise work: each thread handles
// 4 consecutive dims of one (token, head) row with 8-byte loads and stores.
#include <algorithm>

#include "attn_internal.h"
#include "kernels.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

__global__ void __launch_bounds__(256)
merge_states_kernel(const __nv_bfloat16* __restrict__ va, const float* __restrict__ lsea,
                    const __nv_bfloat16* __restrict__ vb, const float* __restrict__ lseb,
                    __nv_bfloat16* vout, float* lseout, int64_t rows, int head_dim) {
    const int per_row = head_dim / 4;
    const int64_t total = rows * per_row;
    for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = idx / per_row;
        const int64_t off = r * head_dim + (idx % per_row) * 4;
        const float la = lsea[r], lb = lseb[r];
        const float L = fmaxf(la, lb);
        float wa = 0.f, wb = 0.f;
        if (L != -INFINITY) {
            wa = ptx::ex2((la - L) * kLog2e);
            wb = ptx::ex2((lb - L) * kLog2e);
        }
        const float W = wa + wb;
        const float inv = W > 0.f ? 1.f / W : 0.f;
        const uint2 xa = *reinterpret_cast<const uint2*>(va + off);
        const uint2 xb = *reinterpret_cast<const uint2*>(vb + off);
        const __nv_bfloat162* pa = reinterpret_cast<const __nv_bfloat162*>(&xa);
        const __nv_bfloat162* pb = reinterpret_cast<const __nv_bfloat162*>(&xb);
        float o[4];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const float2 fa = __bfloat1622float2(pa[k]);
            const float2 fb = __bfloat1622float2(pb[k]);
            o[2 * k] = (wa * fa.x + wb * fb.x) * inv;
            o[2 * k + 1] = (wa * fa.y + wb * fb.y) * inv;
        }
        uint2 y;
        y.x = ptx::pack_bf16x2(o[0], o[1]);
        y.y = ptx::pack_bf16x2(o[2], o[3]);
        *reinterpret_cast<uint2*>(vout + off) = y;
        if (lseout && (idx % per_row) == 0) lseout[r] = W > 0.f ? L + logf(W) : -INFINITY;
    }
}

}  // namespace

attn_status launch_merge_states(const void* va, const float* lsea, const void* vb,
                                const float* lseb, void* vout, float* lseout, int64_t rows,
                                int head_dim, cudaStream_t stream) {
    if (rows == 0) return ATTN_OK;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return ATTN_ERR_CUDA;
    const int64_t work = rows * (head_dim / 4);
    const int64_t blocks = std::min<int64_t>((work + 255) / 256, (int64_t)sms * 8);
    merge_states_kernel<<<(unsigned)blocks, 256, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(va), lsea, static_cast<const __nv_bfloat16*>(vb), lseb,
        static_cast<__nv_bfloat16*>(vout), lseout, rows, head_dim);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace attn
