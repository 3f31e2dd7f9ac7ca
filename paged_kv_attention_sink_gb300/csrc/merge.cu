// attn_merge_states: combine two attention states over disjoint key sets.
//
// The split of attention along the KV length in "GPT-OSS on day 0"
// (Perplexity), section "Sink Attention", implies this log-sum-exp merge
// (the page does not print it): with L = max(lse_a, lse_b) and
// w = exp(lse - L), v = (w_a v_a + w_b v_b) / (w_a + w_b) and
// lse = L + ln(w_a + w_b).  HBM-bound elementwise work: each thread handles
// 4 consecutive dims of one (token, head) row (8-byte bf16 / 16-byte fp32
// loads and stores).  attn_merge_states takes bf16 value states (what the
// attention calls return); attn_merge_states_f32 takes fp32 ones (partial
// states kept unrounded, e.g. from a KV split across devices) and writes fp32
// or bf16.
#include <algorithm>

#include "attn_internal.h"
#include "kernels.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

// Four consecutive values of a state, as fp32.
template <bool kF32>
__device__ __forceinline__ void load4(const void* base, int64_t off, float (&x)[4]) {
    if constexpr (kF32) {
        const float4 v = *reinterpret_cast<const float4*>(static_cast<const float*>(base) + off);
        x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
    } else {
        const uint2 v = *reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(base) + off);
        const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v.x));
        const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v.y));
        x[0] = lo.x; x[1] = lo.y; x[2] = hi.x; x[3] = hi.y;
    }
}
template <bool kF32>
__device__ __forceinline__ void store4(void* base, int64_t off, const float (&x)[4]) {
    if constexpr (kF32) {
        *reinterpret_cast<float4*>(static_cast<float*>(base) + off) = make_float4(x[0], x[1], x[2], x[3]);
    } else {
        uint2 y;
        y.x = ptx::pack_bf16x2(x[0], x[1]);
        y.y = ptx::pack_bf16x2(x[2], x[3]);
        *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(base) + off) = y;
    }
}

// kInF32 / kOutF32: the value states / the merged values are fp32 (else bf16).
template <bool kInF32, bool kOutF32>
__global__ void __launch_bounds__(256)
merge_states_kernel(const void* __restrict__ va, const float* __restrict__ lsea, const void* __restrict__ vb,
                    const float* __restrict__ lseb, void* vout, float* lseout, int64_t rows, int head_dim) {
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
        float xa[4], xb[4], o[4];
        load4<kInF32>(va, off, xa);
        load4<kInF32>(vb, off, xb);
#pragma unroll
        for (int k = 0; k < 4; ++k) o[k] = (wa * xa[k] + wb * xb[k]) * inv;
        store4<kOutF32>(vout, off, o);
        if (lseout && (idx % per_row) == 0) lseout[r] = W > 0.f ? L + logf(W) : -INFINITY;
    }
}

}  // namespace

attn_status launch_merge_states(const void* va, const float* lsea, const void* vb, const float* lseb, void* vout,
                                float* lseout, int64_t rows, int head_dim, bool in_f32, bool out_f32,
                                cudaStream_t stream) {
    if (rows == 0) return ATTN_OK;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return ATTN_ERR_CUDA;
    const int64_t work = rows * (head_dim / 4);
    const unsigned blocks = (unsigned)std::min<int64_t>((work + 255) / 256, (int64_t)sms * 8);
    if (!in_f32)
        merge_states_kernel<false, false><<<blocks, 256, 0, stream>>>(va, lsea, vb, lseb, vout, lseout, rows, head_dim);
    else if (out_f32)
        merge_states_kernel<true, true><<<blocks, 256, 0, stream>>>(va, lsea, vb, lseb, vout, lseout, rows, head_dim);
    else
        merge_states_kernel<true, false><<<blocks, 256, 0, stream>>>(va, lsea, vb, lseb, vout, lseout, rows, head_dim);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace attn
