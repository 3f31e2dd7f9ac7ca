// KV-cache data movement around the attention kernels: appending the step's
// new K/V rows to their HND pages, and packing / unpacking a head slice of
// pages into a contiguous buffer.
//
// Append: "Disaggregated prefill and decode" (Perplexity), section "KV
// Messenger" -- the model appends a layer's new tokens to the KV cache, and
// the cache entries are valid after that append and before attention.  Row i
// of request b (its i-th forwarded token) is cache position
// t = kv_len - qo_len + i (the causal mask's alignment); the plan stores, per
// row, the page-table slot kv_indptr[b] + t / P and the row t % P in the page.
//
// Head-slice pack / unpack: same page, section "Sharded KV transfer" -- the
// HND layout (heads before tokens) keeps a page's slice of heads contiguous,
// so a head-sharded page moves as one block; these kernels gather such blocks
// into one buffer (pack) or scatter them back into pages (unpack) on one GPU.
//
// All three are HBM-bound copies: 16-byte vector loads and stores, coalesced
// along the contiguous dimension, a grid-stride loop over a grid sized to the
// SM count.  Page ids out of range set the device error word and skip the copy.
#include <cuda_runtime.h>

#include "attn_internal.h"
#include "kernels.h"

namespace attn {
namespace {

constexpr int kCopyThreads = 256;

// One warp per query row (grid-stride over rows): the row's page slot and
// page id are loaded once, then the lanes copy its 2 * Hkv * chunks 16-byte
// chunks (K rows of every head, then V), several independent loads in flight
// per lane.  Reads are contiguous per row; writes are D * 2 contiguous bytes
// per (K/V, head).
__global__ void __launch_bounds__(kCopyThreads)
append_kv_kernel(const uint4* __restrict__ k_new, const uint4* __restrict__ v_new, uint4* __restrict__ pool,
                 const int2* __restrict__ slots, const int32_t* __restrict__ page_table, int64_t rows,
                 int32_t Hkv, int32_t P, int32_t chunks, int32_t num_pages, int32_t* err) {
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    const int32_t per_half = Hkv * chunks;   // chunks of one row's K (or V)
    for (int64_t r = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < rows; r += warps) {
        const int2 slot = slots[r];
        const int32_t page = page_table[slot.x];
        if (page < 0 || page >= num_pages) {
            if (lane == 0) atomicOr(err, ATTN_DEVICE_ERR_PAGE_ID);
            continue;
        }
        const uint4* ksrc = k_new + r * per_half;
        const uint4* vsrc = v_new + r * per_half;
        uint4* kdst = pool + ((int64_t)page * 2 * Hkv * P + slot.y) * chunks;   // head 0 of K
        uint4* vdst = kdst + (int64_t)Hkv * P * chunks;                           // head 0 of V
        for (int32_t k = lane; k < per_half; k += 32) {
            const int32_t g = k / chunks, c = k - g * chunks;
            const uint4 kv0 = __ldg(ksrc + k), kv1 = __ldg(vsrc + k);
            kdst[(int64_t)g * P * chunks + c] = kv0;
            vdst[(int64_t)g * P * chunks + c] = kv1;
        }
    }
}

// One CTA walk per (page i, K/V): the head slice [h0, h0 + nh) of that half of
// the page is `slice` contiguous chunks in the pool and in the buffer.
template <bool kUnpack>
__global__ void __launch_bounds__(kCopyThreads)
head_slice_kernel(uint4* __restrict__ pool, uint4* __restrict__ buf, const int32_t* __restrict__ page_ids,
                  int64_t n, int32_t Hkv, int32_t head_chunks, int32_t h0, int32_t nh, int64_t num_pages,
                  int32_t* err) {
    const int64_t slice = (int64_t)nh * head_chunks;
    for (int64_t blk = blockIdx.x; blk < n * 2; blk += gridDim.x) {
        const int64_t i = blk >> 1;
        const int32_t kv = (int32_t)(blk & 1);
        const int32_t page = page_ids[i];
        if (page < 0 || page >= num_pages) {
            if (threadIdx.x == 0 && kv == 0 && err) atomicOr(err, ATTN_DEVICE_ERR_PAGE_ID);
            continue;
        }
        uint4* p = pool + (((int64_t)page * 2 + kv) * Hkv + h0) * head_chunks;
        uint4* b = buf + blk * slice;
        for (int64_t k = threadIdx.x; k < slice; k += blockDim.x) {
            if (kUnpack) p[k] = b[k];
            else b[k] = p[k];
        }
    }
}

// Grid of a grid-stride copy: one CTA per work item up to `per_sm` CTAs per
// SM; 0 when the SM count cannot be queried.
int copy_grid(int64_t work_items, int per_sm) {
    int32_t sms = 0;
    if (!current_sm_count(&sms)) return 0;
    const int64_t cap = (int64_t)sms * per_sm;
    return (int)(work_items < cap ? (work_items > 0 ? work_items : 1) : cap);
}

}  // namespace

attn_status launch_append_kv(attn_plan_s* plan, const void* k_new, const void* v_new, void* kv_cache,
                             cudaStream_t stream) {
    const int64_t rows = plan->info.total_qo_rows;
    if (rows == 0) return ATTN_OK;
    const int32_t chunks = plan->D / 8;
    const int grid = copy_grid((rows + kCopyThreads / 32 - 1) / (kCopyThreads / 32), 8);
    if (grid == 0) return ATTN_ERR_CUDA;
    append_kv_kernel<<<grid, kCopyThreads, 0, stream>>>(
        static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), static_cast<uint4*>(kv_cache),
        reinterpret_cast<const int2*>(plan->ws + plan->layout.append), plan->page_table, rows, plan->Hkv,
        plan->P, chunks, plan->num_pages, reinterpret_cast<int32_t*>(plan->ws + plan->layout.err));
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

attn_status launch_head_slice(bool unpack, void* kv_cache, void* buf, const int32_t* page_ids, int64_t n,
                              int64_t num_pages, int32_t Hkv, int32_t P, int32_t D, int32_t h0, int32_t nh,
                              int32_t* err, cudaStream_t stream) {
    if (n == 0) return ATTN_OK;
    const int32_t head_chunks = P * D / 8;
    const int grid = copy_grid(n * 2, 4);
    if (grid == 0) return ATTN_ERR_CUDA;
    if (unpack)
        head_slice_kernel<true><<<grid, kCopyThreads, 0, stream>>>(
            static_cast<uint4*>(kv_cache), static_cast<uint4*>(buf), page_ids, n, Hkv, head_chunks, h0, nh,
            num_pages, err);
    else
        head_slice_kernel<false><<<grid, kCopyThreads, 0, stream>>>(
            static_cast<uint4*>(kv_cache), static_cast<uint4*>(buf), page_ids, n, Hkv, head_chunks, h0, nh,
            num_pages, err);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace attn
