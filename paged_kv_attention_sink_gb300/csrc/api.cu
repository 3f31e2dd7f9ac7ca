// C entry points of libattn.so: argument checks, workspace binding, TMA
// descriptor construction, and dispatch to the kernel launchers.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "attn_internal.h"
#include "kernels.h"

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult qr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &qr) == cudaSuccess &&
            qr == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// The HND pool as a 3-D tensor {dim, token in page, (page, K/V, KV head)}:
// one box is `box_rows` consecutive tokens x 64 dims of one (page, KV head)
// block of K or V, stored 128-byte swizzled.
bool make_kv_map(void* map, const void* kv, const attn_plan_s* p, int box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)p->D, (cuuint64_t)p->P, (cuuint64_t)p->num_pages * 2 * p->Hkv};
    cuuint64_t strides[2] = {(cuuint64_t)p->D * 2, (cuuint64_t)p->P * p->D * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
    cuuint32_t elem[3] = {1, 1, 1};
    return fn(static_cast<CUtensorMap*>(map), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
              const_cast<void*>(kv), dims, strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Contiguous K or V [tokens][Hkv][D] (ragged plans) as a 3-D tensor
// {dim, KV head, token}: one box is 128 tokens x 64 dims of one KV head,
// stored like a 128-row page box; rows past the end read as zero.
bool make_ragged_map(void* map, const void* x, const attn_plan_s* p) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)p->D, (cuuint64_t)p->Hkv, (cuuint64_t)p->kv_tokens};
    cuuint64_t strides[2] = {(cuuint64_t)p->D * 2, (cuuint64_t)p->Hkv * p->D * 2};
    cuuint32_t box[3] = {64, 1, (cuuint32_t)attn::kPrefillKeys};
    cuuint32_t elem[3] = {1, 1, 1};
    return fn(static_cast<CUtensorMap*>(map), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
              const_cast<void*>(x), dims, strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// q (or out) [rows][Hq][D] as a 3-D tensor {dim, head, row}: one box is 128
// rows x 64 dims of one head; rows past the end read as zero (and are not
// written by a store).
bool make_q_map(void* map, const void* q, const attn_plan_s* p, uint32_t box_rows = attn::kPrefillRows) {
    auto fn = encode_fn();
    if (!fn) return false;
    const int64_t rows = p->info.total_qo_rows;
    cuuint64_t dims[3] = {(cuuint64_t)p->D, (cuuint64_t)p->Hq, (cuuint64_t)rows};
    cuuint64_t strides[2] = {(cuuint64_t)p->D * 2, (cuuint64_t)p->Hq * p->D * 2};
    cuuint32_t box[3] = {64, 1, (cuuint32_t)box_rows};
    cuuint32_t elem[3] = {1, 1, 1};
    return fn(static_cast<CUtensorMap*>(map), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
              const_cast<void*>(q), dims, strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

attn_status check_launch(attn_plan_t plan, const void* q, const void* kv, const void* out) {
    if (!plan) return ATTN_ERR_INVALID_ARG;
    if (!plan->bound) return ATTN_ERR_NOT_BOUND;
    if (!q || !kv || !out) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(kv) || !aligned16(out)) return ATTN_ERR_INVALID_ARG;
    return ATTN_OK;
}

}  // namespace

extern "C" attn_status attn_plan_bind_workspace(attn_plan_t plan, void* workspace, size_t bytes,
                                                void* stream) {
    if (!plan) return ATTN_ERR_INVALID_ARG;
    const attn::WorkspaceLayout& L = plan->layout;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255) != 0) return ATTN_ERR_INVALID_ARG;
    if (bytes < L.total) return ATTN_ERR_WORKSPACE_TOO_SMALL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned char* ws = static_cast<unsigned char*>(workspace);
    // The work lists lie in [0, L.counters): one host image, one copy (graph
    // plans have none: their list is built on the device).
    if (!plan->units.empty() || !plan->items.empty() || !plan->append_slots.empty()) {
        std::vector<unsigned char> img(L.counters, 0);
        auto put = [&](size_t off, const void* src, size_t bytes) {
            if (bytes) std::memcpy(img.data() + off, src, bytes);
        };
        put(L.units, plan->units.data(), plan->units.size() * sizeof(attn::DecodeUnit));
        put(L.items, plan->items.data(), plan->items.size() * sizeof(attn::PrefillItem));
        put(L.item_off, plan->item_off.data(), plan->item_off.size() * sizeof(int32_t));
        put(L.append, plan->append_slots.data(), plan->append_slots.size() * sizeof(int32_t));
        if (cudaMemcpyAsync(ws, img.data(), img.size(), cudaMemcpyHostToDevice, s) != cudaSuccess)
            return ATTN_ERR_CUDA;
    }
    // counters and the error word are adjacent: clear both.
    if (cudaMemsetAsync(ws + L.counters, 0, L.part_lse - L.counters, s) != cudaSuccess) return ATTN_ERR_CUDA;
    plan->ws = ws;
    plan->ws_bytes = bytes;
    plan->bound = true;
    return ATTN_OK;
}

extern "C" attn_status attn_decode(attn_plan_t plan, const void* q, const void* kv_cache,
                                   const float* sinks, void* out, float* lse, void* stream) {
    if (plan && plan->graph) return ATTN_ERR_INVALID_ARG;   // attn_decode_graph
    if (plan && plan->bound && plan->units.empty()) return ATTN_OK;
    attn_status st = check_launch(plan, q, kv_cache, out);
    if (st != ATTN_OK) return st;
    if (plan->kv_map_decode_ptr != kv_cache) {
        if (!make_kv_map(plan->kv_map_decode, kv_cache, plan, attn::kBlockTokens)) return ATTN_ERR_CUDA;
        plan->kv_map_decode_ptr = kv_cache;
    }
    return attn::launch_decode(plan, q, plan->kv_map_decode, sinks, out, lse,
                               static_cast<cudaStream_t>(stream));
}

extern "C" attn_status attn_decode_graph(attn_plan_t plan, const int32_t* kv_indptr, const int32_t* last_page_len,
                                         const int32_t* batch, const void* q, const void* kv_cache,
                                         const float* sinks, void* out, float* lse, void* stream) {
    if (!plan || !plan->graph) return ATTN_ERR_INVALID_ARG;
    attn_status st = check_launch(plan, q, kv_cache, out);
    if (st != ATTN_OK) return st;
    if (!kv_indptr || !last_page_len || !batch) return ATTN_ERR_INVALID_ARG;
    if (plan->kv_map_decode_ptr != kv_cache) {
        if (!make_kv_map(plan->kv_map_decode, kv_cache, plan, attn::kBlockTokens)) return ATTN_ERR_CUDA;
        plan->kv_map_decode_ptr = kv_cache;
    }
    return attn::launch_decode_graph(plan, kv_indptr, last_page_len, batch, q, plan->kv_map_decode, sinks, out, lse,
                                     static_cast<cudaStream_t>(stream));
}

extern "C" attn_status attn_graph_plan_read_units(attn_plan_t plan, int32_t* units, int64_t capacity,
                                                  int64_t* n_units, void* stream) {
    if (!plan || !plan->graph || !n_units || capacity < 0 || (capacity > 0 && !units)) return ATTN_ERR_INVALID_ARG;
    if (!plan->bound) return ATTN_ERR_NOT_BOUND;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return ATTN_ERR_CUDA;
    int32_t n = 0;
    if (cudaMemcpy(&n, plan->ws + plan->layout.n_units, sizeof n, cudaMemcpyDeviceToHost) != cudaSuccess)
        return ATTN_ERR_CUDA;
    *n_units = n;
    const int64_t k = n < capacity ? n : capacity;
    if (k > 0 && cudaMemcpy(units, plan->ws + plan->layout.units, (size_t)k * sizeof(attn::DecodeUnit),
                            cudaMemcpyDeviceToHost) != cudaSuccess)
        return ATTN_ERR_CUDA;
    return ATTN_OK;
}

extern "C" attn_status attn_prefill(attn_plan_t plan, const void* q, const void* kv_cache,
                                    const float* sinks, void* out, float* lse, void* stream) {
    if (plan && plan->ragged) return ATTN_ERR_INVALID_ARG;   // attn_prefill_ragged
    if (plan && plan->bound && plan->items.empty()) return ATTN_OK;
    attn_status st = check_launch(plan, q, kv_cache, out);
    if (st != ATTN_OK) return st;
    if (plan->kv_map_prefill_ptr != kv_cache) {
        const int box = plan->P < attn::kPrefillKeys ? plan->P : attn::kPrefillKeys;
        if (!make_kv_map(plan->kv_map_prefill, kv_cache, plan, box)) return ATTN_ERR_CUDA;
        plan->kv_map_prefill_ptr = kv_cache;
    }
    if (plan->q_map_prefill_ptr != q) {
        if (!make_q_map(plan->q_map_prefill, q, plan)) return ATTN_ERR_CUDA;
        plan->q_map_prefill_ptr = q;
    }
    if (plan->o_map_prefill_ptr != out) {
        if (!make_q_map(plan->o_map_prefill, out, plan, attn::kPrefillOutRows)) return ATTN_ERR_CUDA;
        plan->o_map_prefill_ptr = out;
    }
    return attn::launch_prefill(plan, plan->q_map_prefill, plan->kv_map_prefill, nullptr, plan->o_map_prefill,
                                sinks, out, lse, static_cast<cudaStream_t>(stream));
}

extern "C" attn_status attn_prefill_ragged(attn_plan_t plan, const void* q, const void* k, const void* v,
                                           const float* sinks, void* out, float* lse, void* stream) {
    if (!plan) return ATTN_ERR_INVALID_ARG;
    if (!plan->ragged) return ATTN_ERR_INVALID_ARG;   // paged plans go through attn_prefill
    if (plan->bound && plan->items.empty()) return ATTN_OK;
    attn_status st = check_launch(plan, q, k, out);
    if (st != ATTN_OK) return st;
    if (!v || !aligned16(v)) return ATTN_ERR_INVALID_ARG;
    if (plan->kv_map_prefill_ptr != k) {
        if (!make_ragged_map(plan->kv_map_prefill, k, plan)) return ATTN_ERR_CUDA;
        plan->kv_map_prefill_ptr = k;
    }
    if (plan->v_map_prefill_ptr != v) {
        if (!make_ragged_map(plan->v_map_prefill, v, plan)) return ATTN_ERR_CUDA;
        plan->v_map_prefill_ptr = v;
    }
    if (plan->q_map_prefill_ptr != q) {
        if (!make_q_map(plan->q_map_prefill, q, plan)) return ATTN_ERR_CUDA;
        plan->q_map_prefill_ptr = q;
    }
    if (plan->o_map_prefill_ptr != out) {
        if (!make_q_map(plan->o_map_prefill, out, plan, attn::kPrefillOutRows)) return ATTN_ERR_CUDA;
        plan->o_map_prefill_ptr = out;
    }
    return attn::launch_prefill(plan, plan->q_map_prefill, plan->kv_map_prefill, plan->v_map_prefill,
                                plan->o_map_prefill, sinks, out, lse, static_cast<cudaStream_t>(stream));
}

extern "C" attn_status attn_merge_states(const void* va, const float* lsea, const void* vb,
                                         const float* lseb, void* vout, float* lseout,
                                         int32_t n_tokens, int32_t n_heads, int32_t head_dim,
                                         void* stream) {
    if (n_tokens < 0 || n_heads <= 0 || head_dim <= 0 || head_dim % 4 != 0 || head_dim > 256)
        return ATTN_ERR_INVALID_ARG;
    if (n_tokens == 0) return ATTN_OK;
    if (!va || !lsea || !vb || !lseb || !vout) return ATTN_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(va) | reinterpret_cast<uintptr_t>(vb) |
         reinterpret_cast<uintptr_t>(vout)) & 7)
        return ATTN_ERR_INVALID_ARG;
    return attn::launch_merge_states(va, lsea, vb, lseb, vout, lseout, (int64_t)n_tokens * n_heads,
                                     head_dim, false, false, static_cast<cudaStream_t>(stream));
}

extern "C" attn_status attn_merge_states_f32(const float* va, const float* lsea, const float* vb,
                                             const float* lseb, void* vout, int32_t vout_bf16, float* lseout,
                                             int32_t n_tokens, int32_t n_heads, int32_t head_dim, void* stream) {
    if (n_tokens < 0 || n_heads <= 0 || head_dim <= 0 || head_dim % 4 != 0 || head_dim > 256)
        return ATTN_ERR_INVALID_ARG;
    if (n_tokens == 0) return ATTN_OK;
    if (!va || !lsea || !vb || !lseb || !vout) return ATTN_ERR_INVALID_ARG;
    const uintptr_t out_align = vout_bf16 ? 7 : 15;
    if (((reinterpret_cast<uintptr_t>(va) | reinterpret_cast<uintptr_t>(vb)) & 15) ||
        (reinterpret_cast<uintptr_t>(vout) & out_align))
        return ATTN_ERR_INVALID_ARG;
    return attn::launch_merge_states(va, lsea, vb, lseb, vout, lseout, (int64_t)n_tokens * n_heads, head_dim, true,
                                     vout_bf16 == 0, static_cast<cudaStream_t>(stream));
}

extern "C" attn_status attn_append_kv(attn_plan_t plan, const void* k_new, const void* v_new, void* kv_cache,
                                     void* stream) {
    if (!plan || plan->ragged || plan->graph) return ATTN_ERR_INVALID_ARG;   // no host row list
    if (!plan->bound) return ATTN_ERR_NOT_BOUND;
    if (plan->info.total_qo_rows == 0) return ATTN_OK;
    if (!k_new || !v_new || !kv_cache) return ATTN_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(k_new) | reinterpret_cast<uintptr_t>(v_new) |
         reinterpret_cast<uintptr_t>(kv_cache)) & 15)
        return ATTN_ERR_INVALID_ARG;
    return attn::launch_append_kv(plan, k_new, v_new, kv_cache, static_cast<cudaStream_t>(stream));
}

namespace {
attn_status head_slice(bool unpack, void* kv_cache, int64_t num_pages, int32_t num_kv_heads, int32_t page_size,
                       int32_t head_dim, const int32_t* page_ids, int64_t n_pages, int32_t head_begin,
                       int32_t n_heads, void* buf, int32_t* device_error, void* stream) {
    if (n_pages < 0 || num_pages <= 0 || num_kv_heads <= 0 || page_size <= 0 || head_dim <= 0 ||
        head_dim % 8 != 0 || head_begin < 0 || n_heads <= 0 || head_begin + n_heads > num_kv_heads)
        return ATTN_ERR_INVALID_ARG;
    if (n_pages == 0) return ATTN_OK;
    if (!kv_cache || !buf || !page_ids) return ATTN_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(kv_cache) | reinterpret_cast<uintptr_t>(buf)) & 15)
        return ATTN_ERR_INVALID_ARG;
    return attn::launch_head_slice(unpack, kv_cache, buf, page_ids, n_pages, num_pages, num_kv_heads, page_size,
                                   head_dim, head_begin, n_heads, device_error, static_cast<cudaStream_t>(stream));
}
}  // namespace

extern "C" attn_status attn_pack_kv_heads(const void* kv_cache, int64_t num_pages, int32_t num_kv_heads,
                                         int32_t page_size, int32_t head_dim, const int32_t* page_ids,
                                         int64_t n_pages, int32_t head_begin, int32_t n_heads, void* buf,
                                         int32_t* device_error, void* stream) {
    return head_slice(false, const_cast<void*>(kv_cache), num_pages, num_kv_heads, page_size, head_dim, page_ids,
                      n_pages, head_begin, n_heads, buf, device_error, stream);
}

extern "C" attn_status attn_unpack_kv_heads(const void* buf, int64_t num_pages, int32_t num_kv_heads,
                                           int32_t page_size, int32_t head_dim, const int32_t* page_ids,
                                           int64_t n_pages, int32_t head_begin, int32_t n_heads, void* kv_cache,
                                           int32_t* device_error, void* stream) {
    return head_slice(true, kv_cache, num_pages, num_kv_heads, page_size, head_dim, page_ids, n_pages, head_begin,
                      n_heads, const_cast<void*>(buf), device_error, stream);
}

extern "C" attn_status attn_plan_device_error(attn_plan_t plan, int32_t* code, void* stream) {
    if (!plan || !code) return ATTN_ERR_INVALID_ARG;
    if (!plan->bound) return ATTN_ERR_NOT_BOUND;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int32_t v = 0;
    if (cudaStreamSynchronize(s) != cudaSuccess) return ATTN_ERR_CUDA;
    if (cudaMemcpy(&v, plan->ws + plan->layout.err, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess)
        return ATTN_ERR_CUDA;
    if (v != 0 && cudaMemset(plan->ws + plan->layout.err, 0, sizeof v) != cudaSuccess) return ATTN_ERR_CUDA;
    *code = v;
    return v != 0 ? ATTN_ERR_DEVICE : ATTN_OK;
}

namespace attn {
bool encode_decode_kv_map(void* map, const void* kv_cache, const attn_plan_s* plan) {
    return make_kv_map(map, kv_cache, plan, kBlockTokens);
}
}  // namespace attn
