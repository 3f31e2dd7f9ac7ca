// Launchers of the CUDA kernels (one per translation unit).
#pragma once

#include <cuda_runtime.h>

#include "attn_internal.h"

namespace attn {

// kv_map / q_map point at CUtensorMap objects built by the API layer.
attn_status launch_decode(attn_plan_s* plan, const void* q, const void* kv_map, const float* sinks,
                          void* out, float* lse, cudaStream_t stream);
// v_map: the V tensor map of a ragged plan (NULL for a paged plan); o_map:
// `out` with the same layout and box as q_map (full 128-row tiles are stored
// through it).
attn_status launch_prefill(attn_plan_s* plan, const void* q_map, const void* kv_map, const void* v_map,
                           const void* o_map, const float* sinks, void* out, float* lse, cudaStream_t stream);
// in_f32 / out_f32: value states / merged values are fp32 (else bf16).
attn_status launch_merge_states(const void* va, const float* lsea, const void* vb, const float* lseb, void* vout,
                                float* lseout, int64_t rows, int head_dim, bool in_f32, bool out_f32,
                                cudaStream_t stream);
// CUDA-graph decode: device planner + persistent decode over its work list.
attn_status launch_decode_graph(attn_plan_s* plan, const int32_t* kv_indptr, const int32_t* last_page_len,
                                const int32_t* batch, const void* q, const void* kv_map, const float* sinks,
                                void* out, float* lse, cudaStream_t stream);
// New K/V rows of the plan's query rows into their HND page slots.
attn_status launch_append_kv(attn_plan_s* plan, const void* k_new, const void* v_new, void* kv_cache,
                             cudaStream_t stream);
// Heads [h0, h0 + nh) of pages page_ids[0..n) <-> buf[n][2][nh][P][D].
attn_status launch_head_slice(bool unpack, void* kv_cache, void* buf, const int32_t* page_ids, int64_t n,
                              int64_t num_pages, int32_t Hkv, int32_t P, int32_t D, int32_t h0, int32_t nh,
                              int32_t* err, cudaStream_t stream);

}  // namespace attn

namespace attn {

// Same decode launch as launch_decode, but with the plan's device work list,
// partial states, merge counters and error word taken from `scratch` (laid
// out as the plan's workspace) instead of the bound workspace.
attn_status launch_decode_scratch(attn_plan_s* plan, unsigned char* scratch, const void* q,
                                  const void* kv_map, const float* sinks, void* out, float* lse,
                                  cudaStream_t stream);

// Build the decode kernel's KV tensor map for `kv_cache` into `map` (128 bytes,
// 64-byte aligned).  Returns false if the driver rejects it.
bool encode_decode_kv_map(void* map, const void* kv_cache, const attn_plan_s* plan);

}  // namespace attn
