// Launchers of the CUDA kernels (one per translation unit).
#pragma once

#include <cuda_runtime.h>

#include "attn_internal.h"

namespace attn {

// kv_map / q_map point at CUtensorMap objects built by the API layer.
attn_status launch_decode(attn_plan_s* plan, const void* q, const void* kv_map, const float* sinks,
                          void* out, float* lse, cudaStream_t stream);
attn_status launch_prefill(attn_plan_s* plan, const void* q_map, const void* kv_map,
                           const float* sinks, void* out, float* lse, cudaStream_t stream);
attn_status launch_merge_states(const void* va, const float* lsea, const void* vb,
                                const float* lseb, void* vout, float* lseout, int64_t rows,
                                int head_dim, cudaStream_t stream);

}  // namespace attn
