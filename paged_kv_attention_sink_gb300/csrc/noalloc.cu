// attn_decode_noalloc: attn_decode without a caller-allocated workspace.
//
// Some callers cannot allocate device memory at the point where they run
// attention: an engine that reserves its whole memory budget up front and
// forbids cudaMalloc while it serves (cudaMalloc may also synchronise the
// device and stall every other stream).  attn_decode needs a workspace from
// the caller; this variant instead uses a fixed scratch area compiled into
// the library.
//
// The scratch is one file-scope __device__ array of kNoAllocScratchBytes.  A
// GPU holds it from the moment the library's device code is loaded there
// (with lazy module loading, the first use of this file's code on that GPU)
// until the process exits.  Host code cannot use the array's name as a device
// address, so the first call on each device resolves it with
// cudaGetSymbolAddress (with that device current) and caches the pointer.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "attn_internal.h"
#include "kernels.h"

namespace {

constexpr size_t kNoAllocScratchBytes = 16u << 20;   // 16 MiB per device
using attn::kMaxDevices;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mu;
unsigned char* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set up once per
// device), or nullptr if it cannot be resolved.
unsigned char* scratch_on_current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (g_scratch_ptr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return nullptr;
        }
        g_scratch_ptr[dev] = static_cast<unsigned char*>(p);
    }
    return g_scratch_ptr[dev];
}

}  // namespace

extern "C" attn_status attn_decode_noalloc(attn_plan_t plan, const void* q, const void* kv_cache,
                                           const float* sinks, void* out, float* lse,
                                           void* stream) {
    if (!plan) return ATTN_ERR_INVALID_ARG;
    // A graph plan's work list is built on the device (attn_decode_graph);
    // its host list is empty, so it must not pass for an empty batch.
    if (plan->graph) return ATTN_ERR_INVALID_ARG;
    if (plan->units.empty()) return ATTN_OK;
    if (!q || !kv_cache || !out) return ATTN_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(kv_cache) |
         reinterpret_cast<uintptr_t>(out)) & 15)
        return ATTN_ERR_INVALID_ARG;
    const attn::WorkspaceLayout& L = plan->layout;
    if (L.total > kNoAllocScratchBytes) return ATTN_ERR_WORKSPACE_TOO_SMALL;
    unsigned char* scratch = scratch_on_current_device();
    if (!scratch) return ATTN_ERR_CUDA;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // The array keeps the previous call's contents: upload this plan's work
    // list and zero the split-merge counters and the error word.
    if (cudaMemcpyAsync(scratch + L.units, plan->units.data(),
                        plan->units.size() * sizeof(attn::DecodeUnit), cudaMemcpyHostToDevice,
                        s) != cudaSuccess ||
        cudaMemsetAsync(scratch + L.counters, 0, L.part_lse - L.counters, s) != cudaSuccess) {
        cudaGetLastError();
        return ATTN_ERR_CUDA;
    }
    alignas(64) unsigned char map[128];
    if (!attn::encode_decode_kv_map(map, kv_cache, plan)) return ATTN_ERR_CUDA;
    return attn::launch_decode_scratch(plan, scratch, q, map, sinks, out, lse, s);
}

extern "C" attn_status attn_decode_noalloc_device_error(attn_plan_t plan, int32_t* code, void* stream) {
    if (!plan || !code || plan->graph) return ATTN_ERR_INVALID_ARG;
    const attn::WorkspaceLayout& L = plan->layout;
    if (L.total > kNoAllocScratchBytes) return ATTN_ERR_WORKSPACE_TOO_SMALL;
    unsigned char* scratch = scratch_on_current_device();
    if (!scratch) return ATTN_ERR_CUDA;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return ATTN_ERR_CUDA;
    int32_t v = 0;
    if (cudaMemcpy(&v, scratch + L.err, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return ATTN_ERR_CUDA;
    if (v != 0 && cudaMemset(scratch + L.err, 0, sizeof v) != cudaSuccess) return ATTN_ERR_CUDA;
    *code = v;
    return v != 0 ? ATTN_ERR_DEVICE : ATTN_OK;
}
