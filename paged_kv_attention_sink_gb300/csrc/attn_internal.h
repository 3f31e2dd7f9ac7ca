// Internal declarations shared by the planner (host) and the kernels.
#pragma once

#include <atomic>
#include <cstddef>
#include <cstdint>
#include <vector>

#include <cuda_runtime.h>

#include "../../include/attn.h"

namespace attn {

constexpr int kBlockTokens = 16;          // decode streams K/V in 16-token blocks
constexpr int kMaxSliceHeads = 16;        // query heads per decode CTA (one m16 MMA tile)
constexpr int kDecodeWarps = 4;           // warps per decode CTA
constexpr int kDecodeMinChunkBlocks = 8;  // never split a sequence finer than 128 tokens
constexpr int kDecodeMaxChunkBlocks = 512;
constexpr int kDecodeMaxChunkPages = kDecodeMaxChunkBlocks * kBlockTokens / 16 + 2;
constexpr int kPrefillRows = 128;         // query rows per prefill tile (TMEM lanes)
constexpr int kPrefillOutRows = 32;       // rows per output TMA store (one softmax warp's stripe)
constexpr int kPrefillKeys = 128;         // keys per prefill KV tile
constexpr int kGraphMaxBatch = 4096;      // attn_graph_plan: requests the device planner can order

// One decode CTA: a chunk [tok_begin, tok_end) of one request's KV sequence for
// one KV head and up to 16 of its query heads.
struct DecodeUnit {
    int32_t q_row;      // row of q / out / lse
    int32_t page_base;  // kv_indptr[b]: first slot of the request in page_table
    int32_t kv_head;
    int32_t head0;      // first query head of the slice
    int32_t n_heads;    // query heads in the slice (1..16)
    int32_t tok_begin;  // a multiple of 16
    int32_t tok_end;    // <= kv_len
    int32_t chunk;      // index of this chunk within its group; chunk 0 carries the sink
    int32_t n_chunks;   // 1 = not split
    int32_t group;      // split-merge counter index, -1 when not split
    int32_t partial0;   // first partial-state slot of the group
    int32_t reserved;
};
static_assert(sizeof(DecodeUnit) == 48, "decode unit is 12 int32");

// One prefill CTA: 128 query rows of one request for up to two query heads of
// one GQA group.
struct PrefillItem {
    int32_t q_row0;      // first row of the tile in q / out / lse
    int32_t n_rows;      // valid rows (1..128)
    int32_t page_base;
    int32_t kv_len;
    int32_t pos0;        // absolute position of row 0 (kv_len - qo_len + tile offset)
    int32_t kv_head;
    int32_t head0;
    int32_t n_heads;     // 1 or 2
    int32_t n_kv_tiles;  // 128-key KV tiles visited
    int32_t key_end;     // one past the last key any row of the tile may see
    int32_t reserved0;
    int32_t reserved1;
};
static_assert(sizeof(PrefillItem) == 48, "prefill item is 12 int32");

struct WorkspaceLayout {
    size_t units = 0, items = 0, item_off = 0, append = 0, counters = 0, err = 0, n_units = 0, part_lse = 0,
           part_o = 0, total = 0;
};

// CTAs of the decode kernel resident per SM for a head dim (matches its
// shared-memory footprint); defined next to the kernel.
int decode_ctas_per_sm(int head_dim);

// SM count of the current device, queried once per device (thread-safe).
bool current_sm_count(int32_t* out);

// Device ordinals that the per-device caches below cover; a higher ordinal
// is served without a cache.
constexpr int kMaxDevices = 64;

// Runs `setup` (returning cudaError_t) until it first succeeds on the current
// device, then only checks a flag.  Kernel attributes such as the dynamic
// shared-memory limit belong to one device's context, so a process that
// drives several devices sets them on each.  Two threads may both run setup
// the first time; it must be idempotent.
template <class F>
cudaError_t once_per_device(std::atomic<bool> (&done)[kMaxDevices], F&& setup) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const bool cached = dev >= 0 && dev < kMaxDevices;
    if (cached && done[dev].load(std::memory_order_acquire)) return cudaSuccess;
    e = setup();
    if (e == cudaSuccess && cached) done[dev].store(true, std::memory_order_release);
    return e;
}

}  // namespace attn

struct attn_plan_s {
    int32_t batch = 0, Hq = 0, Hkv = 0, D = 0, P = 0, causal = 0;
    float sm_scale = 0.f;
    int32_t num_pages = 0;
    int32_t num_sms = 0;
    const int32_t* page_table = nullptr;  // device, borrowed
    bool ragged = false;                  // contiguous K / V (attn_plan_ragged), no page table
    bool graph = false;                   // attn_graph_plan: decode work list built on the device
                                          // (batch = max batch; n_partials / n_groups = capacities)
    int64_t kv_tokens = 0;                // ragged: rows of K and V (kv_indptr[batch])
    int64_t graph_kv_blocks = 0;          // graph: 16-token blocks a batch may hold in total

    std::vector<attn::DecodeUnit> units;
    std::vector<attn::PrefillItem> items;
    std::vector<int32_t> append_slots;    // per query row: page-table slot, row in page
    std::vector<int32_t> item_off;        // CTA c runs items [item_off[c], item_off[c+1])
    int32_t prefill_ctas = 0;
    int32_t n_groups = 0;
    int32_t n_partials = 0;
    attn_plan_info info{};
    attn::WorkspaceLayout layout;

    unsigned char* ws = nullptr;  // device, caller-owned
    size_t ws_bytes = 0;
    bool bound = false;

    // Tensor maps are 128-byte opaque driver objects; cached per KV / Q pointer.
    alignas(64) unsigned char kv_map_decode[128];
    const void* kv_map_decode_ptr = nullptr;
    alignas(64) unsigned char kv_map_prefill[128];
    const void* kv_map_prefill_ptr = nullptr;
    alignas(64) unsigned char q_map_prefill[128];
    const void* q_map_prefill_ptr = nullptr;
    alignas(64) unsigned char v_map_prefill[128];   // ragged: K in kv_map_prefill, V here
    const void* v_map_prefill_ptr = nullptr;
    alignas(64) unsigned char o_map_prefill[128];   // out, laid out like q, 32-row boxes
    const void* o_map_prefill_ptr = nullptr;
};
