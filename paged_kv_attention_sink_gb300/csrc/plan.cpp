// Host-side work planner: turns one ragged batch into the decode units and
// prefill items the kernels run, and lays out the device workspace.
//
// Work is spread over heads and over the KV length ("GPT-OSS on day 0",
// section "Sink Attention"); the cost of a request grows with kv_len for both
// prefill and decode ("Disaggregated prefill and decode", section "Prefill vs
// decode performance"), so decode sequences are cut into chunks of similar
// size until the CTAs fill the GPU, and both lists are ordered longest first.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <new>

#include <cuda_runtime.h>

#include "attn_internal.h"

namespace {

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool supported_head_dim(int d) { return d == 64 || d == 128; }
bool supported_page_size(int p) { return p == 16 || p == 32 || p == 64 || p == 128; }

}  // namespace

namespace attn {

bool current_sm_count(int32_t* out) {
    static std::atomic<int32_t> cache[kMaxDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    if (dev >= 0 && dev < kMaxDevices && cache[dev].load(std::memory_order_relaxed) > 0) {
        *out = cache[dev].load(std::memory_order_relaxed);
        return true;
    }
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) {
        cudaGetLastError();
        return false;
    }
    if (dev >= 0 && dev < kMaxDevices) cache[dev].store(sms, std::memory_order_relaxed);
    *out = sms;
    return true;
}

}  // namespace attn

namespace {

// Shared planner.  Paged: kv_indptr is the page CSR into page_table, kv_len
// comes from the page count and last_page_len.  Ragged: kv_indptr is the token
// CSR into contiguous K / V arrays, every request becomes prefill work items
// (there is no cache to split decode over), and page_table / last_page_len /
// num_pages_in_pool are unused.
attn_status make_plan(bool ragged, const int32_t* qo_indptr, const int32_t* kv_indptr,
                      const int32_t* page_table, const int32_t* last_page_len, int32_t batch,
                      int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
                      int32_t causal, float sm_scale, int32_t num_pages_in_pool, int32_t num_sms,
                      attn_plan_t* plan_out, size_t* workspace_bytes_out) {
    using namespace attn;
    if (!plan_out || !workspace_bytes_out || batch < 0) return ATTN_ERR_INVALID_ARG;
    if (batch > 0 && (!qo_indptr || !kv_indptr || (!ragged && !last_page_len))) return ATTN_ERR_INVALID_ARG;
    if (num_qo_heads <= 0 || num_kv_heads <= 0 || num_qo_heads % num_kv_heads != 0)
        return ATTN_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return ATTN_ERR_INVALID_ARG;
    if (!std::isfinite(sm_scale) || !(sm_scale > 0.f)) return ATTN_ERR_INVALID_ARG;
    if (head_dim <= 0 || page_size <= 0 || num_sms < 0) return ATTN_ERR_INVALID_ARG;
    if (!supported_head_dim(head_dim) || !supported_page_size(page_size)) return ATTN_ERR_UNSUPPORTED;

    // Validate the index arrays and derive kv_len.
    std::vector<int64_t> qo_len(batch), kv_len(batch);
    if (batch > 0 && (qo_indptr[0] != 0 || kv_indptr[0] != 0)) return ATTN_ERR_INVALID_ARG;
    int64_t total_pages = 0;
    for (int32_t b = 0; b < batch; ++b) {
        int64_t nq = (int64_t)qo_indptr[b + 1] - qo_indptr[b];
        int64_t np = (int64_t)kv_indptr[b + 1] - kv_indptr[b];
        if (nq < 0 || np < 0) return ATTN_ERR_INVALID_ARG;
        int64_t kv = 0;
        if (ragged) {
            kv = np;   // tokens
            np = 0;
        } else if (np > 0) {
            if (last_page_len[b] < 1 || last_page_len[b] > page_size) return ATTN_ERR_INVALID_ARG;
            kv = (np - 1) * page_size + last_page_len[b];
        }
        if (nq > kv) return ATTN_ERR_INVALID_ARG;
        if (kv > (int64_t)INT32_MAX / 2) return ATTN_ERR_UNSUPPORTED;
        qo_len[b] = nq;
        kv_len[b] = kv;
        total_pages += np;
    }
    if (total_pages > 0 && (!page_table || num_pages_in_pool <= 0)) return ATTN_ERR_INVALID_ARG;
    const int64_t total_rows = batch > 0 ? qo_indptr[batch] : 0;
    if (total_rows * num_qo_heads > (int64_t)INT32_MAX) return ATTN_ERR_UNSUPPORTED;

    if (num_sms == 0 && !current_sm_count(&num_sms)) return ATTN_ERR_CUDA;

    attn_plan_s* plan = new (std::nothrow) attn_plan_s();
    if (!plan) return ATTN_ERR_INVALID_ARG;
    plan->batch = batch;
    plan->Hq = num_qo_heads;
    plan->Hkv = num_kv_heads;
    plan->D = head_dim;
    plan->P = page_size;
    plan->causal = causal;
    plan->sm_scale = sm_scale;
    plan->num_pages = num_pages_in_pool;
    plan->num_sms = num_sms;
    plan->page_table = page_table;
    plan->ragged = ragged;
    plan->kv_tokens = (ragged && batch > 0) ? kv_indptr[batch] : 0;

    const int G = num_qo_heads / num_kv_heads;
    const int n_slices = (G + kMaxSliceHeads - 1) / kMaxSliceHeads;

    // ---- decode: chunk size so that the units fill about two waves of CTAs.
    int64_t total_blocks = 0;
    int32_t n_decode = 0, n_prefill = 0;
    int64_t decode_tokens = 0, prefill_pairs = 0;
    for (int32_t b = 0; b < batch; ++b) {
        if (qo_len[b] == 1 && !ragged) {
            ++n_decode;
            decode_tokens += kv_len[b];
            total_blocks += (kv_len[b] + kBlockTokens - 1) / kBlockTokens * num_kv_heads * n_slices;
        } else if (qo_len[b] > 1 || (ragged && qo_len[b] == 1)) {
            ++n_prefill;
        }
    }
    const int64_t slots = (int64_t)num_sms * decode_ctas_per_sm(head_dim);
    const int64_t target_units = std::max<int64_t>(1, 2 * slots);
    int64_t chunk = (total_blocks + target_units - 1) / target_units;
    chunk = std::min<int64_t>(std::max<int64_t>(chunk, kDecodeMinChunkBlocks), kDecodeMaxChunkBlocks);

    // Chunks of each request (every KV head and head slice of a request has
    // the same chunks): [c * nblk / n, (c + 1) * nblk / n) blocks.  Split
    // groups are numbered in (request, KV head, slice) order, each group's
    // partial slots contiguous.
    struct Piece { int32_t b, c, n, t0, t1, group0, partial0; };
    std::vector<Piece> pieces;
    pieces.reserve((size_t)n_decode * 4);
    const int32_t per_request = num_kv_heads * n_slices;   // (KV head, slice) pairs
    for (int32_t b = 0; b < batch; ++b) {
        if (qo_len[b] != 1 || ragged) continue;
        const int64_t nblk = (kv_len[b] + kBlockTokens - 1) / kBlockTokens;
        int64_t n_chunks = std::max<int64_t>(1, (nblk + chunk / 2) / chunk);
        n_chunks = std::max<int64_t>(n_chunks, (nblk + kDecodeMaxChunkBlocks - 1) / kDecodeMaxChunkBlocks);
        int32_t group0 = -1, partial0 = 0;
        if (n_chunks > 1) {
            group0 = plan->n_groups;
            partial0 = plan->n_partials;
            plan->n_groups += per_request;
            plan->n_partials += per_request * (int32_t)n_chunks;
        }
        for (int64_t c = 0; c < n_chunks; ++c) {
            const int64_t blk0 = c * nblk / n_chunks, blk1 = (c + 1) * nblk / n_chunks;
            pieces.push_back({b, (int32_t)c, (int32_t)n_chunks, (int32_t)(blk0 * kBlockTokens),
                              (int32_t)std::min<int64_t>(kv_len[b], blk1 * kBlockTokens), group0, partial0});
        }
    }
    // Longest first (equal lengths keep request order), then every (KV head,
    // slice) of a chunk in turn.
    std::stable_sort(pieces.begin(), pieces.end(),
                     [](const Piece& x, const Piece& y) { return (x.t1 - x.t0) > (y.t1 - y.t0); });
    plan->units.resize(pieces.size() * (size_t)per_request);
    DecodeUnit* out = plan->units.data();
    for (const Piece& pc : pieces) {
        DecodeUnit u{};
        u.q_row = qo_indptr[pc.b];
        u.page_base = kv_indptr[pc.b];
        u.tok_begin = pc.t0;
        u.tok_end = pc.t1;
        u.chunk = pc.c;
        u.n_chunks = pc.n;
        u.group = -1;
        for (int32_t g = 0, k = 0; g < num_kv_heads; ++g) {
            for (int32_t sl = 0; sl < n_slices; ++sl, ++k) {
                u.kv_head = g;
                u.head0 = g * G + sl * kMaxSliceHeads;
                u.n_heads = std::min(kMaxSliceHeads, G - sl * kMaxSliceHeads);
                if (pc.n > 1) {
                    u.group = pc.group0 + k;
                    u.partial0 = pc.partial0 + k * pc.n;
                }
                *out++ = u;
            }
        }
    }

    // ---- prefill: one item per (128-row tile, pair of query heads of a group),
    // visiting 128-key KV tiles up to the causal diagonal.
    for (int32_t b = 0; b < batch; ++b) {
        if (qo_len[b] == 0 || (qo_len[b] == 1 && !ragged)) continue;
        const int64_t prefix = kv_len[b] - qo_len[b];
        for (int64_t r = 0; r < qo_len[b]; ++r)
            prefill_pairs += causal ? (prefix + r + 1) : kv_len[b];
        for (int64_t t0 = 0; t0 < qo_len[b]; t0 += kPrefillRows) {
            const int32_t rows = (int32_t)std::min<int64_t>(kPrefillRows, qo_len[b] - t0);
            const int64_t pos0 = prefix + t0;
            const int64_t key_end = causal ? std::min<int64_t>(kv_len[b], pos0 + rows) : kv_len[b];
            for (int32_t g = 0; g < num_kv_heads; ++g) {
                for (int hp = 0; hp < G; hp += 2) {
                    PrefillItem it{};
                    it.q_row0 = (int32_t)(qo_indptr[b] + t0);
                    it.n_rows = rows;
                    it.page_base = kv_indptr[b];
                    it.kv_len = (int32_t)kv_len[b];
                    it.pos0 = (int32_t)pos0;
                    it.kv_head = g;
                    it.head0 = g * G + hp;
                    it.n_heads = std::min(2, G - hp);
                    it.n_kv_tiles = (int32_t)((key_end + kPrefillKeys - 1) / kPrefillKeys);
                    it.key_end = (int32_t)key_end;
                    plan->items.push_back(it);
                }
            }
        }
    }
    // Persistent prefill CTAs: greedy longest-processing-time assignment of
    // the items (longest first, each to the least-loaded CTA); each CTA's items
    // are stored contiguously, longest first.
    std::stable_sort(plan->items.begin(), plan->items.end(),
                     [](const PrefillItem& a, const PrefillItem& b) {
                         return a.n_kv_tiles * a.n_heads > b.n_kv_tiles * b.n_heads;
                     });
    if (!plan->items.empty()) {
        const int ctas = (int)std::min<int64_t>(num_sms, (int64_t)plan->items.size());
        std::vector<std::vector<PrefillItem>> per(ctas);
        std::vector<std::pair<int64_t, int>> heap;   // (load, cta), min-heap
        for (int c = 0; c < ctas; ++c) heap.push_back({0, c});
        auto cmp = [](const std::pair<int64_t, int>& x, const std::pair<int64_t, int>& y) { return x > y; };
        std::make_heap(heap.begin(), heap.end(), cmp);
        for (const PrefillItem& it : plan->items) {
            std::pop_heap(heap.begin(), heap.end(), cmp);
            auto& least = heap.back();
            per[least.second].push_back(it);
            least.first += (int64_t)it.n_kv_tiles * it.n_heads + 1;   // +1: per-item overhead
            std::push_heap(heap.begin(), heap.end(), cmp);
        }
        plan->items.clear();
        plan->item_off.assign(1, 0);
        for (int c = 0; c < ctas; ++c) {
            plan->items.insert(plan->items.end(), per[c].begin(), per[c].end());
            plan->item_off.push_back((int32_t)plan->items.size());
        }
        plan->prefill_ctas = ctas;
    }

    // ---- KV append: cache position of every query row (the row's token is
    // appended at t = kv_len - qo_len + i): page-table slot and row in page.
    plan->append_slots.resize(ragged ? 0 : (size_t)total_rows * 2);
    for (int32_t b = 0; b < batch && !ragged; ++b) {
        for (int64_t i = 0; i < qo_len[b]; ++i) {
            const int64_t t = kv_len[b] - qo_len[b] + i;
            const int64_t r = qo_indptr[b] + i;
            plan->append_slots[2 * r] = (int32_t)(kv_indptr[b] + t / page_size);
            plan->append_slots[2 * r + 1] = (int32_t)(t % page_size);
        }
    }

    // ---- workspace layout (every region 256-byte aligned).
    WorkspaceLayout& L = plan->layout;
    size_t off = 0;
    L.units = off;    off = align_up(off + plan->units.size() * sizeof(DecodeUnit), 256);
    L.items = off;    off = align_up(off + plan->items.size() * sizeof(PrefillItem), 256);
    L.append = off;   off = align_up(off + plan->append_slots.size() * sizeof(int32_t), 256);
    L.item_off = off; off = align_up(off + plan->item_off.size() * sizeof(int32_t), 256);
    L.counters = off; off = align_up(off + (size_t)plan->n_groups * sizeof(int32_t), 256);
    L.err = off;      off = align_up(off + sizeof(int32_t), 256);
    L.n_units = off;  off = align_up(off + sizeof(int32_t), 256);
    L.part_lse = off; off = align_up(off + (size_t)plan->n_partials * kMaxSliceHeads * sizeof(float), 256);
    L.part_o = off;   off = align_up(off + (size_t)plan->n_partials * kMaxSliceHeads * head_dim * sizeof(float), 256);
    L.total = off;

    attn_plan_info& I = plan->info;
    I.batch = batch;
    I.total_qo_rows = (int32_t)total_rows;
    I.num_decode_requests = n_decode;
    I.num_prefill_requests = n_prefill;
    I.num_decode_units = (int32_t)plan->units.size();
    I.num_decode_groups_split = plan->n_groups;
    I.num_decode_partials = plan->n_partials;
    I.decode_chunk_blocks = (int32_t)chunk;
    I.num_prefill_items = (int32_t)plan->items.size();
    I.num_sms = num_sms;
    I.decode_kv_tokens = decode_tokens;
    I.prefill_pairs = prefill_pairs;
    I.workspace_bytes = L.total;

    *plan_out = plan;
    *workspace_bytes_out = L.total;
    return ATTN_OK;
}

}  // namespace

extern "C" attn_status attn_plan(const int32_t* qo_indptr, const int32_t* kv_indptr,
                                 const int32_t* page_table, const int32_t* last_page_len,
                                 int32_t batch, int32_t num_qo_heads, int32_t num_kv_heads,
                                 int32_t head_dim, int32_t page_size, int32_t causal,
                                 float sm_scale, int32_t num_pages_in_pool, int32_t num_sms,
                                 attn_plan_t* plan_out, size_t* workspace_bytes_out) {
    return make_plan(false, qo_indptr, kv_indptr, page_table, last_page_len, batch, num_qo_heads, num_kv_heads,
                     head_dim, page_size, causal, sm_scale, num_pages_in_pool, num_sms, plan_out,
                     workspace_bytes_out);
}

extern "C" attn_status attn_plan_ragged(const int32_t* qo_indptr, const int32_t* kv_indptr, int32_t batch,
                                        int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim,
                                        int32_t causal, float sm_scale, int32_t num_sms, attn_plan_t* plan_out,
                                        size_t* workspace_bytes_out) {
    return make_plan(true, qo_indptr, kv_indptr, nullptr, nullptr, batch, num_qo_heads, num_kv_heads, head_dim,
                     attn::kPrefillKeys, causal, sm_scale, 0, num_sms, plan_out, workspace_bytes_out);
}

extern "C" attn_status attn_plan_get_info(attn_plan_t plan, attn_plan_info* info) {
    if (!plan || !info) return ATTN_ERR_INVALID_ARG;
    *info = plan->info;
    return ATTN_OK;
}

extern "C" attn_status attn_plan_get_decode_units(attn_plan_t plan, int32_t* units, int64_t capacity) {
    if (!plan || (!units && capacity > 0) || capacity < 0) return ATTN_ERR_INVALID_ARG;
    const int64_t n = std::min<int64_t>(capacity, (int64_t)plan->units.size());
    if (n > 0) std::memcpy(units, plan->units.data(), (size_t)n * sizeof(attn::DecodeUnit));
    return ATTN_OK;
}

extern "C" attn_status attn_plan_get_prefill_items(attn_plan_t plan, int32_t* items, int64_t capacity) {
    if (!plan || (!items && capacity > 0) || capacity < 0) return ATTN_ERR_INVALID_ARG;
    const int64_t n = std::min<int64_t>(capacity, (int64_t)plan->items.size());
    if (n > 0) std::memcpy(items, plan->items.data(), (size_t)n * sizeof(attn::PrefillItem));
    return ATTN_OK;
}

extern "C" void attn_plan_destroy(attn_plan_t plan) { delete plan; }

extern "C" const char* attn_status_string(attn_status status) {
    switch (status) {
        case ATTN_OK: return "ok";
        case ATTN_ERR_INVALID_ARG: return "invalid argument";
        case ATTN_ERR_UNSUPPORTED: return "unsupported shape";
        case ATTN_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
        case ATTN_ERR_CUDA: return "CUDA error";
        case ATTN_ERR_NOT_BOUND: return "workspace not bound";
        case ATTN_ERR_DEVICE: return "device-side error recorded";
    }
    return "unknown status";
}

extern "C" attn_status attn_graph_plan(int32_t max_batch, int32_t num_qo_heads, int32_t num_kv_heads,
                                       int32_t head_dim, int32_t page_size, float sm_scale,
                                       int32_t num_pages_in_pool, int64_t max_kv_tokens,
                                       const int32_t* page_table, int32_t num_sms, attn_plan_t* plan_out,
                                       size_t* workspace_bytes_out) {
    using namespace attn;
    if (!plan_out || !workspace_bytes_out || max_batch <= 0 || !page_table || num_pages_in_pool <= 0)
        return ATTN_ERR_INVALID_ARG;
    if (num_qo_heads <= 0 || num_kv_heads <= 0 || num_qo_heads % num_kv_heads != 0) return ATTN_ERR_INVALID_ARG;
    if (!std::isfinite(sm_scale) || !(sm_scale > 0.f) || page_size <= 0 || num_sms < 0 || max_kv_tokens < 0)
        return ATTN_ERR_INVALID_ARG;
    if (!supported_head_dim(head_dim) || !supported_page_size(page_size)) return ATTN_ERR_UNSUPPORTED;
    if ((int64_t)max_batch * num_qo_heads > (int64_t)INT32_MAX) return ATTN_ERR_UNSUPPORTED;
    if (max_batch > kGraphMaxBatch) return ATTN_ERR_UNSUPPORTED;   // the device planner's shared memory
    if (num_sms == 0 && !current_sm_count(&num_sms)) return ATTN_ERR_CUDA;
    // Capacity of the device-built work list.  With the host planner's rule
    // (chunk >= total blocks / target, at most 512 blocks, each request at
    // least one chunk per head slice) the units never exceed
    //   target + (batch + kv_blocks / 512 + 1) * Hkv * slices,
    // kv_blocks bounded by the tokens the batch may hold in total (default:
    // the whole pool) plus one partial block per request.
    const int64_t kv_tokens = max_kv_tokens > 0 ? max_kv_tokens : (int64_t)num_pages_in_pool * page_size;
    const int64_t slices = (num_qo_heads / num_kv_heads + kMaxSliceHeads - 1) / kMaxSliceHeads;
    const int64_t target = 2LL * num_sms * decode_ctas_per_sm(head_dim);
    const int64_t kv_blocks = kv_tokens / kBlockTokens + max_batch;
    const int64_t cap_units = target + (max_batch + kv_blocks / kDecodeMaxChunkBlocks + 1) * num_kv_heads * slices;
    const int64_t cap_groups = (int64_t)max_batch * num_kv_heads * slices;
    if (cap_units > (int64_t)INT32_MAX / kMaxSliceHeads / 256) return ATTN_ERR_UNSUPPORTED;

    attn_plan_s* plan = new (std::nothrow) attn_plan_s();
    if (!plan) return ATTN_ERR_INVALID_ARG;
    plan->graph = true;
    plan->batch = max_batch;
    plan->Hq = num_qo_heads;
    plan->Hkv = num_kv_heads;
    plan->D = head_dim;
    plan->P = page_size;
    plan->causal = 1;
    plan->sm_scale = sm_scale;
    plan->num_pages = num_pages_in_pool;
    plan->num_sms = num_sms;
    plan->page_table = page_table;
    plan->n_partials = (int32_t)cap_units;
    plan->n_groups = (int32_t)cap_groups;
    plan->graph_kv_blocks = kv_blocks;

    WorkspaceLayout& L = plan->layout;
    size_t off = 0;
    L.units = off;    off = align_up(off + (size_t)cap_units * sizeof(DecodeUnit), 256);
    L.items = off;
    L.item_off = off;
    L.append = off;
    L.counters = off; off = align_up(off + (size_t)(2 + cap_groups) * sizeof(int32_t), 256);
    L.err = off;      off = align_up(off + sizeof(int32_t), 256);
    L.n_units = off;  off = align_up(off + sizeof(int32_t), 256);
    L.part_lse = off; off = align_up(off + (size_t)cap_units * kMaxSliceHeads * sizeof(float), 256);
    L.part_o = off;   off = align_up(off + (size_t)cap_units * kMaxSliceHeads * head_dim * sizeof(float), 256);
    L.total = off;

    attn_plan_info& I = plan->info;
    I.batch = max_batch;
    I.total_qo_rows = max_batch;
    I.num_decode_requests = max_batch;
    I.num_decode_groups_split = (int32_t)cap_groups;
    I.num_decode_partials = (int32_t)cap_units;
    I.num_sms = num_sms;
    I.workspace_bytes = L.total;
    *plan_out = plan;
    *workspace_bytes_out = L.total;
    return ATTN_OK;
}
