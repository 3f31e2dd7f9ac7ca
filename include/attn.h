/*
 * attn.h -- C ABI of libattn.so: batched GQA attention with a per-head sink
 * logit over a paged KV cache, for one NVIDIA GB300 GPU (sm_103a).
 *
 * What is computed.  "GPT-OSS on day 0" (Perplexity), section "Sink
 * Attention": every query head h owns one learned sink logit that takes part
 * in the softmax.  It enters the denominator only (its value vector is zero)
 * and is not multiplied by sm_scale:
 *
 *   out[i,h] = sum_j exp(s_ij - m) v_j / (sum_j exp(s_ij - m) + exp(sink_h - m))
 *   s_ij     = sm_scale * q[i,h] . k_j            (k, v of KV head h / (Hq/Hkv))
 *   lse[i,h] = m + ln(sum_j exp(s_ij - m) + exp(sink_h - m))   (natural log)
 *
 * The same section describes the kernels as parallel over heads and over the
 * KV length, with the softmax computed online (running max and scale) and
 * the sink placed in the first part of a KV split only; this library does
 * exactly that (split-KV decode with a log-sum-exp merge).
 *
 * Request model, "Disaggregated prefill and decode" (Perplexity), section
 * "Prefill vs decode performance": request b forwards qo_len_b query tokens
 * and reads kv_len_b tokens from the KV cache; decode has qo_len = 1.  Query
 * i of request b sits at absolute position kv_len_b - qo_len_b + i, so with
 * causal masking it sees keys j <= kv_len_b - qo_len_b + i.
 *
 * KV cache layout, "Hosting Qwen on Blackwell" (Perplexity), section
 * "Deploying on GB200 NVL72", and "Disaggregated prefill and decode", section
 * "Sharded KV transfer": HND pages, heads outer and each page's tokens
 * contiguous.  Concretely one pool, bf16, row-major:
 *
 *   kv_cache[num_pages][2][Hkv][page_size][head_dim]      ([.][0] = K, [.][1] = V)
 *
 * Tensors (all caller-owned device memory, row-major, contiguous):
 *   q, out   bf16  [total_qo_rows][Hq][head_dim]   total_qo_rows = qo_indptr[batch]
 *   lse      fp32  [total_qo_rows][Hq]             natural log; may be NULL
 *   sinks    fp32  [Hq]                            may be NULL (no sink, i.e. -inf)
 *
 * Threading and streams: every launch is asynchronous on the caller's
 * cudaStream_t, passed as void* (NULL = legacy default stream).  A plan may be
 * used from one host thread at a time.  Launches that share a plan's
 * workspace must not overlap on the GPU (issue them on one stream).
 *
 * Errors: functions return attn_status and never abort or throw.  Argument
 * and shape checks happen on the host before anything is launched.  Kernels
 * never trap: a page id outside the pool or a wait that runs out is recorded
 * in a device error word of the plan's workspace (read it with
 * attn_plan_device_error) and the offending load is skipped.
 */
#ifndef ATTN_H
#define ATTN_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define ATTN_API __attribute__((visibility("default")))
#else
#define ATTN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_INVALID_ARG = 1,          /* malformed pointer, size or index array */
    ATTN_ERR_UNSUPPORTED = 2,          /* well-formed but outside the supported shapes */
    ATTN_ERR_WORKSPACE_TOO_SMALL = 3,  /* bound workspace smaller than required */
    ATTN_ERR_CUDA = 4,                 /* a CUDA runtime/driver call failed */
    ATTN_ERR_NOT_BOUND = 5,            /* launch before attn_plan_bind_workspace */
    ATTN_ERR_DEVICE = 6                /* a kernel recorded an error (see device error bits) */
} attn_status;

/* Bits of the device error word (attn_plan_device_error). */
#define ATTN_DEVICE_ERR_PAGE_ID 1      /* page id outside [0, num_pages_in_pool) */
#define ATTN_DEVICE_ERR_TIMEOUT 2      /* a bounded wait inside a kernel ran out */
#define ATTN_DEVICE_ERR_PLAN 4         /* attn_decode_graph: malformed request metadata or
                                          work beyond the graph plan's capacity */

/* Opaque plan; owned by the library, freed with attn_plan_destroy. */
typedef struct attn_plan_s* attn_plan_t;

/* Summary of a plan (host-side copy, for callers and tests). */
typedef struct {
    int32_t batch;
    int32_t total_qo_rows;
    int32_t num_decode_requests;     /* requests with qo_len == 1 */
    int32_t num_prefill_requests;    /* requests with qo_len > 1 */
    int32_t num_decode_units;        /* CTAs of one attn_decode launch */
    int32_t num_decode_groups_split; /* (request, kv head, head slice) groups split over >1 chunk */
    int32_t num_decode_partials;     /* partial states held in the workspace */
    int32_t decode_chunk_blocks;     /* target split-KV chunk, in 16-token blocks */
    int32_t num_prefill_items;       /* CTAs of one attn_prefill launch */
    int32_t num_sms;                 /* SM count the plan was balanced for */
    int64_t decode_kv_tokens;        /* sum of kv_len over decode requests */
    int64_t prefill_pairs;           /* visible (query, key) pairs over prefill rows, per query head */
    size_t workspace_bytes;
} attn_plan_info;

/*
 * attn_plan -- build the work list of one batch (host only; launches nothing).
 *
 * The split of the work over heads and over the KV length follows "GPT-OSS on
 * day 0", section "Sink Attention"; the qo_len / kv_len request model follows
 * "Disaggregated prefill and decode", section "Prefill vs decode performance".
 * Requests with qo_len == 1 are decode requests (attn_decode), requests with
 * qo_len > 1 are prefill requests (attn_prefill); qo_len == 0 contributes no
 * rows.  Long decode sequences are split into chunks of whole 16-token blocks
 * so that the number of CTAs fills num_sms SMs; chunk 0 of each split carries
 * the sink and the chunks are merged by log-sum-exp inside the same launch.
 *
 *   qo_indptr      host int32 [batch+1]; qo_indptr[0] = 0, non-decreasing
 *   kv_indptr      host int32 [batch+1]; CSR offsets of each request's pages in
 *                  page_table; kv_indptr[0] = 0, non-decreasing
 *   page_table     DEVICE int32 [kv_indptr[batch]]; page ids into the pool.
 *                  Borrowed: it must stay valid, unchanged, for every launch
 *                  made with this plan.  Not read by attn_plan.
 *   last_page_len  host int32 [batch]; tokens used in the request's last page,
 *                  1..page_size (ignored for a request with no pages);
 *                  kv_len = (n_pages - 1) * page_size + last_page_len
 *   batch >= 0; num_qo_heads % num_kv_heads == 0 (query head h reads KV head
 *   h / (num_qo_heads / num_kv_heads)); head_dim in {64, 128}; page_size in
 *   {16, 32, 64, 128}; qo_len <= kv_len for every request; causal in {0, 1};
 *   sm_scale finite; num_pages_in_pool > 0 when any request has pages;
 *   num_sms > 0, or 0 to query the current CUDA device.
 *
 * On success *plan_out owns host memory only and *workspace_bytes_out is the
 * size of the device workspace the plan needs.  Nothing is written on error.
 */
ATTN_API attn_status attn_plan(const int32_t* qo_indptr, const int32_t* kv_indptr,
                      const int32_t* page_table, const int32_t* last_page_len,
                      int32_t batch, int32_t num_qo_heads, int32_t num_kv_heads,
                      int32_t head_dim, int32_t page_size, int32_t causal, float sm_scale,
                      int32_t num_pages_in_pool, int32_t num_sms, attn_plan_t* plan_out,
                      size_t* workspace_bytes_out);

/*
 * attn_plan_bind_workspace -- attach caller-owned device memory to the plan
 * and upload the work list into it (asynchronous copy on `stream`; the host
 * copy stays valid).  `workspace` must be 256-byte aligned and hold at least
 * the plan's workspace_bytes; it is used by every later launch of the plan
 * and must outlive them.  Clears the device error word and the split-merge
 * counters.  May be called again (e.g. with other memory).
 */
ATTN_API attn_status attn_plan_bind_workspace(attn_plan_t plan, void* workspace, size_t bytes,
                                     void* stream);

/*
 * attn_decode -- sink attention for the plan's decode rows (qo_len == 1):
 * one CTA per (request, KV head, head slice, KV chunk); the GQA group's query
 * heads share every K/V tile read from HBM.  Writes out and lse rows of
 * decode requests only.  Pointers as in the file comment.
 */
ATTN_API attn_status attn_decode(attn_plan_t plan, const void* q, const void* kv_cache,
                        const float* sinks, void* out, float* lse, void* stream);

/*
 * attn_prefill -- sink attention for the plan's prefill rows (qo_len > 1),
 * causal or not as planned: one CTA per (128-row query tile, pair of query
 * heads of one GQA group), QK^T and PV on the tensor cores.  Writes out and
 * lse rows of prefill requests only.  For a mixed batch call attn_prefill
 * and attn_decode with the same plan, in either order, on one stream.
 */
ATTN_API attn_status attn_prefill(attn_plan_t plan, const void* q, const void* kv_cache,
                         const float* sinks, void* out, float* lse, void* stream);

/*
 * attn_plan_ragged / attn_prefill_ragged -- the same sink attention over
 * contiguous, unpadded K and V with no KV cache, for embedding-style serving
 * ("Fast embeddings on GPUs" (Perplexity), section "ROSE": with no KV cache
 * the attention kernels take ragged inputs so that nothing is padded).
 *
 *   qo_indptr  host int32 [batch + 1]: request b's query rows
 *   kv_indptr  host int32 [batch + 1]: request b's rows of k and v (tokens,
 *              not pages); qo_len <= kv_len, queries aligned to the end of
 *              the keys for the causal mask as in attn_plan
 *   q, out     bf16 [qo_indptr[batch]][Hq][head_dim]
 *   k, v       bf16 [kv_indptr[batch]][Hkv][head_dim] (16-byte aligned)
 *   sinks, lse as in attn_prefill
 * Every request (qo_len = 1 included) runs on the tcgen05 prefill kernel; the
 * plan has no decode work (attn_decode on it does nothing) and cannot be used
 * with attn_prefill or attn_append_kv (ATTN_ERR_INVALID_ARG).  Workspace and
 * error word as for attn_plan.
 */
ATTN_API attn_status attn_plan_ragged(const int32_t* qo_indptr, const int32_t* kv_indptr, int32_t batch,
                                      int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim,
                                      int32_t causal, float sm_scale, int32_t num_sms, attn_plan_t* plan_out,
                                      size_t* workspace_bytes_out);
ATTN_API attn_status attn_prefill_ragged(attn_plan_t plan, const void* q, const void* k, const void* v,
                                         const float* sinks, void* out, float* lse, void* stream);

/*
 * attn_merge_states -- combine two attention states over disjoint key sets
 * into the state over their union, by the log-sum-exp rule implied by the
 * split along the KV length in "GPT-OSS on day 0", section "Sink Attention"
 * (the pages do not print it):
 *   L = max(lse_a, lse_b);  w_x = exp(lse_x - L)
 *   v_out = (w_a v_a + w_b v_b) / (w_a + w_b);  lse_out = L + ln(w_a + w_b)
 * A state with lse = -inf (no keys, no sink) is the identity.  The sink must
 * be counted in exactly one of the two inputs.
 *
 *   va, vb, vout   bf16 [n_tokens][n_heads][head_dim]  (vout may alias va or vb)
 *   lsea, lseb     fp32 [n_tokens][n_heads], natural log
 *   lseout         fp32 [n_tokens][n_heads] or NULL
 *   head_dim a multiple of 4, at most 256.  Device pointers, async on stream.
 */
ATTN_API attn_status attn_merge_states(const void* va, const float* lsea, const void* vb,
                              const float* lseb, void* vout, float* lseout, int32_t n_tokens,
                              int32_t n_heads, int32_t head_dim, void* stream);

/*
 * attn_merge_states_f32 -- the same log-sum-exp merge for fp32 value states:
 * partial states kept unrounded (a KV sequence split across calls or
 * devices, the sink counted in one part only, as in "GPT-OSS on day 0",
 * section "Sink Attention") merge without rounding each part to bf16 first.
 *   va, vb         fp32 [n_tokens][n_heads][head_dim], 16-byte aligned
 *   lsea, lseb     fp32 [n_tokens][n_heads], natural log
 *   vout           fp32 (vout_bf16 = 0; 16-byte aligned, may alias va or vb)
 *                  or bf16 (vout_bf16 != 0; 8-byte aligned), [n_tokens][n_heads][head_dim]
 *   lseout         fp32 [n_tokens][n_heads] or NULL
 * head_dim a multiple of 4, at most 256.  Device pointers, async on stream;
 * ATTN_ERR_INVALID_ARG for bad sizes, NULL or misaligned pointers.
 */
ATTN_API attn_status attn_merge_states_f32(const float* va, const float* lsea, const float* vb,
                                           const float* lseb, void* vout, int32_t vout_bf16, float* lseout,
                                           int32_t n_tokens, int32_t n_heads, int32_t head_dim, void* stream);

/*
 * attn_decode_noalloc -- attn_decode for callers that cannot allocate device
 * memory when they run attention: an engine that reserves its whole memory
 * budget up front and forbids cudaMalloc while it serves (cudaMalloc may also
 * synchronise the device and so stall every other stream).  No source
 * describes such a call: this is an interface addition.
 *
 * Same arguments and results as attn_decode (host-planned paged plans; a
 * graph plan is refused with ATTN_ERR_INVALID_ARG), but the plan needs no
 * bound workspace: the work list, split-KV partial states, merge counters and
 * error word live in a static 16 MiB device array inside the library.  A GPU
 * holds that array from the moment the library's device code is loaded there
 * (with lazy module loading, the first use of it on that GPU) until the
 * process exits.  Plans whose workspace_bytes exceed 16 MiB are rejected with
 * ATTN_ERR_WORKSPACE_TOO_SMALL.  It allocates nothing (no cudaMalloc /
 * cudaFree): each call uploads the work list with cudaMemcpyAsync from the
 * plan's host memory (pageable, so the call returns once the copy has been
 * staged, which may wait for earlier work on `stream`) and zeroes the counters
 * and the error word with cudaMemsetAsync on `stream`, then launches the
 * decode kernel.  The results are bit-identical to attn_decode's on the same
 * plan and inputs.
 *
 * The first call on a device resolves the array's device address
 * (cudaGetSymbolAddress, with that device current); make that first call
 * before any stream capture.  All calls share the one array and it keeps the
 * last call's contents, so calls that overlap on the GPU (other streams, other
 * host threads) race: serialise them.  Bad page ids are skipped rather than
 * read and, like bounded-wait timeouts, set bits of the array's error word:
 * read it with attn_decode_noalloc_device_error.
 */
ATTN_API attn_status attn_decode_noalloc(attn_plan_t plan, const void* q, const void* kv_cache,
                                         const float* sinks, void* out, float* lse, void* stream);

/*
 * attn_decode_noalloc_device_error -- wait for `stream`, then read and clear
 * the device error word (ATTN_DEVICE_ERR_* bits) that attn_decode_noalloc
 * calls with this plan's layout left in the current device's static array,
 * into *code.  Returns ATTN_ERR_DEVICE if any bit was set, ATTN_ERR_INVALID_ARG
 * for a NULL argument or a graph plan.  The array is shared by every call, so
 * read it before another call on the device may overwrite it.
 */
ATTN_API attn_status attn_decode_noalloc_device_error(attn_plan_t plan, int32_t* code, void* stream);

/*
 * attn_graph_plan / attn_decode_graph -- decode that can be captured in a CUDA
 * graph and replayed for new batches.  The split-KV plan depends on the
 * requests' lengths, so host planning would freeze it at capture; here the
 * work list is built on the device from device-resident metadata, with the
 * same rule as attn_plan (for plans of up to 128 requests by every CTA of the
 * persistent decode grid itself, else by a planner kernel launched first),
 * and a fixed grid of persistent decode CTAs takes the units from a device
 * queue ("Fast embeddings on GPUs"
 * (Perplexity), section "Managing CUDA graphs": kernels that configure their
 * launches from dynamic host inputs prevent full CUDA graphs; the page's fix
 * is to change those kernels so they can be captured).
 *
 * attn_graph_plan sizes a plan once, for at most `max_batch` decode requests
 * whose KV lengths sum to at most `max_kv_tokens` (0: num_pages_in_pool *
 * page_size); bind a workspace with attn_plan_bind_workspace as usual.  The
 * page table pointer is fixed; its contents may change between replays.
 *
 * attn_decode_graph reads, on the device and at run time:
 *   batch          int32 scalar: B <= max_batch decode requests (query row b =
 *                  request b; q / out are [max_batch][Hq][head_dim], lse
 *                  [max_batch][Hq]; rows >= B are not touched)
 *   kv_indptr      int32 [B + 1] page CSR into page_table, kv_indptr[0] = 0
 *   last_page_len  int32 [B], in [1, page_size]
 * No host synchronisation, copy or allocation happens inside the call, so it
 * can be captured (after one uncaptured call has built the TMA descriptor for
 * this kv_cache pointer).  A request with a malformed entry, or a batch beyond
 * the plan's capacity, sets ATTN_DEVICE_ERR_PLAN; such requests (or, past
 * the capacity, the whole step) produce no output.  attn_decode, attn_prefill
 * and attn_append_kv reject graph plans.
 */
ATTN_API attn_status attn_graph_plan(int32_t max_batch, int32_t num_qo_heads, int32_t num_kv_heads,
                                     int32_t head_dim, int32_t page_size, float sm_scale, int32_t num_pages_in_pool,
                                     int64_t max_kv_tokens, const int32_t* page_table, int32_t num_sms,
                                     attn_plan_t* plan_out, size_t* workspace_bytes_out);
ATTN_API attn_status attn_decode_graph(attn_plan_t plan, const int32_t* kv_indptr, const int32_t* last_page_len,
                                       const int32_t* batch, const void* q, const void* kv_cache, const float* sinks,
                                       void* out, float* lse, void* stream);
/*
 * Copy the work list that the last attn_decode_graph built on the device into
 * host memory (12 int32 per unit, as attn_plan_get_decode_units), after
 * synchronising `stream`; *n_units receives the unit count.  For tests and
 * inspection.
 */
ATTN_API attn_status attn_graph_plan_read_units(attn_plan_t plan, int32_t* units, int64_t capacity,
                                                int64_t* n_units, void* stream);

/*
 * attn_append_kv -- write the step's new K and V rows into the paged cache,
 * the step that runs before attention ("Disaggregated prefill and decode"
 * (Perplexity), section "KV Messenger": the model appends a layer's new tokens
 * to its KV cache, and the entries are valid after that append and before
 * attention).  Every query row of the plan is one new token: row i of request
 * b is cache position t = kv_len - qo_len + i (kv_len as given to attn_plan,
 * i.e. counting the new tokens), stored at page page_table[kv_indptr[b] + t/P],
 * row t % P, so the pages must already be allocated in the plan's page table.
 *
 *   k_new, v_new  bf16 [total_qo_rows][Hkv][head_dim], device, 16-byte aligned
 *   kv_cache      bf16 [num_pages][2][Hkv][page_size][head_dim] HND pool,
 *                 device, 16-byte aligned; only the new tokens' rows change
 * Bit-exact copy.  Needs a bound workspace.  Page ids outside [0, num_pages)
 * set ATTN_DEVICE_ERR_PAGE_ID and that row is skipped.  Async on `stream`.
 */
ATTN_API attn_status attn_append_kv(attn_plan_t plan, const void* k_new, const void* v_new, void* kv_cache,
                                    void* stream);

/*
 * attn_pack_kv_heads / attn_unpack_kv_heads -- move a head slice of HND pages
 * to or from one contiguous buffer, the local half of a head-sharded KV
 * transfer ("Disaggregated prefill and decode", section "Sharded KV transfer":
 * pages are split or rebuilt from head slices when sender and receiver shard
 * the cache over attention heads differently, and the HND layout keeps a
 * page's head slice contiguous).  The network part is not in this library.
 *
 *   kv_cache      bf16 [num_pages][2][num_kv_heads][page_size][head_dim], device
 *   page_ids      int32 [n_pages], device: pages to move, in buffer order
 *   buf           bf16 [n_pages][2][n_heads][page_size][head_dim], device
 *   heads         [head_begin, head_begin + n_heads) of num_kv_heads
 *   device_error  optional device int32; ATTN_DEVICE_ERR_PAGE_ID is OR-ed in
 *                 when a page id lies outside [0, num_pages) (that page is
 *                 skipped).  NULL: such pages are skipped silently.
 * Pack reads the pool and writes buf; unpack reads buf and writes only the
 * slice's bytes of the listed pages.  head_dim a multiple of 8; kv_cache and
 * buf 16-byte aligned.  Bit-exact copies.  Async on `stream`.
 */
ATTN_API attn_status attn_pack_kv_heads(const void* kv_cache, int64_t num_pages, int32_t num_kv_heads,
                                        int32_t page_size, int32_t head_dim, const int32_t* page_ids,
                                        int64_t n_pages, int32_t head_begin, int32_t n_heads, void* buf,
                                        int32_t* device_error, void* stream);
ATTN_API attn_status attn_unpack_kv_heads(const void* buf, int64_t num_pages, int32_t num_kv_heads,
                                          int32_t page_size, int32_t head_dim, const int32_t* page_ids,
                                          int64_t n_pages, int32_t head_begin, int32_t n_heads, void* kv_cache,
                                          int32_t* device_error, void* stream);

/* Copy the plan's summary into *info (host only). */
ATTN_API attn_status attn_plan_get_info(attn_plan_t plan, attn_plan_info* info);

/*
 * Host copies of the plan's work lists, for inspection and tests.  Each
 * decode unit is 12 int32: q_row, page_base, kv_head, head0, n_heads,
 * tok_begin, tok_end, chunk, n_chunks, group, partial0, reserved.  Each
 * prefill item is 12 int32: q_row0, n_rows, page_base, kv_len, pos0, kv_head,
 * head0, n_heads, n_kv_tiles, key_end, reserved, reserved (pos0 = absolute
 * position of the tile's first query; key_end = one past the last key any
 * row of the tile may see).  `capacity` counts units/items; at most that many
 * are copied.
 */
ATTN_API attn_status attn_plan_get_decode_units(attn_plan_t plan, int32_t* units, int64_t capacity);
ATTN_API attn_status attn_plan_get_prefill_items(attn_plan_t plan, int32_t* items, int64_t capacity);

/*
 * attn_plan_device_error -- wait for `stream`, then read and clear the plan's
 * device error word (ATTN_DEVICE_ERR_* bits) into *code.  Returns
 * ATTN_ERR_DEVICE if any bit was set.
 */
ATTN_API attn_status attn_plan_device_error(attn_plan_t plan, int32_t* code, void* stream);

/* Free the plan's host memory.  Does not touch the workspace.  NULL is a no-op. */
ATTN_API void attn_plan_destroy(attn_plan_t plan);

/* Static, human-readable name of a status code. */
ATTN_API const char* attn_status_string(attn_status status);

/*
 * attn_selftest_bounded_wait -- diagnostic of the kernels' failure detection.
 * Launches one warp on `stream` that waits, through the same bounded mbarrier
 * wait every kernel uses, on a barrier nothing arrives on.  The wait gives up
 * after its wall-time limit (2 s), and the kernel writes
 * ATTN_DEVICE_ERR_TIMEOUT to result[0] (0 had the wait completed) and the
 * nanoseconds it waited to result[1], then returns; the context stays usable.
 *   result   DEVICE int64 [2], caller-owned
 * Returns ATTN_ERR_INVALID_ARG for a NULL result, ATTN_ERR_CUDA if the launch
 * fails.
 */
ATTN_API attn_status attn_selftest_bounded_wait(int64_t* result, void* stream);

/*
 * attn_selftest_exp2 -- diagnostic of the prefill softmax's exponentials.
 * The online softmax of "GPT-OSS on day 0" (Perplexity), section "Sink
 * Attention", needs exp(s - m) for every visible score; the prefill kernel
 * evaluates it as 2^(s * sm_scale * log2(e) - m) and takes part of each
 * tile's exponentials as a cubic polynomial on the FMA pipe instead of the
 * MUFU's ex2.approx.  This launches, on `stream`, the kernel's own inline
 * polynomial (with the kernel's argument set-up) next to ex2.approx:
 *   y_poly[k] = polynomial 2^(x[k] * scale_log2 - m)   (argument clamped to [-126, 126])
 *   y_mufu[k] = ex2.approx.ftz(x[k] * scale_log2 - m)
 *   x, y_poly, y_mufu   DEVICE fp32 [n], caller-owned
 * Returns ATTN_ERR_INVALID_ARG for n < 0 or NULL arrays (n > 0), ATTN_ERR_CUDA
 * if the launch fails.  Allocates nothing.
 */
ATTN_API attn_status attn_selftest_exp2(const float* x, float* y_poly, float* y_mufu, int64_t n,
                                        float scale_log2, float m, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_H */
