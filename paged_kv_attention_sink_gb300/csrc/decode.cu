// Decode sink attention (qo_len = 1) over HND pages, with split-KV and an
// in-launch log-sum-exp merge.
//
// Definition: "GPT-OSS on day 0" (Perplexity), section "Sink Attention" -- one
// sink logit per query head in the softmax denominator, online softmax with
// max subtraction, the running state of the first KV part initialised from
// the sink (m = sink, scale d = 1) and the other parts from (-inf, 0).
// Decode is bound by HBM bandwidth ("Hosting Qwen on Blackwell", section
// "Decoder"), so the design goal is to stream each K/V byte exactly once at
// full bandwidth:
//
//  * one CTA = one decode unit (request, KV head, <=16 query heads, KV chunk);
//    the GQA group's query heads share every K/V tile (rows of one m16 MMA);
//  * 4 warps, each with its own TMA pipeline of 16-token blocks: warp w takes
//    blocks w, w+4, ...; lane 0 refills a stage as soon as the warp has read
//    it, so no CTA-wide barrier sits in the streaming loop;
//  * each (page, KV head) block of K or V is one 3-D TMA box loaded with the
//    128-byte swizzle, so ldmatrix reads it without bank conflicts;
//  * S = Q K^T and O += P V are mma.sync m16n8k16 bf16 -> fp32 (tensor cores:
//    at 8-16 flop per KV byte, fp32 FMA would cap below HBM speed); the
//    softmax runs on the S fragments in registers (log2 domain, ex2.approx);
//  * the 4 warps' states are merged through shared memory; a split sequence
//    writes an fp32 partial state, and the last CTA of the group (atomic
//    ticket, no waiting) merges all chunks into out / lse.
#include <cuda.h>

#include "attn_internal.h"
#include "kernels.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

template <int D>
struct DecodeCfg {
    static constexpr int kWarps = kDecodeWarps;
    // Stages per warp.  At D = 64 three (48 KB of pipeline, 4 CTAs per SM)
    // stream faster than four (64 KB, 3 CTAs per SM) with the same bytes in
    // flight per SM: more CTAs absorb the per-unit start-up and the tail.
    static constexpr int kStages = 3;
    static constexpr int kSubTile = kBlockTokens * 128;       // 16 rows x 128 B (64 dims)
    static constexpr int kTileBytes = kBlockTokens * D * 2;   // K or V of one block
    static constexpr int kStageBytes = 2 * kTileBytes;
    static constexpr int kPipeBytes = kWarps * kStages * kStageBytes;
    static constexpr int kPageBytes = (kDecodeMaxChunkPages * 4 + 15) / 16 * 16;
    static constexpr int kBarBytes = kWarps * kStages * 8;
    static constexpr int kStateBytes = kWarps * 48 * 4 + 16;  // per-warp m, l, le + flags
    static constexpr int kSmem = 1024 + kPipeBytes + kPageBytes + kBarBytes + kStateBytes;
    static constexpr int kRowStride = D + 8;                  // floats, combine buffers
    static_assert(kBlockTokens * kRowStride * 4 <= kStages * kStageBytes, "combine fits");
};

struct GraphPlanArgs {
    const int32_t* kv_indptr;       // [batch + 1] page CSR
    const int32_t* last_page_len;   // [batch]
    const int32_t* batch;           // device scalar
    int32_t max_batch, Hq, Hkv, P, n_slices;
    int64_t target_units;
    int64_t cap_blocks;             // 16-token blocks the plan's capacity allows
    int32_t cap_units, cap_groups;
    DecodeUnit* units;
    int32_t* n_units;
    int32_t* queue;                 // [2], then the split-merge counters
    int32_t* err;
};

// Token range [c * nblk / nc, (c + 1) * nblk / nc) blocks, in 32-bit
// arithmetic when the product fits (the common case).
__device__ __forceinline__ int64_t chunk_block(int c, int64_t nblk, int nc) {
    const uint64_t prod = (uint64_t)c * (uint64_t)nblk;
    return prod < 0xFFFFFFFFull ? (int64_t)((uint32_t)prod / (uint32_t)nc) : (int64_t)(prod / (uint64_t)nc);
}

// Graph plans of up to kInPlanMaxBatch requests are planned inside the
// persistent decode grid instead of by decode_graph_plan_kernel: every CTA
// builds the same tables (one request per thread) and derives each unit it
// takes from them, so no planner launch runs before the decode.  The tables
// are indexed by sorted position (longest unit first, ties by request).
constexpr int kInPlanMaxBatch = kDecodeWarps * 32;
struct InPlan {
    int32_t uoff[kInPlanMaxBatch + 1];   // first unit of each sorted request; [n] = unit count
    int32_t nc[kInPlanMaxBatch];         // chunks
    int32_t req[kInPlanMaxBatch];        // request index (query row)
    int32_t base[kInPlanMaxBatch];       // kv_indptr[req]
    int32_t kv[kInPlanMaxBatch];         // kv_len
    int32_t poff[kInPlanMaxBatch];       // first partial slot
    int32_t goff[kInPlanMaxBatch];       // first split group
    int32_t ulen[kInPlanMaxBatch];       // unit length by request (for the ranking)
    int32_t scan[3][kDecodeWarps];
    long long blocks[kDecodeWarps];
    int32_t n, n_groups;
};

// Builds the tables (all threads of the CTA take part; one request per
// thread) and returns the unit count, 0 when the batch is refused.  The rule
// is decode_graph_plan_kernel's: kv lengths from the page CSR, chunk = total
// blocks / target units clamped to 8..512 blocks, each request's chunk count
// and unit length, longest first.  `report`: this CTA sets the error word.
__device__ int plan_in_cta(const GraphPlanArgs& p, InPlan& s, bool report) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int B = *p.batch;
    bool bad = false;
    if (B < 0 || B > p.max_batch) {
        bad = true;
        B = B < 0 ? 0 : p.max_batch;
    }
    int kv = -1, base = 0;
    if (tid < B) {
        base = p.kv_indptr[tid];
        const int64_t np = (int64_t)p.kv_indptr[tid + 1] - base;
        const int32_t lpl = p.last_page_len[tid];
        int64_t len = -1;
        if (np >= 1 && lpl >= 1 && lpl <= p.P) len = (np - 1) * p.P + lpl;
        if (len < 0 || len > INT32_MAX) {
            bad = true;
            len = -1;
        }
        kv = (int)len;
    }
    long long blocks = kv > 0 ? (kv + kBlockTokens - 1) / kBlockTokens : 0;
    for (int o = 16; o > 0; o >>= 1) blocks += __shfl_xor_sync(0xffffffffu, blocks, o);
    if (lane == 0) s.blocks[warp] = blocks;
    bad = __syncthreads_or(bad);
    long long total_blocks = 0;
#pragma unroll
    for (int w = 0; w < kDecodeWarps; ++w) total_blocks += s.blocks[w];
    if (total_blocks > p.cap_blocks) {
        if (report && tid == 0) atomicOr(p.err, ATTN_DEVICE_ERR_PLAN);
        if (tid == 0) s.n_groups = 0;
        __syncthreads();
        return 0;
    }
    total_blocks *= (long long)p.Hkv * p.n_slices;
    const uint32_t chunk = (uint32_t)min((long long)kDecodeMaxChunkBlocks,
                                         max((long long)kDecodeMinChunkBlocks,
                                             (total_blocks + p.target_units - 1) / p.target_units));
    int nc = 0, ulen = 0;
    if (kv >= 0) {
        const uint32_t nblk = ((uint32_t)kv + kBlockTokens - 1) / kBlockTokens;
        const uint32_t n = max(max(1u, (nblk + chunk / 2) / chunk), (nblk + kDecodeMaxChunkBlocks - 1) / kDecodeMaxChunkBlocks);
        nc = (int)n;
        ulen = (int)((nblk + n - 1) / n);
    }
    if (tid < B) s.ulen[tid] = ulen;
    __syncthreads();
    // Sorted position: longer units first, ties by request index (the same
    // order in every CTA).
    if (tid < B) {
        int rank = 0;
        for (int b = 0; b < B; ++b) {
            const int u = s.ulen[b];
            rank += (u > ulen) || (u == ulen && b < tid);
        }
        s.req[rank] = tid;
        s.nc[rank] = nc;
        s.base[rank] = base;
        s.kv[rank] = kv;
    }
    __syncthreads();
    // Exclusive scans over sorted positions: units, partial slots, groups.
    const int per_req = p.Hkv * p.n_slices;
    int v[3] = {0, 0, 0};
    if (tid < B) {
        const int n = s.nc[tid];
        v[0] = n * per_req;
        if (n > 1) {
            v[1] = n * per_req;
            v[2] = per_req;
        }
    }
    int inc[3] = {v[0], v[1], v[2]};
#pragma unroll
    for (int k = 0; k < 3; ++k)
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, inc[k], o);
            if (lane >= o) inc[k] += n;
        }
    if (lane == 31)
#pragma unroll
        for (int k = 0; k < 3; ++k) s.scan[k][warp] = inc[k];
    __syncthreads();
    int tot[3], pre[3];
#pragma unroll
    for (int k = 0; k < 3; ++k) {
        tot[k] = pre[k] = 0;
#pragma unroll
        for (int w = 0; w < kDecodeWarps; ++w) {
            tot[k] += s.scan[k][w];
            if (w < warp) pre[k] += s.scan[k][w];
        }
    }
    if (tid < B) {
        s.uoff[tid] = pre[0] + inc[0] - v[0];
        s.poff[tid] = pre[1] + inc[1] - v[1];
        s.goff[tid] = pre[2] + inc[2] - v[2];
    }
    const bool over = tot[0] > p.cap_units || tot[1] > p.cap_units || tot[2] > p.cap_groups;
    if (tid == 0) {
        s.uoff[B] = tot[0];
        s.n = B;
        s.n_groups = over ? 0 : tot[2];
        if (report && (bad || over)) atomicOr(p.err, ATTN_DEVICE_ERR_PLAN);
    }
    __syncthreads();
    return over ? 0 : tot[0];
}

// Unit `u` of the in-grid plan (the fields decode_graph_plan_kernel writes).
__device__ DecodeUnit unit_of(const InPlan& s, int u, const GraphPlanArgs& p) {
    int lo = 0, hi = s.n - 1;   // last sorted position whose first unit is <= u
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s.uoff[mid] <= u) lo = mid;
        else hi = mid - 1;
    }
    const int k = u - s.uoff[lo], nc = s.nc[lo];
    const int gs = k / nc, c = k - gs * nc;
    const int g = gs / p.n_slices, sl = gs - g * p.n_slices;
    const int G = p.Hq / p.Hkv;
    const int64_t kv = s.kv[lo];
    const int64_t nblk = (kv + kBlockTokens - 1) / kBlockTokens;
    DecodeUnit d;
    d.q_row = s.req[lo];
    d.page_base = s.base[lo];
    d.kv_head = g;
    d.head0 = g * G + sl * kMaxSliceHeads;
    d.n_heads = min(kMaxSliceHeads, G - sl * kMaxSliceHeads);
    d.tok_begin = (int)(chunk_block(c, nblk, nc) * kBlockTokens);
    d.tok_end = (int)min(kv, chunk_block(c + 1, nblk, nc) * kBlockTokens);
    d.chunk = c;
    d.n_chunks = nc;
    d.group = nc > 1 ? s.goff[lo] + gs : -1;
    d.partial0 = nc > 1 ? s.poff[lo] + gs * nc : 0;
    d.reserved = 0;
    return d;
}

struct DecodeArgs {
    const DecodeUnit* units;
    const int32_t* page_table;
    const __nv_bfloat16* q;
    __nv_bfloat16* out;
    float* lse;
    const float* sinks;
    float* part_o;
    float* part_lse;
    int32_t* counters;  // split-merge tickets, one per split group
    int32_t* queue;     // persistent launches: [0] next unit to hand out, [1] CTAs finished
    const int32_t* n_units_dev;   // persistent launches: unit count, written on the device
    int32_t* err;
    int32_t Hq, Hkv, P, num_pages;
    float scale_log2;   // sm_scale * log2(e)
    int32_t in_plan;    // persistent launches: plan inside the grid from `gp`
    GraphPlanArgs gp;
};

__device__ __forceinline__ uint32_t ld_b32(const __nv_bfloat16* p) {
    return *reinterpret_cast<const uint32_t*>(p);
}

__device__ __forceinline__ void store_bf16x4(__nv_bfloat16* dst, float a, float b, float c, float d) {
    uint2 v;
    v.x = ptx::pack_bf16x2(a, b);
    v.y = ptx::pack_bf16x2(c, d);
    *reinterpret_cast<uint2*>(dst) = v;
}

// kPersistent = false: CTA c runs unit c (grid = unit count, host-planned).
// kPersistent = true: a fixed grid takes units from a device queue until the
// device-written unit count is reached (the CUDA-graph path, whose work list
// is built on the device, so neither the grid nor the count is known on the
// host).
template <int D, bool kTwoRows, bool kPersistent>
__global__ void __launch_bounds__(kDecodeWarps * 32)
decode_sink_attn_kernel(const __grid_constant__ CUtensorMap kv_map, const DecodeArgs a) {
    using C = DecodeCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* pipe = smem;
    int32_t* pages_s = reinterpret_cast<int32_t*>(smem + C::kPipeBytes);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kPipeBytes + C::kPageBytes);
    float* ml_s = reinterpret_cast<float*>(smem + C::kPipeBytes + C::kPageBytes + C::kBarBytes);
    int* flag_s = reinterpret_cast<int*>(ml_s + C::kWarps * 48);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int gq = lane >> 2, tq = lane & 3;
    const int P = a.P;
    volatile int* unit_s = flag_s + 1;   // unit handed to this CTA
    volatile int* abort_s = flag_s + 2;
    volatile int* last_s = flag_s + 3;   // persistent: this CTA finished last

    if (lane == 0)
        for (int s = 0; s < C::kStages; ++s) ptx::mbar_init(ptx::smem_u32(&bars[warp * C::kStages + s]), 1);
    if (tid == 0) {
        ptx::prefetch_tmap(&kv_map);
        *abort_s = 0;
    }
    ptx::fence_mbar_init();

    const uint32_t stage0 = ptx::smem_u32(pipe) + warp * C::kStages * C::kStageBytes;
    const uint32_t bar0 = ptx::smem_u32(&bars[warp * C::kStages]);
    const uint64_t policy = ptx::policy_evict_first();
    int gbase = 0;   // stage uses of this warp's ring so far (across units)

    // Behind the planner kernel the persistent grid is launched as its
    // programmatic dependent: its CTAs start (and do the set-up above) while
    // the planner runs, and wait here until the planner's unit list is
    // complete and visible.  Without such a launch the wait returns at once.
    if constexpr (kPersistent) asm volatile("griddepcontrol.wait;" ::: "memory");
    // In-grid plan: its tables sit past the decode's own shared memory.
    InPlan& ip = *reinterpret_cast<InPlan*>(smem + C::kSmem - 1024);
    int n_units = 0;
    if constexpr (kPersistent) {
        if (a.in_plan) {
            n_units = plan_in_cta(a.gp, ip, blockIdx.x == 0);
            if (blockIdx.x == 0) {
                // The unit list and its count, for inspection (attn_graph_plan_read_units);
                // no CTA reads them back.
                for (int u = tid; u < n_units; u += blockDim.x) a.gp.units[u] = unit_of(ip, u, a.gp);
                if (tid == 0) *a.gp.n_units = n_units;
            }
        } else {
            n_units = *a.n_units_dev;
        }
    }
    while (true) {
    int unit = blockIdx.x;
    if constexpr (kPersistent) {
        if (tid == 0) *unit_s = atomicAdd(&a.queue[0], 1);
        __syncthreads();
        unit = *unit_s;
        if (unit >= n_units || *abort_s) break;
    }
    const DecodeUnit u = (kPersistent && a.in_plan) ? unit_of(ip, unit, a.gp) : a.units[unit];
    const int first_page = u.tok_begin / P;
    const int n_pages = (u.tok_end - 1) / P - first_page + 1;
    for (int i = tid; i < n_pages; i += blockDim.x)
        pages_s[i] = a.page_table[u.page_base + first_page + i];
    __syncthreads();

    const int nblk = (u.tok_end - u.tok_begin + kBlockTokens - 1) / kBlockTokens;
    const int n_it = nblk > warp ? (nblk - warp + C::kWarps - 1) / C::kWarps : 0;

    // Lane 0: start the loads of block kb into stage s.
    auto issue = [&](int kb, int s) {
        const int tok = u.tok_begin + kb * kBlockTokens;
        const int page = pages_s[tok / P - first_page];
        const uint32_t bar = bar0 + s * 8;
        if (page < 0 || page >= a.num_pages) {
            atomicOr(a.err, ATTN_DEVICE_ERR_PAGE_ID);
            ptx::mbar_arrive(bar);            // complete the phase without data
            return;
        }
        ptx::mbar_arrive_expect_tx(bar, C::kStageBytes);
        const int off = tok % P;
        const int k_blk = (page * 2) * a.Hkv + u.kv_head;
        const int v_blk = (page * 2 + 1) * a.Hkv + u.kv_head;
        const uint32_t dst = stage0 + s * C::kStageBytes;
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
            ptx::tma_load_3d_hint(dst + c * C::kSubTile, &kv_map, bar, c * 64, off, k_blk, policy);
            ptx::tma_load_3d_hint(dst + C::kTileBytes + c * C::kSubTile, &kv_map, bar, c * 64, off,
                                  v_blk, policy);
        }
    };

    if (lane == 0)
        for (int it = 0; it < C::kStages && it < n_it; ++it) issue(warp + it * C::kWarps, (gbase + it) % C::kStages);

    // Q fragments (A operand, rows = query heads of the slice).
    uint32_t qa[D / 16][4];
    {
        const __nv_bfloat16* q0 = a.q + ((size_t)u.q_row * a.Hq + u.head0 + gq) * D;
        const __nv_bfloat16* q1 = q0 + 8 * D;
        const bool v0 = gq < u.n_heads;
        const bool v1 = kTwoRows && (gq + 8 < u.n_heads);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            qa[kk][0] = v0 ? ld_b32(q0 + 16 * kk + 2 * tq) : 0u;
            qa[kk][2] = v0 ? ld_b32(q0 + 16 * kk + 8 + 2 * tq) : 0u;
            qa[kk][1] = v1 ? ld_b32(q1 + 16 * kk + 2 * tq) : 0u;
            qa[kk][3] = v1 ? ld_b32(q1 + 16 * kk + 8 + 2 * tq) : 0u;
        }
    }

    // Online-softmax state (log2 domain).  l is a per-thread partial sum over
    // this thread's columns of the bf16-rounded P that the PV MMA consumes (it
    // normalises O); e is the same sum of the unrounded P (it gives lse).  The
    // sink's 1 is counted once, on column lane 0.
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f, e0 = 0.f, e1 = 0.f;
    if (warp == 0 && u.chunk == 0 && a.sinks != nullptr) {
        if (gq < u.n_heads) {
            m0 = a.sinks[u.head0 + gq] * kLog2e;
            l0 = e0 = tq == 0 ? 1.f : 0.f;
        }
        if (kTwoRows && gq + 8 < u.n_heads) {
            m1 = a.sinks[u.head0 + gq + 8] * kLog2e;
            l1 = e1 = tq == 0 ? 1.f : 0.f;
        }
    }
    float o[D / 8][4];
#pragma unroll
    for (int j = 0; j < D / 8; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;

    int it = 0;
    bool timed_out = false;
    for (; it < n_it; ++it) {
        const int s = (gbase + it) % C::kStages;
        if (!ptx::mbar_wait(bar0 + s * 8, ((gbase + it) / C::kStages) & 1)) { timed_out = true; break; }
        const int kb = warp + it * C::kWarps;
        const int valid = min(kBlockTokens, u.tok_end - (u.tok_begin + kb * kBlockTokens));
        const uint32_t kt = stage0 + s * C::kStageBytes;
        const uint32_t vt = kt + C::kTileBytes;
        if (valid < kBlockTokens) {
            // Rows past the end of the sequence may hold anything (even NaN):
            // zero those V rows so that P = 0 there contributes exactly 0.
            uint8_t* vrows = pipe + (warp * C::kStages + s) * C::kStageBytes + C::kTileBytes;
            const int per_sub = (kBlockTokens - valid) * 8;
            for (int idx = lane; idx < per_sub * (D / 64); idx += 32) {
                const int sub = idx / per_sub, rem = idx % per_sub;
                *reinterpret_cast<uint4*>(vrows + sub * C::kSubTile + (valid + rem / 8) * 128 +
                                          (rem % 8) * 16) = make_uint4(0, 0, 0, 0);
            }
            __syncwarp();
        }

        // S[head][token] for the block's 16 tokens (two n8 tiles).
        float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            const int mi = lane >> 3;
            const int row = (mi >> 1) * 8 + (lane & 7);
            const int ch = 2 * kk + (mi & 1);
            const uint32_t addr = kt + (ch >> 3) * C::kSubTile + row * 128 + (((ch & 7) ^ (lane & 7)) << 4);
            uint32_t b0, b1, b2, b3;
            ptx::ldmatrix_x4(addr, b0, b1, b2, b3);
            ptx::mma_bf16_16816(sc[0], qa[kk], b0, b1);
            ptx::mma_bf16_16816(sc[1], qa[kk], b2, b3);
        }

        // Online softmax over the block (rows gq and gq + 8).
        float x[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int tok = nt * 8 + 2 * tq + (e & 1);
                x[nt][e] = tok < valid ? sc[nt][e] * a.scale_log2 : -INFINITY;
            }
        float p[2][4];
        float alpha0, alpha1 = 1.f;
        {
            float mx = fmaxf(fmaxf(x[0][0], x[0][1]), fmaxf(x[1][0], x[1][1]));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            const float mn = fmaxf(m0, mx);
            const float base = mn == -INFINITY ? 0.f : mn;
            alpha0 = ptx::ex2(m0 - base);
            p[0][0] = ptx::ex2(x[0][0] - base);
            p[0][1] = ptx::ex2(x[0][1] - base);
            p[1][0] = ptx::ex2(x[1][0] - base);
            p[1][1] = ptx::ex2(x[1][1] - base);
            m0 = mn;
#pragma unroll
            for (int j = 0; j < D / 8; ++j) { o[j][0] *= alpha0; o[j][1] *= alpha0; }
        }
        if (kTwoRows) {
            float mx = fmaxf(fmaxf(x[0][2], x[0][3]), fmaxf(x[1][2], x[1][3]));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            const float mn = fmaxf(m1, mx);
            const float base = mn == -INFINITY ? 0.f : mn;
            alpha1 = ptx::ex2(m1 - base);
            p[0][2] = ptx::ex2(x[0][2] - base);
            p[0][3] = ptx::ex2(x[0][3] - base);
            p[1][2] = ptx::ex2(x[1][2] - base);
            p[1][3] = ptx::ex2(x[1][3] - base);
            m1 = mn;
#pragma unroll
            for (int j = 0; j < D / 8; ++j) { o[j][2] *= alpha1; o[j][3] *= alpha1; }
        } else {
            p[0][2] = p[0][3] = p[1][2] = p[1][3] = 0.f;
        }
        uint32_t pa[4];
        pa[0] = ptx::pack_bf16x2(p[0][0], p[0][1]);
        pa[1] = ptx::pack_bf16x2(p[0][2], p[0][3]);
        pa[2] = ptx::pack_bf16x2(p[1][0], p[1][1]);
        pa[3] = ptx::pack_bf16x2(p[1][2], p[1][3]);
        {
            // Row sums of the same bf16-rounded P that the PV MMA uses.
            const float2 a0 = ptx::unpack_bf16x2(pa[0]), a2 = ptx::unpack_bf16x2(pa[2]);
            l0 = l0 * alpha0 + (a0.x + a0.y) + (a2.x + a2.y);
            e0 = e0 * alpha0 + (p[0][0] + p[0][1]) + (p[1][0] + p[1][1]);
            if (kTwoRows) {
                const float2 a1 = ptx::unpack_bf16x2(pa[1]), a3 = ptx::unpack_bf16x2(pa[3]);
                l1 = l1 * alpha1 + (a1.x + a1.y) + (a3.x + a3.y);
                e1 = e1 * alpha1 + (p[0][2] + p[0][3]) + (p[1][2] + p[1][3]);
            }
        }

        // O[head][dim] += P V (V read transposed by ldmatrix.trans).
#pragma unroll
        for (int j2 = 0; j2 < D / 16; ++j2) {
            const int mi = lane >> 3;
            const int row = (mi & 1) * 8 + (lane & 7);
            const int ch = 2 * j2 + (mi >> 1);
            const uint32_t addr = vt + (ch >> 3) * C::kSubTile + row * 128 + (((ch & 7) ^ (lane & 7)) << 4);
            uint32_t v0, v1, v2, v3;
            ptx::ldmatrix_x4_trans(addr, v0, v1, v2, v3);
            ptx::mma_bf16_16816(o[2 * j2], pa, v0, v1);
            ptx::mma_bf16_16816(o[2 * j2 + 1], pa, v2, v3);
        }

        __syncwarp();
        const int kb_next = kb + C::kStages * C::kWarps;
        if (lane == 0 && kb_next < nblk) {
            ptx::fence_proxy_async_smem();   // generic reads/writes of the stage before TMA rewrites it
            issue(kb_next, s);
        }
    }
    if (timed_out) {
        if (lane == 0) {
            atomicOr(a.err, ATTN_DEVICE_ERR_TIMEOUT);
            *abort_s = 1;
        }
        for (int j = it; j < n_it && j < it + C::kStages; ++j)   // drain loads still in flight
            ptx::mbar_wait(bar0 + ((gbase + j) % C::kStages) * 8, ((gbase + j) / C::kStages) & 1);
    }
    gbase += n_it;

    // Row sums over the quad, then this warp's state into its own stage area.
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    e0 += __shfl_xor_sync(0xffffffffu, e0, 1);
    e0 += __shfl_xor_sync(0xffffffffu, e0, 2);
    e1 += __shfl_xor_sync(0xffffffffu, e1, 1);
    e1 += __shfl_xor_sync(0xffffffffu, e1, 2);
    float* cs = reinterpret_cast<float*>(pipe + warp * C::kStages * C::kStageBytes);
#pragma unroll
    for (int j = 0; j < D / 8; ++j) {
        const int d = 8 * j + 2 * tq;
        *reinterpret_cast<float2*>(&cs[gq * C::kRowStride + d]) = make_float2(o[j][0], o[j][1]);
        *reinterpret_cast<float2*>(&cs[(gq + 8) * C::kRowStride + d]) = make_float2(o[j][2], o[j][3]);
    }
    if (tq == 0) {
        float* st = ml_s + warp * 48;   // [m | l | e] x 16 rows
        st[gq] = m0;
        st[16 + gq] = l0;
        st[32 + gq] = e0;
        st[gq + 8] = kTwoRows ? m1 : -INFINITY;
        st[16 + gq + 8] = kTwoRows ? l1 : 0.f;
        st[32 + gq + 8] = kTwoRows ? e1 : 0.f;
    }
    __syncthreads();

    // Merge the 4 warps: rows < n_heads, 4 dims per item.
    const int items = u.n_heads * (D / 4);
    for (int idx = tid; idx < items; idx += blockDim.x) {
        const int r = idx / (D / 4), d = (idx % (D / 4)) * 4;
        float ms = -INFINITY;
#pragma unroll
        for (int w = 0; w < C::kWarps; ++w) ms = fmaxf(ms, ml_s[w * 48 + r]);
        float L = 0.f, E = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w = 0; w < C::kWarps; ++w) {
            const float mw = ml_s[w * 48 + r];
            const float f = (mw == -INFINITY) ? 0.f : ptx::ex2(mw - ms);
            L += f * ml_s[w * 48 + 16 + r];
            E += f * ml_s[w * 48 + 32 + r];
            const float4 ow = *reinterpret_cast<const float4*>(
                reinterpret_cast<const float*>(pipe + w * C::kStages * C::kStageBytes) + r * C::kRowStride + d);
            acc.x += f * ow.x; acc.y += f * ow.y; acc.z += f * ow.z; acc.w += f * ow.w;
        }
        const float inv = L > 0.f ? 1.f / L : 0.f;
        const float lse2 = E > 0.f ? ms + log2f(E) : -INFINITY;
        if (u.n_chunks == 1) {
            store_bf16x4(a.out + ((size_t)u.q_row * a.Hq + u.head0 + r) * D + d, acc.x * inv,
                         acc.y * inv, acc.z * inv, acc.w * inv);
            if (d == 0 && a.lse) a.lse[(size_t)u.q_row * a.Hq + u.head0 + r] = lse2 * kLn2;
        } else {
            const size_t slot = (size_t)(u.partial0 + u.chunk) * kMaxSliceHeads + r;
            *reinterpret_cast<float4*>(a.part_o + slot * D + d) =
                make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
            if (d == 0) a.part_lse[slot] = lse2;
        }
    }
    if (u.n_chunks > 1) {
    // Split sequence: the last chunk to finish merges all chunks (no waiting).
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        const int prev = atomicAdd(&a.counters[u.group], 1);
        *flag_s = (prev == u.n_chunks - 1);
    }
    __syncthreads();
    if (*flag_s) {
    __threadfence();
    // One (head, 4 dims) item per thread.  Chunks are read in batches of
    // kMergeBatch with every load of a batch independent (so a batch costs
    // about one L2 round trip, not one per chunk), and merged online: the
    // running max only moves between batches.
    constexpr int kMergeBatch = 8;
    for (int idx = tid; idx < items; idx += blockDim.x) {
        const int r = idx / (D / 4), d = (idx % (D / 4)) * 4;
        float M = -INFINITY, W = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int c0 = 0; c0 < u.n_chunks; c0 += kMergeBatch) {
            float lc[kMergeBatch];
            float4 oc[kMergeBatch];
#pragma unroll
            for (int k = 0; k < kMergeBatch; ++k) {
                const int c = c0 + k;
                const size_t slot = (size_t)(u.partial0 + c) * kMaxSliceHeads + r;
                lc[k] = c < u.n_chunks ? __ldcg(a.part_lse + slot) : -INFINITY;
                oc[k] = c < u.n_chunks ? __ldcg(reinterpret_cast<const float4*>(a.part_o + slot * D + d))
                                       : make_float4(0.f, 0.f, 0.f, 0.f);
            }
            float mb = M;
#pragma unroll
            for (int k = 0; k < kMergeBatch; ++k) mb = fmaxf(mb, lc[k]);
            if (mb == -INFINITY) continue;   // nothing visible so far
            const float sc = M == -INFINITY ? 0.f : ptx::ex2(M - mb);
            W *= sc;
            acc.x *= sc; acc.y *= sc; acc.z *= sc; acc.w *= sc;
#pragma unroll
            for (int k = 0; k < kMergeBatch; ++k) {
                const float w = lc[k] == -INFINITY ? 0.f : ptx::ex2(lc[k] - mb);
                W += w;
                acc.x += w * oc[k].x; acc.y += w * oc[k].y; acc.z += w * oc[k].z; acc.w += w * oc[k].w;
            }
            M = mb;
        }
        const float inv = W > 0.f ? 1.f / W : 0.f;
        store_bf16x4(a.out + ((size_t)u.q_row * a.Hq + u.head0 + r) * D + d, acc.x * inv,
                     acc.y * inv, acc.z * inv, acc.w * inv);
        if (d == 0 && a.lse)
            a.lse[(size_t)u.q_row * a.Hq + u.head0 + r] = (W > 0.f ? M + log2f(W) : -INFINITY) * kLn2;
    }
    if (tid == 0) a.counters[u.group] = 0;   // ready for the next launch
    }
    }
    if constexpr (!kPersistent) break;
    __syncthreads();   // shared memory is reused by the next unit
    }

    // The last CTA to finish resets the queue for the next launch (and, with
    // the in-grid plan, clears this launch's split counters: after a launch
    // that ran to the end they are zero already, after one that gave up early
    // they may not be).
    if constexpr (kPersistent) {
        if (tid == 0) {
            __threadfence();
            *last_s = atomicAdd(&a.queue[1], 1) == (int)gridDim.x - 1;
        }
        __syncthreads();
        if (*last_s) {
            if (a.in_plan)
                for (int g = tid; g < ip.n_groups; g += blockDim.x) a.counters[g] = 0;
            if (tid == 0) {
                atomicExch(&a.queue[0], 0);
                atomicExch(&a.queue[1], 0);
            }
        }
    }
}

// ------------------------------------------------------------ device planner
// The CUDA-graph decode path plans on the device: the same split rule as the
// host planner, from request metadata that lives in device memory, so that a
// captured graph replays with new lengths and batch sizes (decode requests
// only: request b is query row b).  One CTA: each thread owns requests
// tid + k * kPlanThreads while it measures and sorts them, and a contiguous
// range of sorted positions while it scans the unit counts.
constexpr int kPlanThreads = 1024;


// Exclusive block-wide scan of three counters (kPlanThreads threads).
__device__ void block_scan3(int (&v)[3], int (&total)[3], int* sh /* [3][32] */) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int inc[3] = {v[0], v[1], v[2]};
#pragma unroll
    for (int k = 0; k < 3; ++k)
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, inc[k], o);
            if (lane >= o) inc[k] += n;
        }
    if (lane == 31)
        for (int k = 0; k < 3; ++k) sh[k * 32 + warp] = inc[k];
    __syncthreads();
    if (warp == 0)
        for (int k = 0; k < 3; ++k) {
            int w = sh[k * 32 + lane];
            for (int o = 1; o < 32; o <<= 1) {
                const int n = __shfl_up_sync(0xffffffffu, w, o);
                if (lane >= o) w += n;
            }
            sh[k * 32 + lane] = w;   // inclusive over warps
        }
    __syncthreads();
    for (int k = 0; k < 3; ++k) {
        total[k] = sh[k * 32 + 31];
        v[k] = inc[k] - v[k] + (warp > 0 ? sh[k * 32 + warp - 1] : 0);
    }
    __syncthreads();
}

// Dynamic shared memory of the planner: 7 int32 per request slot (page base
// and kv_len by request; request, chunk count and the exclusive offsets of
// units, partial slots and groups by sorted position).
inline size_t plan_smem_bytes(int max_batch) { return (size_t)max_batch * 7 * sizeof(int); }

// Requests one planner thread owns (request tid + k * kPlanThreads); their
// lengths, chunk counts and unit lengths stay in registers.
constexpr int kPlanPerThread = (kGraphMaxBatch + kPlanThreads - 1) / kPlanThreads;
static_assert(kPlanPerThread * kPlanThreads >= kGraphMaxBatch, "planner request ownership");


__global__ void __launch_bounds__(kPlanThreads) decode_graph_plan_kernel(const GraphPlanArgs p) {
    extern __shared__ int plan_smem[];
    constexpr int kLenBuckets = kDecodeMaxChunkBlocks + 1;   // unit length 0 (malformed) .. 512 blocks
    __shared__ int s_hist[kLenBuckets];
    __shared__ long long s_blocks[32];
    __shared__ int s_scan[3 * 32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int* s_base = plan_smem;                 // [max_batch] kv_indptr[b]
    int* s_kv = s_base + p.max_batch;        // [max_batch] kv_len, -1 malformed
    int* s_order = s_kv + p.max_batch;       // [max_batch] request at sorted position i
    int* s_nc = s_order + p.max_batch;       // [max_batch] chunks (sorted order)
    int* s_uoff = s_nc + p.max_batch;        // [max_batch] exclusive offsets (sorted order)
    int* s_poff = s_uoff + p.max_batch;
    int* s_goff = s_poff + p.max_batch;

    // Let the persistent decode grid launch now: its CTAs set up and then wait
    // (griddepcontrol.wait) for this grid to finish.
    asm volatile("griddepcontrol.launch_dependents;");
    int B = *p.batch;
    if (B < 0 || B > p.max_batch) {
        if (tid == 0) atomicOr(p.err, ATTN_DEVICE_ERR_PLAN);
        B = B < 0 ? 0 : p.max_batch;
    }
    for (int k = tid; k < kLenBuckets; k += kPlanThreads) s_hist[k] = 0;

    // Pass 1: kv lengths of the owned requests, and all 16-token blocks ->
    // chunk size (two waves of CTAs).  kv_len fits 32 bits (checked), so
    // block counts (< 2^27) do too.
    int kv[kPlanPerThread], nc[kPlanPerThread], ulen[kPlanPerThread];
    long long blocks = 0;
#pragma unroll
    for (int k = 0; k < kPlanPerThread; ++k) {
        const int b = tid + k * kPlanThreads;
        kv[k] = -1;
        if (b >= B) continue;
        const int32_t base = p.kv_indptr[b];
        const int64_t np = (int64_t)p.kv_indptr[b + 1] - base;
        const int32_t lpl = p.last_page_len[b];
        int64_t len = -1;
        if (np >= 1 && lpl >= 1 && lpl <= p.P) len = (np - 1) * p.P + lpl;
        if (len < 0 || len > INT32_MAX) {
            atomicOr(p.err, ATTN_DEVICE_ERR_PLAN);
            len = -1;
        }
        kv[k] = (int)len;
        s_base[b] = base;
        s_kv[b] = kv[k];
        if (len > 0) blocks += (len + kBlockTokens - 1) / kBlockTokens;
    }
    for (int o = 16; o > 0; o >>= 1) blocks += __shfl_xor_sync(0xffffffffu, blocks, o);
    if (lane == 0) s_blocks[warp] = blocks;
    __syncthreads();
    long long total_blocks = 0;
    for (int w = 0; w < kPlanThreads / 32; ++w) total_blocks += s_blocks[w];
    if (total_blocks > p.cap_blocks) {
        // More KV than the plan was sized for: the unit bound below (and the
        // 32-bit counts that rely on it) would not hold.  Same value in every
        // thread, so the whole block leaves here.
        if (tid == 0) {
            atomicOr(p.err, ATTN_DEVICE_ERR_PLAN);
            *p.n_units = 0;
            p.queue[0] = p.queue[1] = 0;
        }
        return;
    }
    total_blocks *= (long long)p.Hkv * p.n_slices;
    const uint32_t chunk = (uint32_t)min((long long)kDecodeMaxChunkBlocks,
                                         max((long long)kDecodeMinChunkBlocks,
                                             (total_blocks + p.target_units - 1) / p.target_units));

    // Pass 2: order the requests by unit length (blocks in the request's
    // longest chunk), longest first, as the host planner orders its units: a
    // counting sort over the 513 possible lengths.
#pragma unroll
    for (int k = 0; k < kPlanPerThread; ++k) {
        nc[k] = 0;
        ulen[k] = 0;
        if (kv[k] >= 0) {
            const uint32_t nblk = ((uint32_t)kv[k] + kBlockTokens - 1) / kBlockTokens;
            const uint32_t n = max(max(1u, (nblk + chunk / 2) / chunk),
                                   (nblk + kDecodeMaxChunkBlocks - 1) / kDecodeMaxChunkBlocks);
            nc[k] = (int)n;
            ulen[k] = (int)((nblk + n - 1) / n);
        }
        if (tid + k * kPlanThreads < B) atomicAdd(&s_hist[kDecodeMaxChunkBlocks - ulen[k]], 1);
    }
    __syncthreads();
    if (warp == 0) {   // exclusive scan of the histogram, 17 buckets per lane
        constexpr int kPer = (kLenBuckets + 31) / 32;
        int local[kPer], sum = 0;
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            const int idx = lane * kPer + k;
            local[k] = idx < kLenBuckets ? s_hist[idx] : 0;
            sum += local[k];
        }
        int inc = sum;
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += n;
        }
        int run = inc - sum;
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            const int idx = lane * kPer + k;
            if (idx < kLenBuckets) s_hist[idx] = run;
            run += local[k];
        }
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < kPlanPerThread; ++k) {
        const int b = tid + k * kPlanThreads;
        if (b >= B) continue;
        const int pos = atomicAdd(&s_hist[kDecodeMaxChunkBlocks - ulen[k]], 1);
        s_order[pos] = b;
        s_nc[pos] = nc[k];
    }
    __syncthreads();

    // Pass 3: units, partial slots and groups in sorted order, scanned (each
    // thread a contiguous range of sorted positions).
    const int per_req = p.Hkv * p.n_slices;
    const int per = (B + kPlanThreads - 1) / kPlanThreads;
    const int i0 = min(B, tid * per), i1 = min(B, i0 + per);
    int v[3] = {0, 0, 0}, tot[3];
    for (int i = i0; i < i1; ++i) {
        const int nc = s_nc[i];
        v[0] += nc * per_req;
        if (nc > 1) {
            v[1] += nc * per_req;
            v[2] += per_req;
        }
    }
    block_scan3(v, tot, s_scan);
    if (tot[0] > p.cap_units || tot[1] > p.cap_units || tot[2] > p.cap_groups) {
        if (tid == 0) {
            atomicOr(p.err, ATTN_DEVICE_ERR_PLAN);
            *p.n_units = 0;
            p.queue[0] = p.queue[1] = 0;
        }
        return;
    }
    for (int i = i0; i < i1; ++i) {
        s_uoff[i] = v[0];
        s_poff[i] = v[1];
        s_goff[i] = v[2];
        const int nc = s_nc[i];
        v[0] += nc * per_req;
        if (nc > 1) {
            v[1] += nc * per_req;
            v[2] += per_req;
        }
    }
    __syncthreads();

    // Pass 4: one warp per sorted request, its lanes over the request's units
    // (head slice major, chunk minor; chunk 0 of a group carries the sink);
    // each unit is written as three 16-byte stores.
    const int G = p.Hq / p.Hkv;
    for (int i = warp; i < B; i += kPlanThreads / 32) {
        const int nc = s_nc[i];
        if (nc == 0) continue;
        const int b = s_order[i];
        const int64_t kv = s_kv[b];
        const int64_t nblk = (kv + kBlockTokens - 1) / kBlockTokens;
        const int base = s_base[b], uoff = s_uoff[i], goff = s_goff[i], poff = s_poff[i];
        for (int k = lane; k < nc * per_req; k += 32) {
            const int gs = k / nc, c = k - gs * nc;
            const int g = gs / p.n_slices, sl = gs - g * p.n_slices;
            const int tok0 = (int)(chunk_block(c, nblk, nc) * kBlockTokens);
            const int tok1 = (int)min(kv, chunk_block(c + 1, nblk, nc) * kBlockTokens);
            int4* dst = reinterpret_cast<int4*>(p.units + uoff + k);
            dst[0] = make_int4(b, base, g, g * G + sl * kMaxSliceHeads);
            dst[1] = make_int4(min(kMaxSliceHeads, G - sl * kMaxSliceHeads), tok0, tok1, c);
            dst[2] = make_int4(nc, nc > 1 ? goff + gs : -1, nc > 1 ? poff + gs * nc : 0, 0);
        }
    }
    for (int k = tid; k < tot[2]; k += kPlanThreads) p.queue[2 + k] = 0;
    if (tid == 0) {
        *p.n_units = tot[0];
        p.queue[0] = p.queue[1] = 0;
    }
}

template <int D, bool kTwoRows, bool kPersistent>
cudaError_t launch(const CUtensorMap& map, const DecodeArgs& args, int grid, cudaStream_t stream) {
    using C = DecodeCfg<D>;
    auto kernel = decode_sink_attn_kernel<D, kTwoRows, kPersistent>;
    // The persistent form also holds the in-grid plan's tables.
    constexpr int smem = C::kSmem + (kPersistent ? (int)sizeof(InPlan) : 0);
    static std::atomic<bool> configured[kMaxDevices];
    cudaError_t e = once_per_device(configured, [&] {
        return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    });
    if (e != cudaSuccess) return e;
    if constexpr (kPersistent) {
        // Behind the device planner: a programmatic dependent of it (see
        // griddepcontrol in both kernels).
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(grid);
        cfg.blockDim = dim3(C::kWarps * 32);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = args.in_plan ? 0 : 1;
        return cudaLaunchKernelEx(&cfg, kernel, map, args);
    }
    kernel<<<grid, C::kWarps * 32, C::kSmem, stream>>>(map, args);
    return cudaGetLastError();
}

template <bool kPersistent>
attn_status dispatch(const attn_plan_s* plan, const CUtensorMap& map, const DecodeArgs& a, int grid,
                     cudaStream_t stream) {
    const bool two_rows = plan->Hq / plan->Hkv > 8;
    cudaError_t e;
    if (plan->D == 64)
        e = two_rows ? launch<64, true, kPersistent>(map, a, grid, stream)
                     : launch<64, false, kPersistent>(map, a, grid, stream);
    else
        e = two_rows ? launch<128, true, kPersistent>(map, a, grid, stream)
                     : launch<128, false, kPersistent>(map, a, grid, stream);
    return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

// Kernel arguments with the plan's device regions taken from `base` (the bound
// workspace, or the caller's scratch laid out the same way).
DecodeArgs make_args(const attn_plan_s* plan, unsigned char* base, const void* q, const float* sinks, void* out,
                     float* lse) {
    DecodeArgs a;
    a.units = reinterpret_cast<const DecodeUnit*>(base + plan->layout.units);
    a.page_table = plan->page_table;
    a.q = static_cast<const __nv_bfloat16*>(q);
    a.out = static_cast<__nv_bfloat16*>(out);
    a.lse = lse;
    a.sinks = sinks;
    a.part_o = reinterpret_cast<float*>(base + plan->layout.part_o);
    a.part_lse = reinterpret_cast<float*>(base + plan->layout.part_lse);
    a.counters = reinterpret_cast<int32_t*>(base + plan->layout.counters);
    a.queue = nullptr;
    a.n_units_dev = nullptr;
    a.err = reinterpret_cast<int32_t*>(base + plan->layout.err);
    a.Hq = plan->Hq;
    a.Hkv = plan->Hkv;
    a.P = plan->P;
    a.num_pages = plan->num_pages;
    a.scale_log2 = plan->sm_scale * kLog2e;
    a.in_plan = 0;
    a.gp = GraphPlanArgs{};
    return a;
}

}  // namespace

constexpr int kSmemPerSm = 233472;   // 228 KB; 1 KB of it is reserved per CTA
// The persistent form's in-grid plan tables must not cost a CTA per SM.
static_assert(kSmemPerSm / (DecodeCfg<64>::kSmem + (int)sizeof(InPlan) + 1024) ==
                  kSmemPerSm / (DecodeCfg<64>::kSmem + 1024), "in-grid plan and CTAs per SM (D = 64)");
static_assert(kSmemPerSm / (DecodeCfg<128>::kSmem + (int)sizeof(InPlan) + 1024) ==
                  kSmemPerSm / (DecodeCfg<128>::kSmem + 1024), "in-grid plan and CTAs per SM (D = 128)");

int decode_ctas_per_sm(int head_dim) {
    const int per_cta = (head_dim == 64 ? DecodeCfg<64>::kSmem : DecodeCfg<128>::kSmem) + 1024;
    return kSmemPerSm / per_cta;
}

attn_status launch_decode(attn_plan_s* plan, const void* q, const void* kv_map, const float* sinks,
                          void* out, float* lse, cudaStream_t stream) {
    if (plan->units.empty()) return ATTN_OK;
    const DecodeArgs a = make_args(plan, plan->ws, q, sinks, out, lse);
    return dispatch<false>(plan, *static_cast<const CUtensorMap*>(kv_map), a, (int)plan->units.size(), stream);
}

attn_status launch_decode_scratch(attn_plan_s* plan, unsigned char* scratch, const void* q,
                                  const void* kv_map, const float* sinks, void* out, float* lse,
                                  cudaStream_t stream) {
    if (plan->units.empty()) return ATTN_OK;
    const DecodeArgs a = make_args(plan, scratch, q, sinks, out, lse);
    return dispatch<false>(plan, *static_cast<const CUtensorMap*>(kv_map), a, (int)plan->units.size(), stream);
}

attn_status launch_decode_graph(attn_plan_s* plan, const int32_t* kv_indptr, const int32_t* last_page_len,
                                const int32_t* batch, const void* q, const void* kv_map, const float* sinks,
                                void* out, float* lse, cudaStream_t stream) {
    GraphPlanArgs gp;
    gp.kv_indptr = kv_indptr;
    gp.last_page_len = last_page_len;
    gp.batch = batch;
    gp.max_batch = plan->batch;
    gp.Hq = plan->Hq;
    gp.Hkv = plan->Hkv;
    gp.P = plan->P;
    gp.n_slices = (plan->Hq / plan->Hkv + kMaxSliceHeads - 1) / kMaxSliceHeads;
    gp.target_units = 2LL * plan->num_sms * decode_ctas_per_sm(plan->D);
    gp.cap_blocks = plan->graph_kv_blocks;
    gp.cap_units = plan->n_partials;   // graph plans size units and partial slots alike
    gp.cap_groups = plan->n_groups;
    gp.units = reinterpret_cast<DecodeUnit*>(plan->ws + plan->layout.units);
    gp.n_units = reinterpret_cast<int32_t*>(plan->ws + plan->layout.n_units);
    gp.queue = reinterpret_cast<int32_t*>(plan->ws + plan->layout.counters);
    gp.err = reinterpret_cast<int32_t*>(plan->ws + plan->layout.err);
    DecodeArgs a = make_args(plan, plan->ws, q, sinks, out, lse);
    a.queue = gp.queue;
    a.counters = gp.queue + 2;
    a.n_units_dev = gp.n_units;
    const int grid = plan->num_sms * decode_ctas_per_sm(plan->D);
    if (plan->batch <= kInPlanMaxBatch) {
        // Small plans: every CTA of the persistent grid plans for itself.
        a.in_plan = 1;
        a.gp = gp;
        return dispatch<true>(plan, *static_cast<const CUtensorMap*>(kv_map), a, grid, stream);
    }
    // The shared-memory limit is raised once per device to what the largest
    // graph plan needs; each launch asks only for its own plan's share.
    static std::atomic<bool> configured[kMaxDevices];
    if (once_per_device(configured, [] {
            return cudaFuncSetAttribute(decode_graph_plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)plan_smem_bytes(kGraphMaxBatch));
        }) != cudaSuccess)
        return ATTN_ERR_CUDA;
    decode_graph_plan_kernel<<<1, kPlanThreads, plan_smem_bytes(plan->batch), stream>>>(gp);
    if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;
    return dispatch<true>(plan, *static_cast<const CUtensorMap*>(kv_map), a, grid, stream);
}

}  // namespace attn
