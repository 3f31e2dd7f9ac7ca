// Prefill sink attention (qo_len > 1) on the 5th-generation tensor cores.
//
// Definition: "GPT-OSS on day 0" (Perplexity), section "Sink Attention": one
// sink logit per query head in the softmax denominator, softmax computed
// online with max subtraction, the running max initialised to the sink (scale
// 1).  Prefill is compute-bound ("Disaggregated prefill and decode", section
// "Prefill vs decode performance"), so QK^T and PV run as tcgen05.mma with
// fp32 accumulators in tensor memory:
//
//  * one CTA = 128 query rows of one request x two query heads of one GQA
//    group; both heads share every K/V tile (each tile feeds four MMAs);
//  * warp 0 (one lane) streams K/V tiles of 128 keys with TMA, one box per
//    HND page, 128-byte swizzled, into a 3-stage ring; rows past the end of
//    the sequence are zeroed in V before the MMA may read them;
//  * warp 1 (one lane) issues the MMAs: S_h = Q_h K^T (both operands K-major
//    in shared memory) and O_h += P_h V (P read straight from tensor memory,
//    V as an MN-major shared-memory operand);
//  * warps 4-7 and 8-11 run the softmax of head 0 and head 1: one thread per
//    row (= TMEM lane) loads its 128 scores, applies the causal / length mask,
//    updates the running max lazily (O is rescaled only when the max grew by
//    more than 2^8), writes P as bf16 back over S in tensor memory, and at
//    the end normalises O and stores out and lse.
// Every wait is bounded; a timeout sets the device error word.
#include <cuda.h>

#include "attn_internal.h"
#include "kernels.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;   // log2 units: P stays <= 2^8 between rescales

template <int D>
struct PrefillCfg {
    static constexpr int kThreads = 384;                 // 3 warpgroups
    // Register split (setmaxnreg): the launch gives every thread kRegsLaunch;
    // warpgroup 0 (producer, MMA) drops to kRegsCtrl and the two softmax
    // warpgroups grow to kRegsSoftmax.  128 * kRegsCtrl + 256 * kRegsSoftmax
    // must not exceed 384 * kRegsLaunch, or setmaxnreg.inc would wait forever.
    static constexpr int kRegsLaunch = 168;
    static constexpr int kRegsCtrl = 56;
    static constexpr int kRegsSoftmax = 224;
    static_assert(128 * kRegsCtrl + 256 * kRegsSoftmax <= kThreads * kRegsLaunch, "register split");
    static constexpr int kStagesK = (D == 64) ? 3 : 2;
    static constexpr int kStagesV = (D == 64) ? 3 : 2;
    static constexpr int kAtom = 128 * 128;              // 128 rows x 64 bf16, swizzled
    static constexpr int kTile = kAtom * (D / 64);       // Q, K or V tile of 128 rows
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = 2 * kTile;
    static constexpr int kOffV = kOffK + kStagesK * kTile;
    static constexpr int kOffBar = kOffV + kStagesV * kTile;
    static constexpr int kNumBars = 1 + 2 * kStagesK + 2 * kStagesV + 6 + 2;
    static constexpr int kSmem = 1024 + kOffBar + kNumBars * 8 + 16;
    static constexpr uint32_t kTmemCols = 512;           // S0 S1 (128 each), O0 O1 (D each)
};

struct PrefillArgs {
    const PrefillItem* items;
    const int32_t* page_table;
    __nv_bfloat16* out;
    float* lse;
    const float* sinks;
    int32_t* err;
    int32_t Hq, Hkv, P, num_pages, causal;
    float scale_log2;
};

struct Bars {
    uint32_t q_full, k_full, k_empty, v_full, v_empty, s_full, p_full, o_done, v_aux, drain;
};

template <int D>
__global__ void __launch_bounds__(PrefillCfg<D>::kThreads, 1)
prefill_sink_attn_kernel(const __grid_constant__ CUtensorMap q_map,
                         const __grid_constant__ CUtensorMap kv_map, const PrefillArgs a) {
    using C = PrefillCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = ptx::smem_u32(smem);
    uint64_t* bar_mem = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_mem + C::kNumBars);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    Bars B;
    B.q_full = ptx::smem_u32(bar_mem);
    B.k_full = B.q_full + 8;
    B.k_empty = B.k_full + 8 * C::kStagesK;
    B.v_full = B.k_empty + 8 * C::kStagesK;
    B.v_empty = B.v_full + 8 * C::kStagesV;
    B.s_full = B.v_empty + 8 * C::kStagesV;
    B.p_full = B.s_full + 16;
    B.o_done = B.p_full + 16;
    B.v_aux = B.o_done + 16;
    B.drain = B.v_aux + 8;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const PrefillItem it = a.items[blockIdx.x];
    const int n_tiles = it.n_kv_tiles;
    const int nh = it.n_heads;

    if (tid == 0) {
        ptx::mbar_init(B.q_full, 1);
        for (int s = 0; s < C::kStagesK; ++s) {
            ptx::mbar_init(B.k_full + 8 * s, 1);
            ptx::mbar_init(B.k_empty + 8 * s, 1);
        }
        for (int s = 0; s < C::kStagesV; ++s) {
            ptx::mbar_init(B.v_full + 8 * s, 1);
            ptx::mbar_init(B.v_empty + 8 * s, 1);
        }
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(B.s_full + 8 * i, 1);
            ptx::mbar_init(B.p_full + 8 * i, 4);
            ptx::mbar_init(B.o_done + 8 * i, 1);
        }
        ptx::mbar_init(B.v_aux, 1);
        ptx::mbar_init(B.drain, 1);
        *abort_flag = 0;
        ptx::prefetch_tmap(&q_map);
        ptx::prefetch_tmap(&kv_map);
        ptx::fence_mbar_init();
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_u32(tmem_slot), C::kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    auto fail = [&](int code) {
        atomicOr(a.err, code);
        *abort_flag = 1;
    };

    if (warp < 4) ptx::setmaxnreg_dec<C::kRegsCtrl>();

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            ptx::mbar_arrive_expect_tx(B.q_full, nh * C::kTile);
            for (int i = 0; i < nh; ++i)
                for (int c = 0; c < D / 64; ++c)
                    ptx::tma_load_3d(sbase + C::kOffQ + i * C::kTile + c * C::kAtom, &q_map, B.q_full,
                                     c * 64, it.head0 + i, it.q_row0);
        }
        const int P = a.P;
        const int pages_per_tile = kPrefillKeys / P;
        const int box_bytes = P * 128;               // P rows x 64 bf16
        const uint64_t policy = ptx::policy_evict_last();
        int issued = 0;   // tiles whose loads were started
        for (int j = 0; j < n_tiles; ++j) {
            if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
            const int valid = min(kPrefillKeys, it.kv_len - j * kPrefillKeys);
            const int n_load = (valid + P - 1) / P;
            // Page ids of this tile, one per lane.
            int page = -1;
            if (lane < n_load) page = a.page_table[it.page_base + j * pages_per_tile + lane];
            const bool bad = lane < n_load && (page < 0 || page >= a.num_pages);
            const unsigned bad_mask = __ballot_sync(0xffffffffu, bad);
            if (bad_mask && lane == 0) atomicOr(a.err, ATTN_DEVICE_ERR_PAGE_ID);
            const int n_good = n_load - __popc(bad_mask);

            // K tile.
            const int ks = j % C::kStagesK;
            if (j >= C::kStagesK &&
                !__all_sync(0xffffffffu, ptx::mbar_wait(B.k_empty + 8 * ks, ((j / C::kStagesK) - 1) & 1))) {
                fail(ATTN_DEVICE_ERR_TIMEOUT);
                break;
            }
            if (lane == 0) ptx::mbar_arrive_expect_tx(B.k_full + 8 * ks, n_good * box_bytes * (D / 64));
            __syncwarp();
            for (int p = 0; p < n_load; ++p) {
                const int pg = __shfl_sync(0xffffffffu, page, p);
                if (lane == 0 && pg >= 0 && pg < a.num_pages)
                    for (int c = 0; c < D / 64; ++c)
                        ptx::tma_load_3d_hint(sbase + C::kOffK + ks * C::kTile + c * C::kAtom + p * box_bytes,
                                              &kv_map, B.k_full + 8 * ks, c * 64, 0,
                                              (pg * 2) * a.Hkv + it.kv_head, policy);
            }
            // V tile.
            const int vs = j % C::kStagesV;
            if (j >= C::kStagesV &&
                !__all_sync(0xffffffffu, ptx::mbar_wait(B.v_empty + 8 * vs, ((j / C::kStagesV) - 1) & 1))) {
                fail(ATTN_DEVICE_ERR_TIMEOUT);
                break;
            }
            const uint32_t vdst = sbase + C::kOffV + vs * C::kTile;
            const bool ragged = valid < kPrefillKeys;
            const uint32_t vbar = ragged ? B.v_aux : B.v_full + 8 * vs;
            if (lane == 0) ptx::mbar_arrive_expect_tx(vbar, n_good * box_bytes * (D / 64));
            __syncwarp();
            for (int p = 0; p < n_load; ++p) {
                const int pg = __shfl_sync(0xffffffffu, page, p);
                if (lane == 0 && pg >= 0 && pg < a.num_pages)
                    for (int c = 0; c < D / 64; ++c)
                        ptx::tma_load_3d_hint(vdst + c * C::kAtom + p * box_bytes, &kv_map, vbar, c * 64, 0,
                                              (pg * 2 + 1) * a.Hkv + it.kv_head, policy);
            }
            if (ragged) {
                // Only the last tile can be ragged: wait for its rows to land,
                // zero V rows [valid, 128) (they may hold anything), then
                // publish the stage to the MMA warp.
                if (!__all_sync(0xffffffffu, ptx::mbar_wait(B.v_aux, 0))) {
                    fail(ATTN_DEVICE_ERR_TIMEOUT);
                    break;
                }
                uint8_t* vrow = smem + C::kOffV + vs * C::kTile;
                const int n16 = (kPrefillKeys - valid) * 8;     // 16-byte chunks per atom
                for (int c = 0; c < D / 64; ++c)
                    for (int idx = lane; idx < n16; idx += 32)
                        *reinterpret_cast<uint4*>(vrow + c * C::kAtom + (valid + idx / 8) * 128 + (idx % 8) * 16) =
                            make_uint4(0, 0, 0, 0);
                ptx::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(B.v_full + 8 * vs);
            }
            issued = j + 1;
        }
        if (__any_sync(0xffffffffu, *abort_flag != 0)) {
            // Let the copies still in flight land before the CTA exits.
            for (int j = max(0, issued - C::kStagesK); j < issued; ++j)
                ptx::mbar_wait(B.k_full + 8 * (j % C::kStagesK), (j / C::kStagesK) & 1);
            for (int j = max(0, issued - C::kStagesV); j < issued; ++j)
                ptx::mbar_wait(B.v_full + 8 * (j % C::kStagesV), (j / C::kStagesV) & 1);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_qk = ptx::idesc_bf16(128, 128, false, false);
            constexpr uint32_t idesc_pv = ptx::idesc_bf16(128, D, false, true);
            bool ok = ptx::mbar_wait(B.q_full, 0);
            for (int j = 0; ok && j < n_tiles; ++j) {
                const int ks = j % C::kStagesK, vs = j % C::kStagesV;
                if (!ptx::mbar_wait(B.k_full + 8 * ks, (j / C::kStagesK) & 1)) { ok = false; break; }
                for (int i = 0; i < nh; ++i) {
                    if (j > 0 && !ptx::mbar_wait(B.o_done + 8 * i, (j - 1) & 1)) { ok = false; break; }
                    ptx::tc_fence_after();
                    const uint32_t qa = sbase + C::kOffQ + i * C::kTile;
                    const uint32_t kb = sbase + C::kOffK + ks * C::kTile;
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t off = (kk / 4) * C::kAtom + (kk % 4) * 32;
                        ptx::tc_mma_ss(tmem + i * 128, ptx::smem_desc_sw128(qa + off, 16, 1024),
                                       ptx::smem_desc_sw128(kb + off, 16, 1024), idesc_qk, kk > 0);
                    }
                    ptx::tc_commit(B.s_full + 8 * i);
                }
                if (!ok) break;
                ptx::tc_commit(B.k_empty + 8 * ks);
                if (!ptx::mbar_wait(B.v_full + 8 * vs, (j / C::kStagesV) & 1)) { ok = false; break; }
                for (int i = 0; i < nh; ++i) {
                    if (!ptx::mbar_wait(B.p_full + 8 * i, j & 1)) { ok = false; break; }
                    ptx::tc_fence_after();
                    const uint32_t vb = sbase + C::kOffV + vs * C::kTile;
#pragma unroll
                    for (int kk = 0; kk < kPrefillKeys / 16; ++kk)
                        ptx::tc_mma_ts(tmem + 256 + i * D, tmem + i * 128 + kk * 8,
                                       ptx::smem_desc_sw128(vb + kk * 2048, C::kAtom, 1024), idesc_pv,
                                       (j > 0 || kk > 0) ? 1u : 0u);
                    ptx::tc_commit(B.o_done + 8 * i);
                }
                if (!ok) break;
                ptx::tc_commit(B.v_empty + 8 * vs);
            }
            if (!ok) fail(ATTN_DEVICE_ERR_TIMEOUT);
            // Arrives once every MMA issued above has finished (tear-down waits on it).
            ptx::tc_commit(B.drain);
        }
    } else if (warp >= 4) {
        // ------------------------------------------------------------ softmax
        ptx::setmaxnreg_inc<C::kRegsSoftmax>();
        const int i = (warp - 4) >> 2;                     // head slot 0 or 1
        const int quad = warp & 3;                         // TMEM lane quadrant of this warp
        const int r = quad * 32 + lane;                    // row within the tile
        if (i < nh) {
            const int head = it.head0 + i;
            const uint32_t t_s = tmem + ((uint32_t)(quad * 32) << 16) + i * 128;
            const uint32_t t_o = tmem + ((uint32_t)(quad * 32) << 16) + 256 + i * D;
            const float sl2 = a.scale_log2;
            // l: row sum of the bf16-rounded P that the PV MMA consumes (it
            // normalises O); le: the same sum of the unrounded P (it gives lse).
            float m_use = -INFINITY, l = 0.f, le = 0.f;
            if (a.sinks != nullptr) {
                m_use = a.sinks[head] * kLog2e;
                l = le = 1.f;
            }
            // Last key this row may see, and the first tile that needs a mask
            // (every earlier tile is fully visible to every row of the tile).
            const int last_key = it.kv_len - 1;
            const int row_limit = a.causal ? min(it.pos0 + r, last_key) : last_key;
            const int first_masked = ((a.causal ? min(it.pos0, last_key) : last_key) + 1) / kPrefillKeys;
            bool ok = true;
            for (int j = 0; j < n_tiles; ++j) {
                if (!__all_sync(0xffffffffu, ptx::mbar_wait(B.s_full + 8 * i, j & 1))) { ok = false; break; }
                ptx::tc_fence_after();
                float s[128];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t v[32];
                    ptx::tmem_ld32(t_s + c * 32, v);
#pragma unroll
                    for (int e = 0; e < 32; ++e) s[c * 32 + e] = __uint_as_float(v[e]);
                }
                ptx::tc_wait_ld();
                if (j >= first_masked) {
                    const int ncol = row_limit - j * kPrefillKeys + 1;
#pragma unroll
                    for (int c = 0; c < 128; ++c)
                        if (c >= ncol) s[c] = -INFINITY;
                }
                float mx = s[0];
#pragma unroll
                for (int c = 1; c < 128; ++c) mx = fmaxf(mx, s[c]);
                const float m_tile = mx * sl2;
                const float m_new = fmaxf(m_use, m_tile);
                float alpha = 1.f;
                bool rescale = false;
                if (m_new > m_use + kRescaleThreshold || (m_use == -INFINITY && m_new != -INFINITY)) {
                    alpha = ptx::ex2(m_use - m_new);
                    l *= alpha;
                    le *= alpha;
                    m_use = m_new;
                    rescale = j > 0;
                }
                if (__any_sync(0xffffffffu, rescale)) {
                    // O (complete up to tile j-1) is rescaled in place.
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t v[32];
                        ptx::tmem_ld32(t_o + c * 32, v);
                        ptx::tc_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
                        ptx::tmem_st32(t_o + c * 32, v);
                    }
                }
                const float neg_m = m_use == -INFINITY ? 0.f : -m_use;
                float ls0 = 0.f, ls1 = 0.f, le0 = 0.f, le1 = 0.f;
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    uint32_t pk[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const float p0 = ptx::ex2(fmaf(s[c * 64 + 2 * e], sl2, neg_m));
                        const float p1 = ptx::ex2(fmaf(s[c * 64 + 2 * e + 1], sl2, neg_m));
                        pk[e] = ptx::pack_bf16x2(p0, p1);
                        const float2 pr = ptx::unpack_bf16x2(pk[e]);
                        ls0 += pr.x;
                        ls1 += pr.y;
                        le0 += p0;
                        le1 += p1;
                    }
                    ptx::tmem_st32(t_s + c * 32, pk);
                }
                l += ls0 + ls1;
                le += le0 + le1;
                ptx::tc_wait_st();
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(B.p_full + 8 * i);
            }
            if (ok && !__all_sync(0xffffffffu, ptx::mbar_wait(B.o_done + 8 * i, (n_tiles - 1) & 1))) ok = false;
            if (!ok) {
                fail(ATTN_DEVICE_ERR_TIMEOUT);
            } else {
                ptx::tc_fence_after();
                const float inv = l > 0.f ? 1.f / l : 0.f;
                const bool store = r < it.n_rows;
                __nv_bfloat16* orow = a.out + ((size_t)(it.q_row0 + r) * a.Hq + head) * D;
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t v[32];
                    ptx::tmem_ld32(t_o + c * 32, v);
                    ptx::tc_wait_ld();
                    if (store) {
#pragma unroll
                        for (int e = 0; e < 32; e += 8) {
                            uint4 w;
                            w.x = ptx::pack_bf16x2(__uint_as_float(v[e]) * inv, __uint_as_float(v[e + 1]) * inv);
                            w.y = ptx::pack_bf16x2(__uint_as_float(v[e + 2]) * inv, __uint_as_float(v[e + 3]) * inv);
                            w.z = ptx::pack_bf16x2(__uint_as_float(v[e + 4]) * inv, __uint_as_float(v[e + 5]) * inv);
                            w.w = ptx::pack_bf16x2(__uint_as_float(v[e + 6]) * inv, __uint_as_float(v[e + 7]) * inv);
                            *reinterpret_cast<uint4*>(orow + c * 32 + e) = w;
                        }
                    }
                }
                if (store && a.lse)
                    a.lse[(size_t)(it.q_row0 + r) * a.Hq + head] =
                        le > 0.f ? (m_use + log2f(le)) * kLn2 : -INFINITY;
            }
        }
    }

    // Tear-down: every TMEM access and MMA is complete (the softmax warps
    // waited for the last PV of their head), so the columns can be released.
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        if (lane == 0) ptx::mbar_wait(B.drain, 0);
        __syncwarp();
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, C::kTmemCols);
    }
}

template <int D>
cudaError_t launch(const CUtensorMap& qm, const CUtensorMap& km, const PrefillArgs& args, int n,
                   cudaStream_t stream) {
    using C = PrefillCfg<D>;
    auto kernel = prefill_sink_attn_kernel<D>;
    static bool configured = false;
    if (!configured) {
        cudaFuncAttributes fa;
        cudaError_t e = cudaFuncGetAttributes(&fa, kernel);
        if (e != cudaSuccess) return e;
        // The register split above assumes this launch size; refuse otherwise.
        if (fa.numRegs < C::kRegsLaunch) return cudaErrorInvalidConfiguration;
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    kernel<<<n, C::kThreads, C::kSmem, stream>>>(qm, km, args);
    return cudaGetLastError();
}

}  // namespace

attn_status launch_prefill(attn_plan_s* plan, const void* q_map, const void* kv_map,
                           const float* sinks, void* out, float* lse, cudaStream_t stream) {
    if (plan->items.empty()) return ATTN_OK;
    PrefillArgs a;
    a.items = reinterpret_cast<const PrefillItem*>(plan->ws + plan->layout.items);
    a.page_table = plan->page_table;
    a.out = static_cast<__nv_bfloat16*>(out);
    a.lse = lse;
    a.sinks = sinks;
    a.err = reinterpret_cast<int32_t*>(plan->ws + plan->layout.err);
    a.Hq = plan->Hq;
    a.Hkv = plan->Hkv;
    a.P = plan->P;
    a.num_pages = plan->num_pages;
    a.causal = plan->causal;
    a.scale_log2 = plan->sm_scale * kLog2e;
    const CUtensorMap& qm = *static_cast<const CUtensorMap*>(q_map);
    const CUtensorMap& km = *static_cast<const CUtensorMap*>(kv_map);
    const int n = (int)plan->items.size();
    const cudaError_t e = plan->D == 64 ? launch<64>(qm, km, a, n, stream) : launch<128>(qm, km, a, n, stream);
    return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace attn
