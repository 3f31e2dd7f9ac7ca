// Prefill sink attention (qo_len > 1) on the 5th-generation tensor cores.
//
// Definition: "GPT-OSS on day 0" (Perplexity), section "Sink Attention": one
// sink logit per query head in the softmax denominator, softmax computed
// online with max subtraction, the running max initialised to the sink (scale
// 1).  Prefill is compute-bound ("Disaggregated prefill and decode", section
// "Prefill vs decode performance"), so QK^T and PV run as tcgen05.mma with
// fp32 accumulators in tensor memory.
//
// Work item = 128 query rows of one request x two query heads of one GQA group
// (both heads share every K/V tile).  The grid is persistent: CTA c walks the
// items the planner assigned to it (greedy longest-processing-time), so the
// next item's Q and K/V loads and QK^T overlap the current item's last
// softmax and epilogue.  Roles (12 warps = 3 warpgroups):
//
//  * warps 0 and 3: TMA producers, warp 0 for Q (double-buffered at D = 64)
//    and the K ring, warp 3 for the V ring, each walking the tiles on its own.
//    Tiles are 128 keys; one box per HND page, issued by its own lane (the
//    boxes of a tile leave in one warp instruction), 128-byte swizzled.  V rows
//    past the end of the sequence are zeroed before the MMA may read them.
//  * warps 1 and 2: tcgen05.mma issuers, one warp per head slot (neither
//    head's MMAs queue behind the other's softmax), one elected lane issuing.
//    S_h = Q_h K^T (both operands K-major in shared memory); O_h += P_h V with
//    V an MN-major shared-memory operand.  At D = 64, P keys 0..95 come from
//    their own TMEM columns and keys 96..127 from shared memory, and V is
//    extended by a ones column so the same MMA accumulates the row sum of the
//    rounded P; S_h of tile j+1 is computed while the softmax of tile j runs,
//    and an item's first QK^T goes ahead of the previous item's last PV.  At
//    D = 128, P is read from tensor memory where S was.
//  * warps 4-7 / 8-11: softmax of head 0 / head 1, one thread per query row
//    (= TMEM lane).  Causal / length mask on diagonal and ragged tiles only;
//    the row max is taken on an item's first tile only; later tiles keep it
//    in one pass, and S stays in TMEM until the tile's P row sum is checked:
//    past 2^64 the tile is redone from TMEM with the max raised and O
//    rescaled.  P is rounded to bf16 and O is normalised by the row sum of
//    that rounded P, while lse uses the unrounded sum.  An item's epilogue
//    runs during the head slot's next item's first tile; at D = 64 each
//    warp's 32 full rows leave through a staging tile and one TMA store;
//    ragged last tiles use plain stores.
//
// TMEM (512 columns): S0 S1 (128 each), O0 O1 (D each, plus at D = 64 the
// 16 row-sum columns), and at D = 64 P0 P1 (keys 0..95, 48 columns each); at
// D = 128 P aliases the first half of S.
// Every wait is bounded; a timeout sets the device error word.
#include <cuda.h>

#include "attn_internal.h"
#include "exp2_poly.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kSumLimit = 18446744073709551616.0f;   // 2^64: tile row sum that forces a new max
// D = 64: keys of P kept in TMEM (the rest of the tile's P goes through
// shared memory); TMEM holds S, O with its row-sum columns and these.
constexpr int kPTmemKeys = 96;
// Every kPolyEvery-th pair of score columns takes its exponentials on the FMA
// pipe (exp2_poly.cuh) instead of the MUFU; 0 = none.  The polynomial clamps
// its argument to 2^126, which still trips the 2^64 row-sum check below.
#ifndef ATTN_PREFILL_POLY_EVERY
#define ATTN_PREFILL_POLY_EVERY 0
#endif
constexpr int kPolyEvery = ATTN_PREFILL_POLY_EVERY;

template <int D>
struct PrefillCfg {
    static constexpr int kThreads = 384;
    // Register split (setmaxnreg): the launch gives every thread kRegsLaunch;
    // warpgroup 0 (producer, MMA) drops to kRegsCtrl and the two softmax
    // warpgroups grow to kRegsSoftmax.  128 * kRegsCtrl + 256 * kRegsSoftmax
    // must not exceed 384 * kRegsLaunch, or setmaxnreg.inc would wait forever.
    static constexpr int kRegsLaunch = 168;
    static constexpr int kRegsCtrl = 56;
    static constexpr int kRegsSoftmax = 224;
    static_assert(128 * kRegsCtrl + 256 * kRegsSoftmax <= kThreads * kRegsLaunch, "register split");

    static constexpr bool kSeparateP = (D == 64);
    static constexpr int kQBufs = (D == 64) ? 2 : 1;
    static constexpr int kStagesK = (D == 64) ? 3 : 2;
    static constexpr int kStagesV = 2;
    static constexpr int kAtom = 128 * 128;              // 128 rows x 64 bf16, swizzled
    static constexpr int kTile = kAtom * (D / 64);       // Q, K or V tile of 128 rows
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = kQBufs * 2 * kTile;
    static constexpr int kOffV = kOffK + kStagesK * kTile;
    // At D = 64, P is split by keys: keys 0..95 go to TMEM (PV as TS MMA),
    // keys 96..127 to shared memory (SS MMA), and the PV B operand is V
    // extended by a ones column, so the same MMA also accumulates the row sum
    // of the bf16-rounded P next to O (N = D + 16 costs no tensor time over
    // N = D here).  TMEM then holds exactly S, O and P of both head slots.
    static constexpr bool kSplitP = (D == 64);
    static constexpr int kON = kSplitP ? D + 16 : D;      // O accumulator columns
    static constexpr int kOffPb = kOffV + kStagesV * kTile;                 // per head 128 rows x 128 B
    // D = 64: per head slot, the output tile staged for its TMA store (each
    // warp's 32-row stripe leaves in its own store).
    static constexpr int kOffStage = kOffPb + (kSplitP ? 2 * kAtom : 0);
    static constexpr int kOffOnes = kOffStage + (kSplitP ? 2 * kAtom : 0);  // 16 key rows x 128 B
    static constexpr int kOffBar = kOffOnes + (kSplitP ? 2048 : 0);
    static constexpr int kNumBars = 2 * kQBufs + 2 * kStagesK + 2 * kStagesV + 8 + 2 + 8;
    static constexpr int kSmem = 1024 + kOffBar + kNumBars * 8 + 16;
    static constexpr uint32_t kTmemCols = 512;
    // TMEM columns of head slot i (every region starts on a multiple of 32).
    // D = 64:  S 0 | 128, O (+ row sum) 256 | 384, P keys 0..95 at 336 | 464.
    // D = 128: S 0 | 128, O 256 | 384, P aliases the first half of S.
    static __device__ __forceinline__ uint32_t col_s(int i) { return i * 128; }
    static __device__ __forceinline__ uint32_t col_o(int i) { return 256 + i * 128; }
    static __device__ __forceinline__ uint32_t col_p(int i) { return kSplitP ? 256 + i * 128 + kON : i * 128; }
};

struct PrefillArgs {
    const PrefillItem* items;
    const int32_t* item_off;     // CTA c runs items [item_off[c], item_off[c+1])
    const int32_t* page_table;
    __nv_bfloat16* out;
    float* lse;
    const float* sinks;
    int32_t* err;
    int32_t Hq, Hkv, P, num_pages, causal;
    float scale_log2;
};

struct Bars {
    uint32_t q_full, q_empty, k_full, k_empty, v_full, v_empty, s_full, s_free, p_full, o_done,
        v_aux, drain, turn;
};

// Warp-uniform bounded wait.
__device__ __forceinline__ bool wait_all(uint32_t bar, uint32_t parity) {
    return __all_sync(0xffffffffu, ptx::mbar_wait(bar, parity));
}

// kRagged: K and V are contiguous [tokens][Hkv][D] arrays (kv_map over K,
// v_map over V) instead of the paged HND pool (kv_map; v_map unused), and an
// item's page_base is its first token.
template <int D, bool kRagged>
__global__ void __launch_bounds__(PrefillCfg<D>::kThreads, 1)
prefill_sink_attn_kernel(const __grid_constant__ CUtensorMap q_map,
                         const __grid_constant__ CUtensorMap kv_map,
                         const __grid_constant__ CUtensorMap v_map,
                         const __grid_constant__ CUtensorMap o_map, const PrefillArgs a) {
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
    B.q_empty = B.q_full + 8 * C::kQBufs;
    B.k_full = B.q_empty + 8 * C::kQBufs;
    B.k_empty = B.k_full + 8 * C::kStagesK;
    B.v_full = B.k_empty + 8 * C::kStagesK;
    B.v_empty = B.v_full + 8 * C::kStagesV;
    B.s_full = B.v_empty + 8 * C::kStagesV;
    B.s_free = B.s_full + 16;
    B.p_full = B.s_free + 16;
    B.o_done = B.p_full + 16;
    B.v_aux = B.o_done + 16;
    B.drain = B.v_aux + 8;
    B.turn = B.drain + 8;   // [quadrant][head slot]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int item_begin = a.item_off[blockIdx.x], item_end = a.item_off[blockIdx.x + 1];

    if (tid == 0) {
        // The "empty" barriers and `drain` take one arrival from each of the
        // two MMA threads (head slots 0 and 1).
        for (int b = 0; b < C::kQBufs; ++b) {
            ptx::mbar_init(B.q_full + 8 * b, 1);
            ptx::mbar_init(B.q_empty + 8 * b, 2);
        }
        for (int s = 0; s < C::kStagesK; ++s) {
            ptx::mbar_init(B.k_full + 8 * s, 1);
            ptx::mbar_init(B.k_empty + 8 * s, 2);
        }
        for (int s = 0; s < C::kStagesV; ++s) {
            ptx::mbar_init(B.v_full + 8 * s, 1);
            ptx::mbar_init(B.v_empty + 8 * s, 2);
        }
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(B.s_full + 8 * i, 1);
            ptx::mbar_init(B.s_free + 8 * i, 4);
            ptx::mbar_init(B.p_full + 8 * i, 4);
            ptx::mbar_init(B.o_done + 8 * i, 1);
        }
        ptx::mbar_init(B.v_aux, 1);
        ptx::mbar_init(B.drain, 2);
        for (int k = 0; k < 8; ++k) ptx::mbar_init(B.turn + 8 * k, 1);
        *abort_flag = 0;
        ptx::prefetch_tmap(&q_map);
        ptx::prefetch_tmap(&kv_map);
        ptx::prefetch_tmap(&o_map);
        ptx::fence_mbar_init();
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_u32(tmem_slot), C::kTmemCols);
        ptx::tmem_relinquish();
    }
    if (C::kSplitP && warp == 2) {
        // The ones block of the PV B operand: 16 key rows x 64 N values, N
        // value 0 (the row-sum column) = 1.0 bf16, laid out with the same
        // 128-byte swizzle as V (16-byte chunk c of row k sits at c ^ (k % 8)).
        for (int idx = lane; idx < 2048 / 16; idx += 32) {
            const int k = idx >> 3, c = idx & 7;
            *reinterpret_cast<uint4*>(smem + C::kOffOnes + idx * 16) =
                make_uint4(c == (k & 7) ? 0x3F80u : 0u, 0u, 0u, 0u);
        }
        ptx::fence_proxy_async_smem();
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

    if (warp == 0 || warp == 3) {
        // ================================================================ producers
        // Warp 0 loads Q and K, warp 3 loads V: two independent walks over this
        // CTA's tiles, so a K tile never waits behind a V stage (or vice versa).
        const bool is_k = warp == 0;
        const int P = a.P;
        const int pages_per_tile = kPrefillKeys / P;
        const int box_bytes = P * 128;               // P rows x 64 bf16
        const int n_stages = is_k ? C::kStagesK : C::kStagesV;
        const uint32_t full0 = is_k ? B.k_full : B.v_full;
        const uint32_t empty0 = is_k ? B.k_empty : B.v_empty;
        const uint32_t dst0 = sbase + (is_k ? C::kOffK : C::kOffV);
        const uint64_t policy = ptx::policy_evict_last();
        int jg = 0, n_item = 0, n_aux = 0, issued = 0;
        bool ok = true;
        // The page ids of the next tile are loaded (one per lane) while the
        // current tile is issued, so the dependent global load never sits
        // between two tiles.
        auto n_load_of = [&](const PrefillItem& x, int j) {
            return (min(kPrefillKeys, x.kv_len - j * kPrefillKeys) + P - 1) / P;
        };
        auto load_pages = [&](const PrefillItem& x, int j) {
            if constexpr (kRagged) return 0;
            return lane < n_load_of(x, j) ? a.page_table[x.page_base + j * pages_per_tile + lane] : -1;
        };
        int item = item_begin, j = 0;
        PrefillItem it = a.items[item];
        int page = load_pages(it, 0);
        while (item < item_end) {
            if (__any_sync(0xffffffffu, *abort_flag != 0)) { ok = false; break; }
            int item_n = item, j_n = j + 1;
            PrefillItem it_n = it;
            if (j_n == it.n_kv_tiles) {
                item_n = item + 1;
                j_n = 0;
                if (item_n < item_end) it_n = a.items[item_n];
            }
            const int page_n = item_n < item_end ? load_pages(it_n, j_n) : -1;

            if (is_k && j == 0) {
                const int qb = n_item % C::kQBufs;
                if (n_item >= C::kQBufs && !wait_all(B.q_empty + 8 * qb, ((n_item / C::kQBufs) - 1) & 1)) {
                    fail(ATTN_DEVICE_ERR_TIMEOUT);
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    ptx::mbar_arrive_expect_tx(B.q_full + 8 * qb, it.n_heads * C::kTile);
                    for (int i = 0; i < it.n_heads; ++i)
                        for (int c = 0; c < D / 64; ++c)
                            ptx::tma_load_3d(sbase + C::kOffQ + (qb * 2 + i) * C::kTile + c * C::kAtom, &q_map,
                                             B.q_full + 8 * qb, c * 64, it.head0 + i, it.q_row0);
                }
            }
            const int valid = min(kPrefillKeys, it.kv_len - j * kPrefillKeys);
            const int n_load = (valid + P - 1) / P;
            const bool bad = !kRagged && lane < n_load && (page < 0 || page >= a.num_pages);
            const unsigned bad_mask = __ballot_sync(0xffffffffu, bad);
            if (bad_mask && lane == 0) atomicOr(a.err, ATTN_DEVICE_ERR_PAGE_ID);
            // Ragged: one box of 128 tokens per 64 dims (rows past the request
            // or the array arrive too, and are masked or zeroed like a page tail).
            const int tx = kRagged ? C::kTile : (n_load - __popc(bad_mask)) * box_bytes * (D / 64);

            const int st = jg % n_stages;
            if (jg >= n_stages && !wait_all(empty0 + 8 * st, ((jg / n_stages) - 1) & 1)) {
                fail(ATTN_DEVICE_ERR_TIMEOUT);
                ok = false;
                break;
            }
            // V rows past the end of the sequence must be zeroed before the MMA
            // may read them, so a ragged V tile lands on `v_aux` first.
            const bool ragged = !is_k && valid < kPrefillKeys;
            const uint32_t bar = ragged ? B.v_aux : full0 + 8 * st;
            if (lane == 0) ptx::mbar_arrive_expect_tx(bar, tx);
            // One page box per lane: the boxes of a tile leave in one warp instruction.
            __syncwarp();
            if constexpr (kRagged) {
                if (lane == 0)
                    for (int c = 0; c < D / 64; ++c)
                        ptx::tma_load_3d_hint(dst0 + st * C::kTile + c * C::kAtom, is_k ? &kv_map : &v_map, bar,
                                              c * 64, it.kv_head, it.page_base + j * kPrefillKeys, policy);
            } else if (lane < n_load && page >= 0 && page < a.num_pages) {
                for (int c = 0; c < D / 64; ++c)
                    ptx::tma_load_3d_hint(dst0 + st * C::kTile + c * C::kAtom + lane * box_bytes, &kv_map, bar,
                                          c * 64, 0, (page * 2 + (is_k ? 0 : 1)) * a.Hkv + it.kv_head, policy);
            }
            if (ragged) {
                // Only an item's last tile can be ragged: wait for its rows,
                // zero V rows [valid, 128) (they may hold anything), publish.
                if (!wait_all(B.v_aux, n_aux & 1)) {
                    fail(ATTN_DEVICE_ERR_TIMEOUT);
                    ok = false;
                    break;
                }
                ++n_aux;
                uint8_t* vrow = smem + C::kOffV + st * C::kTile;
                const int n16 = (kPrefillKeys - valid) * 8;   // 16-byte chunks per atom
                for (int c = 0; c < D / 64; ++c)
                    for (int idx = lane; idx < n16; idx += 32)
                        *reinterpret_cast<uint4*>(vrow + c * C::kAtom + (valid + idx / 8) * 128 + (idx % 8) * 16) =
                            make_uint4(0, 0, 0, 0);
                ptx::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(B.v_full + 8 * st);
            }
            issued = jg + 1;

            ++jg;
            if (j_n == 0) ++n_item;
            item = item_n;
            j = j_n;
            it = it_n;
            page = page_n;
        }
        if (!ok) {
            // Let the copies still in flight land before the CTA exits.
            for (int t = max(0, issued - n_stages); t < issued; ++t)
                ptx::mbar_wait(full0 + 8 * (t % n_stages), (t / n_stages) & 1);
        }
    } else if (warp == 1 || warp == 2) {
        // ================================================================ MMA issuers
        // One warp per head slot, so neither head's MMAs wait behind the other
        // head's softmax.  The whole warp walks the schedule (descriptors and
        // TMEM addresses stay warp-uniform, in uniform registers) and one
        // elected lane issues each group of tcgen05.mma and commits.  Both
        // warps release the shared K, V and Q stages.
        const int i = __shfl_sync(0xffffffffu, warp - 1, 0);
        constexpr uint32_t idesc_qk = ptx::idesc_bf16(128, 128, false, false);
        constexpr uint32_t idesc_pv = ptx::idesc_bf16(128, C::kON, false, true);
        const uint32_t t_s = tmem + C::col_s(i);
        const uint32_t t_o = tmem + C::col_o(i);
        const uint32_t t_p = tmem + C::col_p(i);
        const bool leader = ptx::elect_one();
        int jg = 0, n_item = 0, hj = 0;
        bool ok = true;

        // S = Q K^T of the K stage ks, then free the stage (and Q after the
        // item's last QK^T).
        auto qk = [&](int qb, int ks, bool last_of_item) {
            if (leader) {
                ptx::tc_fence_after();
                const uint32_t qa = sbase + C::kOffQ + (qb * 2 + i) * C::kTile;
                const uint32_t kb = sbase + C::kOffK + ks * C::kTile;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk / 4) * C::kAtom + (kk % 4) * 32;
                    ptx::tc_mma_ss(t_s, ptx::smem_desc_sw128(qa + off, 16, 1024),
                                   ptx::smem_desc_sw128(kb + off, 16, 1024), idesc_qk, kk > 0);
                }
                ptx::tc_commit(B.s_full + 8 * i);
                ptx::tc_commit(B.k_empty + 8 * ks);
                if (last_of_item) ptx::tc_commit(B.q_empty + 8 * qb);
            }
            __syncwarp();
        };
        // O += P V of the V stage vs, then free the stage.
        auto pv = [&](int vs, bool first) {
            if (leader) {
                ptx::tc_fence_after();
                const uint32_t vb = sbase + C::kOffV + vs * C::kTile;
                if constexpr (C::kSplitP) {
                    // B = [V | ones]: the second 64-wide N atom of every K step
                    // is the same 16-row ones block (its own LBO per step).
                    const uint32_t ones = sbase + C::kOffOnes;
                    const uint32_t pb = sbase + C::kOffPb + i * C::kAtom;
#pragma unroll
                    for (int kk = 0; kk < kPrefillKeys / 16; ++kk) {
                        const uint32_t vk = vb + kk * 2048;
                        const uint64_t bd = ptx::smem_desc_sw128(vk, ones - vk, 1024);
                        if (kk < kPTmemKeys / 16)
                            ptx::tc_mma_ts(t_o, t_p + kk * 8, bd, idesc_pv, (!first || kk > 0) ? 1u : 0u);
                        else
                            ptx::tc_mma_ss(t_o, ptx::smem_desc_sw128(pb + (kk - kPTmemKeys / 16) * 32, 16, 1024), bd,
                                           idesc_pv, 1u);
                    }
                } else {
#pragma unroll
                    for (int kk = 0; kk < kPrefillKeys / 16; ++kk)
                        ptx::tc_mma_ts(t_o, t_p + kk * 8, ptx::smem_desc_sw128(vb + kk * 2048, C::kAtom, 1024),
                                       idesc_pv, (!first || kk > 0) ? 1u : 0u);
                }
                ptx::tc_commit(B.o_done + 8 * i);
                ptx::tc_commit(B.v_empty + 8 * vs);
            }
            __syncwarp();
        };
        auto kfull = [&](int t) { return wait_all(B.k_full + 8 * (t % C::kStagesK), (t / C::kStagesK) & 1); };
        auto vfull = [&](int t) { return wait_all(B.v_full + 8 * (t % C::kStagesV), (t / C::kStagesV) & 1); };

        // The next item's tile and head counts are loaded one item ahead, so
        // their global load never sits between two items' MMAs.
        int nx_tiles = 0, nx_heads = 0;
        if (item_begin < item_end) {
            nx_tiles = a.items[item_begin].n_kv_tiles;
            nx_heads = a.items[item_begin].n_heads;
        }
        // D = 64: an item's last PV waits for its P, so the next item's first
        // QK^T (which needs only its Q, K and the S buffer) goes ahead of it.
        bool pre = false;   // this item's first QK^T is already issued
        for (int item = item_begin; ok && item < item_end; ++item, ++n_item) {
            if (*abort_flag) { ok = false; break; }
            const int n = nx_tiles, n_heads = nx_heads;
            if (item + 1 < item_end) {
                nx_tiles = a.items[item + 1].n_kv_tiles;
                nx_heads = a.items[item + 1].n_heads;
            }
            const int qb = n_item % C::kQBufs;
            if (!pre && !wait_all(B.q_full + 8 * qb, (n_item / C::kQBufs) & 1)) { ok = false; break; }
            if (i >= n_heads) {
                // This head slot has no work in the item: only keep the
                // shared stages' arrival counts (after each stage is loaded).
                for (int j = 0; j < n && ok; ++j) {
                    const int t = jg + j;
                    if (!kfull(t)) { ok = false; break; }
                    if (leader) ptx::mbar_arrive(B.k_empty + 8 * (t % C::kStagesK));
                    if (!vfull(t)) { ok = false; break; }
                    if (leader) ptx::mbar_arrive(B.v_empty + 8 * (t % C::kStagesV));
                }
                if (leader) ptx::mbar_arrive(B.q_empty + 8 * qb);
                __syncwarp();
                jg += n;
                continue;
            }
            if (C::kSeparateP) {
                // QK^T of tile j+1 is issued before PV of tile j.
                if (!pre) {
                    if (!kfull(jg)) { ok = false; break; }
                    if (hj > 0 && !wait_all(B.s_free + 8 * i, (hj - 1) & 1)) { ok = false; break; }
                    qk(qb, jg % C::kStagesK, n == 1);
                }
                pre = false;
                for (int j = 0; j < n; ++j) {
                    const int t = jg + j;
                    if (j + 1 < n) {
                        if (!kfull(t + 1) || !wait_all(B.s_free + 8 * i, (hj + j) & 1)) { ok = false; break; }
                        qk(qb, (t + 1) % C::kStagesK, j + 2 == n);
                    } else if (item + 1 < item_end && i < nx_heads) {
                        const int qb2 = (n_item + 1) % C::kQBufs;
                        if (!wait_all(B.q_full + 8 * qb2, ((n_item + 1) / C::kQBufs) & 1) || !kfull(t + 1) ||
                            !wait_all(B.s_free + 8 * i, (hj + j) & 1)) { ok = false; break; }
                        qk(qb2, (t + 1) % C::kStagesK, nx_tiles == 1);
                        pre = true;
                    }
                    if (!vfull(t) || !wait_all(B.p_full + 8 * i, (hj + j) & 1)) { ok = false; break; }
                    pv(t % C::kStagesV, j == 0);
                }
            } else {
                // P aliases S: QK^T of tile j waits for PV of tile j-1.
                for (int j = 0; j < n; ++j) {
                    const int t = jg + j;
                    if (!kfull(t)) { ok = false; break; }
                    if (hj + j > 0 && !wait_all(B.o_done + 8 * i, (hj + j - 1) & 1)) { ok = false; break; }
                    qk(qb, t % C::kStagesK, j + 1 == n);
                    if (!vfull(t) || !wait_all(B.p_full + 8 * i, (hj + j) & 1)) { ok = false; break; }
                    pv(t % C::kStagesV, j == 0);
                }
            }
            jg += n;
            hj += n;
        }
        if (!ok && leader) fail(ATTN_DEVICE_ERR_TIMEOUT);
        // Arrives once every MMA this warp issued has finished.
        if (leader) ptx::tc_commit(B.drain);
        __syncwarp();
    } else if (warp >= 4) {
        // ================================================================ softmax
        ptx::setmaxnreg_inc<C::kRegsSoftmax>();
        const int i = (warp - 4) >> 2;                     // head slot 0 or 1
        const int quad = warp & 3;                         // TMEM lane quadrant of this warp
        const int r = quad * 32 + lane;                    // row within the tile
        const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
        const uint32_t t_s = tmem + lane_off + C::col_s(i);
        const uint32_t t_o = tmem + lane_off + C::col_o(i);
        const uint32_t t_p = tmem + lane_off + C::col_p(i);
        // This thread's row of P keys 96..127 in shared memory (D = 64): the
        // first 64 bytes of a 128-byte row, 16-byte chunks swizzled by the
        // row (K-major SW128 A operand).
        const uint32_t pb_row = sbase + C::kOffPb + i * C::kAtom + (r >> 3) * 1024 + (r & 7) * 128;
        const float sl2 = a.scale_log2;
        const float poly_a = sl2 * exp2poly::kInvRange;   // scale of the FMA-pipe pairs' argument
        int hj = 0;
        bool ok = true;
        // Turn-taking with the other head slot's warp on the same SM
        // sub-partition (same quadrant): in items with two heads the two warps
        // run their exp loops one after the other, so each loop has the
        // multi-function unit to itself while the other warp does its loads,
        // waits and stores.  Head slot 0 goes first.
        const uint32_t my_turn = B.turn + 8 * (quad * 2 + i), other_turn = B.turn + 8 * (quad * 2 + (i ^ 1));
        int n_turn = 0;
        // Deferred epilogue: an item's O is read from TMEM, normalised and
        // stored during this head slot's next item's first tile, after its
        // exponentials -- the item's last PV has finished by then (the MMA
        // warp issues the next item's first QK^T ahead of it), and the work
        // overlaps the other head slot's exponentials instead of stalling
        // both.  PV of that tile overwrites O, so it runs before P is stored.
        // D = 64: a warp's 32 full rows leave through the staging tile and
        // one TMA store (rows one thread apart are 8 KB apart in `out`, so
        // per-thread stores would touch 32 lines per instruction); the stripe
        // is reused one item later, after this warp's store has read it.
        const uint32_t st_stripe = sbase + C::kOffStage + i * C::kAtom + quad * 4096;
        const uint32_t st_row = st_stripe + (lane >> 3) * 1024 + (lane & 7) * 128;
        // The pending item is kept as its index, its lse and the sink's part
        // of its row sum (three registers across the next item's tile).
        bool epi = false;
        int e_item = 0;
        float e_l = 0.f, e_lse = 0.f;
        auto epilogue = [&]() -> bool {
            if (!wait_all(B.o_done + 8 * i, (hj - 1) & 1)) return false;   // its last PV
            const PrefillItem ei = a.items[e_item];
            const int e_row0 = ei.q_row0, e_head = ei.head0 + i, e_rows = ei.n_rows;
            ptx::tc_fence_after();
            float lt = e_l;
            if constexpr (C::kSplitP) {   // the keys' part of the row sum, next to O
                uint32_t v[16];
                ptx::tmem_ld16(t_o + D, v);
                ptx::tc_wait_ld();
                lt += __uint_as_float(v[0]);
            }
            const float inv = lt > 0.f ? 1.f / lt : 0.f;
            if (C::kSplitP && quad * 32 + 32 <= e_rows) {
                if (lane == 0) ptx::bulk_wait_read_all();   // the stripe's previous store has read it
                __syncwarp();
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t v[32];
                    ptx::tmem_ld32(t_o + c * 32, v);
                    ptx::tc_wait_ld();
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int e = 8 * q;
                        ptx::st_shared_v4(
                            st_row + (((c * 4 + q) ^ (lane & 7)) << 4),
                            ptx::pack_bf16x2(__uint_as_float(v[e]) * inv, __uint_as_float(v[e + 1]) * inv),
                            ptx::pack_bf16x2(__uint_as_float(v[e + 2]) * inv, __uint_as_float(v[e + 3]) * inv),
                            ptx::pack_bf16x2(__uint_as_float(v[e + 4]) * inv, __uint_as_float(v[e + 5]) * inv),
                            ptx::pack_bf16x2(__uint_as_float(v[e + 6]) * inv, __uint_as_float(v[e + 7]) * inv));
                    }
                }
                ptx::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    ptx::tma_store_3d(&o_map, st_stripe, 0, e_head, e_row0 + quad * 32);
                    ptx::bulk_commit_group();
                }
            } else {
                // Rows of a ragged last tile (a box would overwrite the next
                // request's rows) and D = 128: per-thread stores.
                const bool store = r < e_rows;
                __nv_bfloat16* orow = a.out + ((size_t)(e_row0 + r) * a.Hq + e_head) * D;
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
            }
            if (r < e_rows && a.lse) a.lse[(size_t)(e_row0 + r) * a.Hq + e_head] = e_lse;
            return true;
        };
        if (i == 1 && lane == 0) ptx::mbar_arrive(other_turn);
        // Item descriptors and sinks are read from L1: the sinks' lines are
        // prefetched here, each next descriptor after the current item's last
        // tile.
        if (a.sinks != nullptr && lane * 32 < a.Hq) ptx::prefetch_l1(a.sinks + lane * 32);
        for (int item = item_begin; ok && item < item_end; ++item) {
            const PrefillItem it = a.items[item];
            if (i >= it.n_heads) continue;
            const int head = it.head0 + i;
            const int n = it.n_kv_tiles;
            // l: row sum of the bf16-rounded P that the PV MMA consumes (it
            // normalises O); le: the same sum of the unrounded P (it gives lse).
            // At D = 64 the keys' part of l accumulates in TMEM next to O (the
            // ones column), and l here holds only the sink's term.
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
            // The first tile of an item sets the running max.  Later tiles
            // reuse it and skip the max: P = 2^(s - m) is computed directly,
            // and only when the tile's row sum exceeds 2^64 (some P could then
            // be large enough to overflow the sums) is the tile redone: S is
            // loaded again (it stays in TMEM until the check has passed), the
            // max raised and O rescaled.  Any max is a valid softmax shift, so
            // the result does not depend on when it moves.  The redo re-enters
            // the loop body for the same tile (the S wait returns at once), so
            // the scores need not stay live past the exponentials.
            bool redo = false;
            for (int j = 0; j < n; ++j) {
                const int t = hj + j;
                if (!wait_all(B.s_full + 8 * i, t & 1)) { ok = false; break; }
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
                // At D = 64 the previous PV must be done before O is touched or
                // P is overwritten (at D = 128 it is: S of tile j waited for it).
                bool prev_done = !C::kSeparateP || t == 0;
                if (j == 0 || redo) {
                    // Raise the running max to cover this tile (row max: 16
                    // independent chains of 3-input max, then a tree).
                    float mq[16];
#pragma unroll
                    for (int k = 0; k < 16; ++k)
                        mq[k] = ptx::max3(ptx::max3(s[k], s[16 + k], s[32 + k]),
                                          ptx::max3(s[48 + k], s[64 + k], s[80 + k]),
                                          ptx::max3(s[96 + k], s[112 + k], s[112 + k]));
#pragma unroll
                    for (int k = 0; k < 5; ++k) mq[k] = ptx::max3(mq[k], mq[5 + k], mq[10 + k]);
                    const float tmax = ptx::max3(ptx::max3(mq[0], mq[1], mq[2]), ptx::max3(mq[3], mq[4], mq[15]), mq[15]);
                    const float m_new = fmaxf(m_use, tmax * sl2);
                    const float alpha = m_new > m_use ? ptx::ex2(m_use - m_new) : 1.f;
                    l *= alpha;
                    le *= alpha;
                    m_use = m_new;
                    if (redo) {   // rescale what the earlier tiles put in O
                        if (!prev_done) {
                            if (!wait_all(B.o_done + 8 * i, (t - 1) & 1)) { ok = false; break; }
                            prev_done = true;
                            ptx::tc_fence_after();
                        }
#pragma unroll
                        for (int c = 0; c < D / 32; ++c) {
                            uint32_t v[32];
                            ptx::tmem_ld32(t_o + c * 32, v);
                            ptx::tc_wait_ld();
#pragma unroll
                            for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
                            ptx::tmem_st32(t_o + c * 32, v);
                        }
                        if constexpr (C::kSplitP) {   // the row-sum columns
                            uint32_t v[16];
                            ptx::tmem_ld16(t_o + D, v);
                            ptx::tc_wait_ld();
#pragma unroll
                            for (int e = 0; e < 16; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
                            ptx::tmem_st16(t_o + D, v);
                        }
                        ptx::tc_wait_st();
                    }
                }
                uint32_t pk[2][32];
                float tile_l = 0.f, tile_le = 0.f;
                const bool take_turns = C::kSplitP && it.n_heads == 2;
                // The turn is handed over right after the exponentials, before the
                // overflow check.  A redo runs outside the turn order: the turn
                // only spaces out the two warps' MUFU use, and each warp must
                // take exactly one turn per tile, or a warp that redoes tiles
                // would wait for hand-overs that its partner, tiles ahead,
                // cannot give before the K and V rings wait for this warp.
                if (take_turns && !redo && !wait_all(my_turn, n_turn & 1)) { ok = false; break; }
                {
                    const float neg_m = m_use == -INFINITY ? 0.f : -m_use;
                    const float2 sl2x2 = make_float2(sl2, sl2), negm2 = make_float2(neg_m, neg_m);
                    // Pairs on the FMA pipe: y = sat(s * sl2 / R + 1/2 - m / R).
                    const float pb = fmaf(neg_m, exp2poly::kInvRange, 0.5f);
                    float2 ls2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
                    float2 lx2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
#pragma unroll
                        for (int e = 0; e < 32; ++e) {
                            const float s0 = s[c * 64 + 2 * e], s1 = s[c * 64 + 2 * e + 1];
                            float2 p;
                            if (kPolyEvery > 0 && (c * 32 + e) % (kPolyEvery > 0 ? kPolyEvery : 1) == kPolyEvery - 1) {
                                p = exp2poly::exp2_pair(s0, s1, poly_a, pb);
                            } else {
                                const float2 x = ptx::fma2(make_float2(s0, s1), sl2x2, negm2);
                                p = make_float2(ptx::ex2(x.x), ptx::ex2(x.y));
                            }
                            pk[c][e] = ptx::pack_bf16x2(p.x, p.y);
                            if constexpr (!C::kSplitP)
                                ls2[e & 1] = ptx::add2(ls2[e & 1], ptx::unpack_bf16x2(pk[c][e]));
                            lx2[e & 1] = ptx::add2(lx2[e & 1], p);
                        }
                    }
                    const float2 lsum = ptx::add2(ls2[0], ls2[1]), lxsum = ptx::add2(lx2[0], lx2[1]);
                    tile_l = lsum.x + lsum.y;
                    tile_le = lxsum.x + lxsum.y;
                }
                if (take_turns && !redo) {
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive(other_turn);
                    ++n_turn;
                }
                if (j > 0 && !redo && __any_sync(0xffffffffu, tile_le > kSumLimit)) {
                    redo = true;
                    --j;
                    continue;
                }
                redo = false;
                if (C::kSeparateP) {
                    // S is no longer needed: the MMA warp may overwrite it with the next tile.
                    ptx::tc_fence_before();
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive(B.s_free + 8 * i);
                }
                if (!ok) break;
                if (epi) {   // the previous item's output (only ever pending at j == 0)
                    if (!epilogue()) { ok = false; break; }
                    epi = false;
                }
                l += tile_l;
                le += tile_le;
                if (!prev_done) {
                    if (!wait_all(B.o_done + 8 * i, (t - 1) & 1)) { ok = false; break; }
                    ptx::tc_fence_after();
                }
                ptx::tmem_st32(t_p, pk[0]);
                if constexpr (C::kSplitP) {
                    // keys 64..95 to TMEM, 96..127 to shared memory
                    uint32_t mid[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) mid[e] = pk[1][e];
                    ptx::tmem_st16(t_p + 32, mid);
#pragma unroll
                    for (int c = 0; c < (kPrefillKeys - kPTmemKeys) / 8; ++c)
                        ptx::st_shared_v4(pb_row + ((c ^ (r & 7)) << 4), pk[1][16 + 4 * c], pk[1][16 + 4 * c + 1],
                                          pk[1][16 + 4 * c + 2], pk[1][16 + 4 * c + 3]);
                    ptx::fence_proxy_async_smem();   // the SS MMA reads it through the async proxy
                } else {
                    ptx::tmem_st32(t_p + 32, pk[1]);
                }
                ptx::tc_wait_st();
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(B.p_full + 8 * i);
            }
            if (!ok) break;
            if (item + 1 < item_end && lane < 2)   // a descriptor may straddle two lines
                ptx::prefetch_l1(reinterpret_cast<const char*>(a.items + item + 1) + lane * (sizeof(PrefillItem) - 1));
            epi = true;
            e_item = item;
            e_l = l;
            // le >= 1 here (the term that set the running max contributes 1), so
            // the MUFU's approximate lg2 is within 2^-22 of log2(le).
            e_lse = le > 0.f ? (m_use + __log2f(le)) * kLn2 : -INFINITY;
            hj += n;
        }
        if (ok && epi) ok = epilogue();
        if (!ok) fail(ATTN_DEVICE_ERR_TIMEOUT);
        if (lane == 0) ptx::bulk_wait_all();   // output stores complete before the CTA exits
    }

    // Tear-down: each MMA thread's last commit arrives on `drain` once every
    // MMA it issued is complete; then the TMEM columns are released.
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        if (lane == 0) ptx::mbar_wait(B.drain, 0);
        __syncwarp();
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, C::kTmemCols);
    }
}

template <int D, bool kRagged>
cudaError_t launch(const CUtensorMap& qm, const CUtensorMap& km, const CUtensorMap& vm, const CUtensorMap& om,
                   const PrefillArgs& args, int grid, cudaStream_t stream) {
    using C = PrefillCfg<D>;
    auto kernel = prefill_sink_attn_kernel<D, kRagged>;
    static std::atomic<bool> configured[kMaxDevices];
    cudaError_t e = once_per_device(configured, [&] {
        cudaFuncAttributes fa;
        cudaError_t err = cudaFuncGetAttributes(&fa, kernel);
        if (err != cudaSuccess) return err;
        // The register split above assumes this launch size; refuse otherwise.
        if (fa.numRegs < C::kRegsLaunch) return cudaErrorInvalidConfiguration;
        return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    });
    if (e != cudaSuccess) return e;
    kernel<<<grid, C::kThreads, C::kSmem, stream>>>(qm, km, vm, om, args);
    return cudaGetLastError();
}

}  // namespace

attn_status launch_prefill(attn_plan_s* plan, const void* q_map, const void* kv_map, const void* v_map,
                           const void* o_map, const float* sinks, void* out, float* lse, cudaStream_t stream) {
    if (plan->items.empty()) return ATTN_OK;
    PrefillArgs a;
    a.items = reinterpret_cast<const PrefillItem*>(plan->ws + plan->layout.items);
    a.item_off = reinterpret_cast<const int32_t*>(plan->ws + plan->layout.item_off);
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
    const CUtensorMap& vm = *static_cast<const CUtensorMap*>(v_map ? v_map : kv_map);
    const CUtensorMap& om = *static_cast<const CUtensorMap*>(o_map);
    // Persistent grid: one CTA per planned item list (at most one per SM; the
    // kernel holds all of an SM's TMEM).
    const int grid = plan->prefill_ctas;
    cudaError_t e;
    if (plan->ragged)
        e = plan->D == 64 ? launch<64, true>(qm, km, vm, om, a, grid, stream)
                          : launch<128, true>(qm, km, vm, om, a, grid, stream);
    else
        e = plan->D == 64 ? launch<64, false>(qm, km, vm, om, a, grid, stream)
                          : launch<128, false>(qm, km, vm, om, a, grid, stream);
    return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace attn
