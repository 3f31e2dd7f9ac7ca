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
    static constexpr int kStages = (D == 64) ? 4 : 3;       // per warp
    static constexpr int kSubTile = kBlockTokens * 128;       // 16 rows x 128 B (64 dims)
    static constexpr int kTileBytes = kBlockTokens * D * 2;   // K or V of one block
    static constexpr int kStageBytes = 2 * kTileBytes;
    static constexpr int kPipeBytes = kWarps * kStages * kStageBytes;
    static constexpr int kPageBytes = (kDecodeMaxChunkPages * 4 + 15) / 16 * 16;
    static constexpr int kBarBytes = kWarps * kStages * 8;
    static constexpr int kStateBytes = kWarps * 48 * 4 + 16;  // per-warp m, l, le + flag
    static constexpr int kSmem = 1024 + kPipeBytes + kPageBytes + kBarBytes + kStateBytes;
    static constexpr int kRowStride = D + 8;                  // floats, combine buffers
    static_assert(kBlockTokens * kRowStride * 4 <= kStages * kStageBytes, "combine fits");
};

struct DecodeArgs {
    const DecodeUnit* units;
    const int32_t* page_table;
    const __nv_bfloat16* q;
    __nv_bfloat16* out;
    float* lse;
    const float* sinks;
    float* part_o;
    float* part_lse;
    int32_t* counters;
    int32_t* err;
    int32_t Hq, Hkv, P, num_pages;
    float scale_log2;   // sm_scale * log2(e)
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

template <int D, bool kTwoRows>
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
    const DecodeUnit u = a.units[blockIdx.x];
    const int P = a.P;
    const int first_page = u.tok_begin / P;
    const int n_pages = (u.tok_end - 1) / P - first_page + 1;

    for (int i = tid; i < n_pages; i += blockDim.x)
        pages_s[i] = a.page_table[u.page_base + first_page + i];
    if (lane == 0)
        for (int s = 0; s < C::kStages; ++s) ptx::mbar_init(ptx::smem_u32(&bars[warp * C::kStages + s]), 1);
    if (tid == 0) ptx::prefetch_tmap(&kv_map);
    ptx::fence_mbar_init();
    __syncthreads();

    const int nblk = (u.tok_end - u.tok_begin + kBlockTokens - 1) / kBlockTokens;
    const int n_it = nblk > warp ? (nblk - warp + C::kWarps - 1) / C::kWarps : 0;
    const uint32_t stage0 = ptx::smem_u32(pipe) + warp * C::kStages * C::kStageBytes;
    const uint32_t bar0 = ptx::smem_u32(&bars[warp * C::kStages]);
    const uint64_t policy = ptx::policy_evict_first();

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
        for (int it = 0; it < C::kStages && it < n_it; ++it) issue(warp + it * C::kWarps, it);

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
        const int s = it % C::kStages;
        if (!ptx::mbar_wait(bar0 + s * 8, (it / C::kStages) & 1)) { timed_out = true; break; }
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
        if (lane == 0) atomicOr(a.err, ATTN_DEVICE_ERR_TIMEOUT);
        for (int j = it; j < n_it && j < it + C::kStages; ++j)   // drain loads still in flight
            ptx::mbar_wait(bar0 + (j % C::kStages) * 8, (j / C::kStages) & 1);
    }

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
    if (u.n_chunks == 1) return;

    // Split sequence: the last chunk to finish merges all chunks (no waiting).
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        const int prev = atomicAdd(&a.counters[u.group], 1);
        *flag_s = (prev == u.n_chunks - 1);
    }
    __syncthreads();
    if (!*flag_s) return;
    __threadfence();
    for (int idx = tid; idx < items; idx += blockDim.x) {
        const int r = idx / (D / 4), d = (idx % (D / 4)) * 4;
        float Lm = -INFINITY;
        for (int c = 0; c < u.n_chunks; ++c)
            Lm = fmaxf(Lm, __ldcg(a.part_lse + (size_t)(u.partial0 + c) * kMaxSliceHeads + r));
        float W = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int c = 0; c < u.n_chunks; ++c) {
            const size_t slot = (size_t)(u.partial0 + c) * kMaxSliceHeads + r;
            const float lc = __ldcg(a.part_lse + slot);
            const float w = (lc == -INFINITY) ? 0.f : ptx::ex2(lc - Lm);
            const float4 oc = __ldcg(reinterpret_cast<const float4*>(a.part_o + slot * D + d));
            W += w;
            acc.x += w * oc.x; acc.y += w * oc.y; acc.z += w * oc.z; acc.w += w * oc.w;
        }
        const float inv = W > 0.f ? 1.f / W : 0.f;
        store_bf16x4(a.out + ((size_t)u.q_row * a.Hq + u.head0 + r) * D + d, acc.x * inv,
                     acc.y * inv, acc.z * inv, acc.w * inv);
        if (d == 0 && a.lse)
            a.lse[(size_t)u.q_row * a.Hq + u.head0 + r] = (W > 0.f ? Lm + log2f(W) : -INFINITY) * kLn2;
    }
    if (tid == 0) a.counters[u.group] = 0;   // ready for the next launch
}

template <int D, bool kTwoRows>
cudaError_t launch(const CUtensorMap& map, const DecodeArgs& args, int n_units, cudaStream_t stream) {
    using C = DecodeCfg<D>;
    auto kernel = decode_sink_attn_kernel<D, kTwoRows>;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    kernel<<<n_units, C::kWarps * 32, C::kSmem, stream>>>(map, args);
    return cudaGetLastError();
}

}  // namespace

int decode_ctas_per_sm(int head_dim) {
    constexpr int kSmemPerSm = 233472;   // 228 KB; 1 KB of it is reserved per CTA
    const int per_cta = (head_dim == 64 ? DecodeCfg<64>::kSmem : DecodeCfg<128>::kSmem) + 1024;
    return kSmemPerSm / per_cta;
}

attn_status launch_decode(attn_plan_s* plan, const void* q, const void* kv_map, const float* sinks,
                          void* out, float* lse, cudaStream_t stream) {
    if (plan->units.empty()) return ATTN_OK;
    DecodeArgs a;
    a.units = reinterpret_cast<const DecodeUnit*>(plan->ws + plan->layout.units);
    a.page_table = plan->page_table;
    a.q = static_cast<const __nv_bfloat16*>(q);
    a.out = static_cast<__nv_bfloat16*>(out);
    a.lse = lse;
    a.sinks = sinks;
    a.part_o = reinterpret_cast<float*>(plan->ws + plan->layout.part_o);
    a.part_lse = reinterpret_cast<float*>(plan->ws + plan->layout.part_lse);
    a.counters = reinterpret_cast<int32_t*>(plan->ws + plan->layout.counters);
    a.err = reinterpret_cast<int32_t*>(plan->ws + plan->layout.err);
    a.Hq = plan->Hq;
    a.Hkv = plan->Hkv;
    a.P = plan->P;
    a.num_pages = plan->num_pages;
    a.scale_log2 = plan->sm_scale * kLog2e;
    const CUtensorMap& map = *static_cast<const CUtensorMap*>(kv_map);
    const bool two_rows = plan->Hq / plan->Hkv > 8;
    const int n = (int)plan->units.size();
    cudaError_t e;
    if (plan->D == 64)
        e = two_rows ? launch<64, true>(map, a, n, stream) : launch<64, false>(map, a, n, stream);
    else
        e = two_rows ? launch<128, true>(map, a, n, stream) : launch<128, false>(map, a, n, stream);
    return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace attn

namespace attn {

attn_status launch_decode_scratch(attn_plan_s* plan, unsigned char* scratch, const void* q,
                                  const void* kv_map, const float* sinks, void* out, float* lse,
                                  cudaStream_t stream) {
    if (plan->units.empty()) return ATTN_OK;
    DecodeArgs a;
    a.units = reinterpret_cast<const DecodeUnit*>(scratch + plan->layout.units);
    a.page_table = plan->page_table;
    a.q = static_cast<const __nv_bfloat16*>(q);
    a.out = static_cast<__nv_bfloat16*>(out);
    a.lse = lse;
    a.sinks = sinks;
    a.part_o = reinterpret_cast<float*>(scratch + plan->layout.part_o);
    a.part_lse = reinterpret_cast<float*>(scratch + plan->layout.part_lse);
    a.counters = reinterpret_cast<int32_t*>(scratch + plan->layout.counters);
    a.err = reinterpret_cast<int32_t*>(scratch + plan->layout.err);
    a.Hq = plan->Hq;
    a.Hkv = plan->Hkv;
    a.P = plan->P;
    a.num_pages = plan->num_pages;
    a.scale_log2 = plan->sm_scale * kLog2e;
    const CUtensorMap& map = *static_cast<const CUtensorMap*>(kv_map);
    const bool two_rows = plan->Hq / plan->Hkv > 8;
    const int n = (int)plan->units.size();
    cudaError_t e;
    if (plan->D == 64)
        e = two_rows ? launch<64, true>(map, a, n, stream) : launch<64, false>(map, a, n, stream);
    else
        e = two_rows ? launch<128, true>(map, a, n, stream) : launch<128, false>(map, a, n, stream);
    return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace attn
