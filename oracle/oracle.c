/*
 * Oracle: paged GQA attention with a per-head sink logit, in plain fp64 C.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously-correct CPU
 * statement of what the CUDA path computes.  Only the test suite, the smoke
 * check and the benchmark's CPU-baseline leg may load it; the library under
 * paged_kv_attention_sink_gb300/ never links, loads or calls it, and the two
 * share no code (not even the bf16 conversion or the page walk).
 *
 * What it computes (per request b, query row i, query head h):
 *
 *   "GPT-OSS on day 0" (Perplexity), section "Sink Attention": every attention
 *   head carries one pretrained sink parameter that takes part in the softmax,
 *   and the attention is written as softmax(q k^T * sm_scale + sink) V.  With
 *   one scalar per head a literal "+ sink" on every logit would cancel inside
 *   the softmax, so the reading taken here (and by the same section's remark
 *   that the running max is initialised to the sink with scale 1) is that the
 *   sink is one extra logit whose value vector is zero: it appears in the
 *   denominator only.  The sink is in post-scale logit units and is indexed by
 *   the query head.
 *
 *       s_j  = sm_scale * sum_d q[i,h,d] k[j,g,d]          g = h / (Hq/Hkv)
 *       m    = max(max_j s_j, sink_h)
 *       den  = sum_j exp(s_j - m) + exp(sink_h - m)
 *       out  = sum_j exp(s_j - m) v[j,g,:] / den
 *       lse  = m + ln(den)                                  natural log
 *
 *   The same section's max-subtraction form of the softmax is used as is (it
 *   is exact in real arithmetic; here it only keeps exp() in range).
 *
 *   Keys visible to row i: j < kv_len, and with causal masking j <= kv_len -
 *   qo_len + i (query i sits at absolute position kv_len - qo_len + i; this
 *   bottom-right alignment is the reading taken for a cached prefix, on which
 *   the pages are silent).  "Disaggregated prefill and decode" (Perplexity),
 *   section "Prefill vs decode performance", gives the request model:
 *   qo_len tokens go forward, kv_len tokens are read from the KV cache, and a
 *   decode request has qo_len = 1.
 *
 *   KV cache, "Hosting Qwen on Blackwell" (Perplexity), section "Deploying on
 *   GB200 NVL72", and "Disaggregated prefill and decode", section "Sharded KV
 *   transfer": pages in HND order -- heads outermost, the page's tokens
 *   contiguous.  The pool here is [num_pages][2 (K,V)][Hkv][P][D] bf16; the
 *   request's pages are page_table[kv_indptr[b] .. kv_indptr[b+1]) and
 *   kv_len = (n_pages - 1) * P + last_page_len[b] (0 when it has no pages).
 *
 *   Split along the KV length ("GPT-OSS on day 0", section "Sink Attention":
 *   when attention is split into blocks along the sequence, the sink belongs
 *   to the first part only): oracle_sink_attention takes a key window
 *   [kv_lo, kv_hi) and a with_sink switch so that the tests can build split
 *   partial states, and oracle_merge_states combines two (out, lse) states by
 *   the log-sum-exp rule that the split implies (the pages do not print it):
 *       L = max(lse_a, lse_b), w_x = exp(lse_x - L),
 *       out = (w_a out_a + w_b out_b) / (w_a + w_b),  lse = L + ln(w_a + w_b).
 *
 * Precision: inputs are bf16 bit patterns converted exactly to double; every
 * sum, exp and log is fp64 (host libm).  No blocking, no fusion, no reordering
 * beyond the definition above.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* bf16 -> double: a bf16 value is the top 16 bits of an IEEE binary32. */
static double oracle_bf16_value(uint16_t bits) {
    uint32_t word = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &word, sizeof f);
    return (double)f;
}

/* Length of request b's KV sequence from its page count and last-page fill. */
static int64_t oracle_kv_len(const int32_t* kv_indptr, const int32_t* last_page_len,
                             int32_t b, int32_t P) {
    int64_t n_pages = (int64_t)kv_indptr[b + 1] - kv_indptr[b];
    if (n_pages <= 0) return 0;
    return (n_pages - 1) * P + last_page_len[b];
}

/* Address of token j's row (K if kv == 0, V if kv == 1) for kv head g. */
static const uint16_t* oracle_kv_row(const uint16_t* pool, const int32_t* page_table,
                                     int32_t first_page_slot, int64_t j, int kv, int32_t g,
                                     int32_t Hkv, int32_t P, int32_t D) {
    int64_t page = page_table[first_page_slot + j / P];
    int64_t token_in_page = j % P;
    int64_t offset = (((page * 2 + kv) * Hkv + g) * P + token_in_page) * (int64_t)D;
    return pool + offset;
}

/* Request that owns query row `row` (qo_indptr is non-decreasing). */
static int32_t oracle_request_of_row(const int32_t* qo_indptr, int32_t B, int64_t row) {
    int32_t lo = 0, hi = B - 1;
    while (lo < hi) {
        int32_t mid = (lo + hi + 1) / 2;
        if (qo_indptr[mid] <= row) lo = mid; else hi = mid - 1;
    }
    return lo;
}

/* One (row, head) output: writes D values to out_row and one lse. */
static int oracle_one_row(int32_t B, const int32_t* qo_indptr, const int32_t* kv_indptr,
                          const int32_t* page_table, const int32_t* last_page_len,
                          const uint16_t* q, const uint16_t* kv_pool, const float* sinks,
                          int32_t Hq, int32_t Hkv, int32_t D, int32_t P, int32_t causal,
                          double sm_scale, int64_t kv_lo, int64_t kv_hi, int32_t with_sink,
                          int64_t row, int32_t h, double* scores, double* out_row,
                          double* lse_out) {
    int32_t b = oracle_request_of_row(qo_indptr, B, row);
    int64_t qo_len = (int64_t)qo_indptr[b + 1] - qo_indptr[b];
    int64_t i = row - qo_indptr[b];
    int64_t kv_len = oracle_kv_len(kv_indptr, last_page_len, b, P);
    if (qo_len > kv_len) return 2;
    int32_t group = Hq / Hkv;
    int32_t g = h / group;

    /* Last key this row may see (inclusive). */
    int64_t last = kv_len - 1;
    if (causal) {
        int64_t diag = kv_len - qo_len + i;
        if (diag < last) last = diag;
    }
    int64_t first = kv_lo > 0 ? kv_lo : 0;
    if (kv_hi - 1 < last) last = kv_hi - 1;

    const uint16_t* q_row = q + (row * Hq + h) * (int64_t)D;
    double sink = (with_sink && sinks) ? (double)sinks[h] : -INFINITY;

    /* Scores s_j and their maximum, together with the sink. */
    double m = sink;
    for (int64_t j = first; j <= last; ++j) {
        const uint16_t* k_row = oracle_kv_row(kv_pool, page_table, kv_indptr[b], j, 0, g, Hkv, P, D);
        double dot = 0.0;
        for (int32_t d = 0; d < D; ++d) dot += oracle_bf16_value(q_row[d]) * oracle_bf16_value(k_row[d]);
        scores[j - first] = sm_scale * dot;
        if (scores[j - first] > m) m = scores[j - first];
    }

    for (int32_t d = 0; d < D; ++d) out_row[d] = 0.0;
    if (m == -INFINITY) {         /* no visible key and no sink: empty softmax */
        *lse_out = -INFINITY;
        return 0;
    }

    double den = (sink == -INFINITY) ? 0.0 : exp(sink - m);
    for (int64_t j = first; j <= last; ++j) {
        double w = exp(scores[j - first] - m);
        den += w;
        const uint16_t* v_row = oracle_kv_row(kv_pool, page_table, kv_indptr[b], j, 1, g, Hkv, P, D);
        for (int32_t d = 0; d < D; ++d) out_row[d] += w * oracle_bf16_value(v_row[d]);
    }
    for (int32_t d = 0; d < D; ++d) out_row[d] /= den;
    *lse_out = m + log(den);
    return 0;
}

/*
 * Paged sink attention over all (row, head) pairs, or over a selected list.
 *
 *   q        [total_rows][Hq][D] bf16 bits, total_rows = qo_indptr[B]
 *   kv_pool  [num_pages][2][Hkv][P][D] bf16 bits (HND pages)
 *   sinks    [Hq] float, or NULL for no sink (-inf)
 *   kv_lo, kv_hi   key window (use 0 and INT64_MAX for all keys)
 *   with_sink      0 drops the sink term (a split part other than the first)
 *   n_sel < 0: out [total_rows][Hq][D], lse [total_rows][Hq]
 *   n_sel >= 0: only pairs (sel_row[k], sel_head[k]); out [n_sel][D], lse [n_sel]
 *   n_threads: OpenMP threads (0 = runtime default)
 *
 * Returns 0, 1 on a malformed argument, 2 if some request has qo_len > kv_len.
 */
int oracle_sink_attention(int32_t B, const int32_t* qo_indptr, const int32_t* kv_indptr,
                          const int32_t* page_table, const int32_t* last_page_len,
                          const uint16_t* q, const uint16_t* kv_pool, const float* sinks,
                          int32_t Hq, int32_t Hkv, int32_t D, int32_t P, int32_t causal,
                          double sm_scale, int64_t kv_lo, int64_t kv_hi, int32_t with_sink,
                          int64_t n_sel, const int64_t* sel_row, const int32_t* sel_head,
                          int32_t n_threads, double* out, double* lse) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || D <= 0 || P <= 0) return 1;
    int64_t total_rows = B > 0 ? qo_indptr[B] : 0;
    int64_t max_kv = 0;
    for (int32_t b = 0; b < B; ++b) {
        int64_t kv_len = oracle_kv_len(kv_indptr, last_page_len, b, P);
        if (kv_len > max_kv) max_kv = kv_len;
        if ((int64_t)qo_indptr[b + 1] - qo_indptr[b] > kv_len) return 2;
    }
    int64_t n_pairs = n_sel >= 0 ? n_sel : total_rows * Hq;
    int status = 0;
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#else
    (void)n_threads;
#endif
#pragma omp parallel
    {
        double* scores = (double*)malloc(sizeof(double) * (size_t)(max_kv > 0 ? max_kv : 1));
#pragma omp for schedule(dynamic, 16)
        for (int64_t k = 0; k < n_pairs; ++k) {
            int64_t row = n_sel >= 0 ? sel_row[k] : k / Hq;
            int32_t h = n_sel >= 0 ? sel_head[k] : (int32_t)(k % Hq);
            int rc = 1;
            if (row >= 0 && row < total_rows && h >= 0 && h < Hq && scores) {
                rc = oracle_one_row(B, qo_indptr, kv_indptr, page_table, last_page_len, q,
                                    kv_pool, sinks, Hq, Hkv, D, P, causal, sm_scale, kv_lo,
                                    kv_hi, with_sink, row, h, scores, out + k * (int64_t)D,
                                    lse + k);
            }
            if (rc) {
#pragma omp critical
                status = rc;
            }
        }
        free(scores);
    }
    return status;
}

/*
 * Merge two attention states over disjoint key sets into the state over their
 * union (log-sum-exp rule; see the header comment).  va, vb, vout: [n][D];
 * lsea, lseb, lseout: [n], natural log.
 */
void oracle_merge_states(int64_t n, int32_t D, const double* va, const double* lsea,
                         const double* vb, const double* lseb, double* vout, double* lseout) {
    for (int64_t r = 0; r < n; ++r) {
        double L = lsea[r] > lseb[r] ? lsea[r] : lseb[r];
        if (L == -INFINITY) {
            for (int32_t d = 0; d < D; ++d) vout[r * D + d] = 0.0;
            lseout[r] = -INFINITY;
            continue;
        }
        double wa = exp(lsea[r] - L), wb = exp(lseb[r] - L);
        for (int32_t d = 0; d < D; ++d)
            vout[r * D + d] = (wa * va[r * D + d] + wb * vb[r * D + d]) / (wa + wb);
        lseout[r] = L + log(wa + wb);
    }
}

/*
 * KV append.  "Disaggregated prefill and decode" (Perplexity), section "KV
 * Messenger": a layer's page copies start as soon as the model has finished
 * appending the step's tokens to that layer's KV cache, and the cache entries
 * are valid after the append and before attention.  The pages give no
 * indexing; the reading taken here is that the qo_len tokens request b
 * forwards are its newest cache positions, t = kv_len - qo_len + i for its
 * i-th row (the same alignment as the causal mask), so row r = qo_indptr[b] + i
 * of k_new / v_new ([rows][Hkv][D] bf16) goes to pool[page][0 / 1][g][t % P][:]
 * with page = page_table[kv_indptr[b] + t / P].  Pure data movement: the bit
 * patterns are copied unchanged.  A row whose page id lies outside
 * [0, num_pages) is skipped and the return value is 1 (else 0).
 */
int oracle_append_kv(int32_t B, const int32_t* qo_indptr, const int32_t* kv_indptr,
                     const int32_t* page_table, const int32_t* last_page_len, int32_t Hkv,
                     int32_t D, int32_t P, int64_t num_pages, const uint16_t* k_new,
                     const uint16_t* v_new, uint16_t* pool) {
    int status = 0;
    for (int32_t b = 0; b < B; ++b) {
        int64_t kv_len = oracle_kv_len(kv_indptr, last_page_len, b, P);
        int64_t qo_len = (int64_t)qo_indptr[b + 1] - qo_indptr[b];
        for (int64_t i = 0; i < qo_len; ++i) {
            int64_t t = kv_len - qo_len + i;
            int64_t page = page_table[kv_indptr[b] + t / P];
            if (page < 0 || page >= num_pages) {
                status = 1;
                continue;
            }
            int64_t r = qo_indptr[b] + i;
            for (int32_t g = 0; g < Hkv; ++g) {
                for (int kv = 0; kv < 2; ++kv) {
                    const uint16_t* src = (kv == 0 ? k_new : v_new) + (r * Hkv + g) * (int64_t)D;
                    uint16_t* dst = pool + (((page * 2 + kv) * Hkv + g) * P + t % P) * (int64_t)D;
                    for (int32_t d = 0; d < D; ++d) dst[d] = src[d];
                }
            }
        }
    }
    return status;
}

/*
 * Head-slice pack and unpack of HND pages.  "Disaggregated prefill and
 * decode", section "Sharded KV transfer": when the sending and receiving
 * sides shard the KV cache over attention heads differently, pages are split
 * or rebuilt from head slices, and the HND layout (heads before tokens) keeps
 * a page's slice of heads contiguous so that it moves as one write.  Pack
 * copies heads [h0, h0 + nh) of pages page_ids[0 .. n) out of the pool into
 * buf[n][2][nh][P][D]; unpack writes such a buffer back into those heads of
 * those pages.  Pages outside [0, num_pages) are skipped; the return value is
 * then 1 (else 0).
 */
int oracle_pack_heads(const uint16_t* pool, int64_t num_pages, int32_t Hkv, int32_t P, int32_t D,
                      const int32_t* page_ids, int64_t n, int32_t h0, int32_t nh, uint16_t* buf) {
    int status = 0;
    for (int64_t i = 0; i < n; ++i) {
        int64_t page = page_ids[i];
        if (page < 0 || page >= num_pages) {
            status = 1;
            continue;
        }
        for (int kv = 0; kv < 2; ++kv)
            for (int32_t h = 0; h < nh; ++h)
                for (int32_t p = 0; p < P; ++p)
                    for (int32_t d = 0; d < D; ++d)
                        buf[(((i * 2 + kv) * nh + h) * P + p) * (int64_t)D + d] =
                            pool[(((page * 2 + kv) * Hkv + h0 + h) * P + p) * (int64_t)D + d];
    }
    return status;
}

int oracle_unpack_heads(const uint16_t* buf, int64_t num_pages, int32_t Hkv, int32_t P, int32_t D,
                        const int32_t* page_ids, int64_t n, int32_t h0, int32_t nh, uint16_t* pool) {
    int status = 0;
    for (int64_t i = 0; i < n; ++i) {
        int64_t page = page_ids[i];
        if (page < 0 || page >= num_pages) {
            status = 1;
            continue;
        }
        for (int kv = 0; kv < 2; ++kv)
            for (int32_t h = 0; h < nh; ++h)
                for (int32_t p = 0; p < P; ++p)
                    for (int32_t d = 0; d < D; ++d)
                        pool[(((page * 2 + kv) * Hkv + h0 + h) * P + p) * (int64_t)D + d] =
                            buf[(((i * 2 + kv) * nh + h) * P + p) * (int64_t)D + d];
    }
    return status;
}
