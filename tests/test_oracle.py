"""Pins for the fp64 oracle: each test checks it against something other than
itself -- a library routine for a special case, a closed form, an invariant, or
brute force in 50-digit decimal arithmetic.  CPU only.

The definition being pinned is the sink attention of "GPT-OSS on day 0"
(Perplexity), section "Sink Attention": one sink logit per query head that sits
in the softmax denominator only, over a paged HND KV cache ("Hosting Qwen on
Blackwell", section "Deploying on GB200 NVL72").
"""
import decimal
import math

import numpy as np
import pytest
import torch

import oracle
from paged_kv_attention_sink_gb300 import synthetic as syn


def _dense_kv(batch, b):
    """Gather request b's K and V into dense [kv_len, Hkv, D] float64 arrays by
    plain numpy fancy indexing (a second, independent page walk)."""
    P = batch.page_size
    pages = batch.page_table[batch.kv_indptr[b]:batch.kv_indptr[b + 1]]
    kv_len = int(batch.kv_lens[b])
    blk = batch.kv_pool[pages]                      # [n_pages, 2, Hkv, P, D]
    blk = np.transpose(blk, (1, 0, 3, 2, 4))        # [2, n_pages, P, Hkv, D]
    blk = blk.reshape(2, -1, batch.num_kv_heads, batch.head_dim)[:, :kv_len]
    f = syn.bf16_to_float(blk).astype(np.float64)
    return f[0], f[1]


def _small_batch(seed, qo, kv, Hq=4, Hkv=2, D=16, P=4, sinks=True, causal=True, pool=None):
    return syn.make_batch("t", qo, kv, Hq, Hkv, D, P, causal=causal, with_sinks=sinks,
                          pool_pages=pool, seed=seed)


@pytest.mark.parametrize("causal", [True, False])
def test_no_sink_equals_library_attention(causal):
    """sink = -inf: the oracle must equal torch's scaled_dot_product_attention
    (fp64, explicit mask, GQA by repeating KV heads) and torch.logsumexp."""
    batch = _small_batch(1, [1, 5, 3, 7], [9, 5, 12, 7], Hq=6, Hkv=2, sinks=False,
                         causal=causal)
    out, lse = oracle.sink_attention(batch)
    G = batch.num_qo_heads // batch.num_kv_heads
    for b in range(batch.batch_size):
        k, v = _dense_kv(batch, b)
        r0, r1 = batch.qo_indptr[b], batch.qo_indptr[b + 1]
        qo_len, kv_len = r1 - r0, int(batch.kv_lens[b])
        q = torch.from_numpy(syn.bf16_to_float(batch.q[r0:r1]).astype(np.float64))
        qh = q.permute(1, 0, 2)                                   # [Hq, qo, D]
        kh = torch.from_numpy(k).permute(1, 0, 2).repeat_interleave(G, 0)
        vh = torch.from_numpy(v).permute(1, 0, 2).repeat_interleave(G, 0)
        i = torch.arange(qo_len)[:, None]
        j = torch.arange(kv_len)[None, :]
        allowed = (j <= kv_len - qo_len + i) if causal else torch.ones(qo_len, kv_len, dtype=bool)
        ref = torch.nn.functional.scaled_dot_product_attention(
            qh, kh, vh, attn_mask=allowed, scale=batch.sm_scale)
        scores = torch.einsum("hqd,hkd->hqk", qh, kh) * batch.sm_scale
        ref_lse = torch.logsumexp(scores.masked_fill(~allowed, -math.inf), dim=-1)
        np.testing.assert_allclose(out[r0:r1], ref.permute(1, 0, 2).numpy(), rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[r0:r1], ref_lse.T.numpy(), rtol=0, atol=1e-12)


def test_sink_as_extra_zero_value_column_library():
    """With a sink, the oracle must equal torch.softmax over the scores with one
    extra column holding the sink, whose value row is zero (fp64)."""
    batch = _small_batch(2, [3, 1, 4], [6, 9, 4], Hq=4, Hkv=1, D=8, P=2)
    out, lse = oracle.sink_attention(batch)
    G = batch.num_qo_heads
    for b in range(batch.batch_size):
        k, v = _dense_kv(batch, b)
        r0, r1 = batch.qo_indptr[b], batch.qo_indptr[b + 1]
        qo_len, kv_len = r1 - r0, int(batch.kv_lens[b])
        q = torch.from_numpy(syn.bf16_to_float(batch.q[r0:r1]).astype(np.float64))
        scores = torch.einsum("qhd,kd->hqk", q, torch.from_numpy(k[:, 0])) * batch.sm_scale
        i = torch.arange(qo_len)[:, None]
        j = torch.arange(kv_len)[None, :]
        scores = scores.masked_fill(~(j <= kv_len - qo_len + i), -math.inf)
        sink_col = torch.from_numpy(batch.sinks.astype(np.float64))[:, None, None].expand(G, qo_len, 1)
        logits = torch.cat([scores, sink_col], dim=-1)
        p = torch.softmax(logits, dim=-1)
        v_ext = torch.cat([torch.from_numpy(v[:, 0]), torch.zeros(1, batch.head_dim, dtype=torch.float64)])
        ref = torch.einsum("hqk,kd->qhd", p, v_ext)
        np.testing.assert_allclose(out[r0:r1], ref.numpy(), rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[r0:r1], torch.logsumexp(logits, -1).T.numpy(), rtol=0, atol=1e-12)


def test_huge_sink_drives_output_to_zero():
    """sink = 80 dwarfs every score: out -> 0 and lse -> sink."""
    batch = _small_batch(3, [1, 4], [40, 17], Hq=4, Hkv=2, D=16)
    sinks = np.full(batch.num_qo_heads, 80.0, dtype=np.float32)
    out, lse = oracle.sink_attention(batch, sinks=sinks)
    assert np.abs(out).max() < 1e-25
    np.testing.assert_allclose(lse, 80.0, rtol=0, atol=1e-20)
    assert np.all(lse >= 80.0)


def _constant_qk_batch(seed, qo, kv, sinks, D=64):
    """q = 1 and k = 0.5 everywhere (bf16-exact), so every score is exactly
    sm_scale * D * 0.5 = 4 with sm_scale = 1/8 (D = 64)."""
    batch = _small_batch(seed, qo, kv, Hq=2, Hkv=1, D=D, P=8)
    batch.q[:] = syn.bf16_bits(np.ones(1, np.float32))[0]
    pool = batch.kv_pool
    valid = pool[:, 0] != syn.BF16_NAN
    pool[:, 0][valid] = syn.bf16_bits(np.full(1, 0.5, np.float32))[0]
    batch.sinks = np.asarray(sinks, dtype=np.float32)
    return batch


def test_identical_keys_closed_form():
    """All scores equal s: out = mean(V_visible) * n / (n + exp(sink - s)),
    lse = s + ln(n + exp(sink - s)), n = number of visible keys."""
    sinks = [0.75, -2.0]
    batch = _constant_qk_batch(4, [1, 6, 3], [33, 6, 20], sinks)
    out, lse = oracle.sink_attention(batch)
    s = 4.0
    for b in range(batch.batch_size):
        _, v = _dense_kv(batch, b)
        r0, r1 = batch.qo_indptr[b], batch.qo_indptr[b + 1]
        qo_len, kv_len = r1 - r0, int(batch.kv_lens[b])
        for i in range(qo_len):
            n = kv_len - qo_len + i + 1
            for h in range(2):
                scale = n / (n + math.exp(sinks[h] - s))
                np.testing.assert_allclose(out[r0 + i, h], v[:n, 0].mean(0) * scale, rtol=0, atol=1e-13)
                np.testing.assert_allclose(lse[r0 + i, h], s + math.log(n + math.exp(sinks[h] - s)),
                                           rtol=0, atol=1e-13)


def test_one_key_closed_form():
    """One key, D = 1: out = v * sigmoid(s - sink), lse = logaddexp(s, sink)."""
    batch = syn.make_batch("one", [1], [1], 1, 1, 1, 1, pool_pages=3, seed=5)
    batch.q[0, 0, 0] = syn.bf16_bits(np.array([2.0], np.float32))[0]
    batch.kv_pool[batch.page_table[0], 0, 0, 0, 0] = syn.bf16_bits(np.array([0.75], np.float32))[0]
    batch.kv_pool[batch.page_table[0], 1, 0, 0, 0] = syn.bf16_bits(np.array([-3.5], np.float32))[0]
    for sink in (0.7, -1.25, 3.0):
        out, lse = oracle.sink_attention(batch, sm_scale=1.0, sinks=np.array([sink], np.float32))
        s = 1.5
        sink64 = float(np.float32(sink))
        assert out[0, 0, 0] == pytest.approx(-3.5 / (1.0 + math.exp(sink64 - s)), abs=1e-15)
        assert lse[0, 0] == pytest.approx(np.logaddexp(s, sink64), abs=1e-15)


def test_page_permutation_invariance():
    """Moving pages to other pool slots (and the page table with them) must not
    change a single bit of the result."""
    batch = _small_batch(6, [2, 5, 1], [23, 11, 30], Hq=4, Hkv=2, D=8, P=4, pool=40)
    out_a, lse_a = oracle.sink_attention(batch)
    rng = np.random.default_rng(0)
    perm = rng.permutation(batch.num_pages)           # new slot of old page p = perm[p]
    new_pool = np.empty_like(batch.kv_pool)
    new_pool[perm] = batch.kv_pool
    batch.kv_pool = new_pool
    batch.page_table = perm[batch.page_table].astype(np.int32)
    out_b, lse_b = oracle.sink_attention(batch)
    assert np.array_equal(out_a, out_b) and np.array_equal(lse_a, lse_b)


@pytest.mark.parametrize("sink_part", [0, 1, 2])
def test_split_kv_merge_equals_unsplit(sink_part):
    """Splitting the keys into windows, giving the sink to exactly one window
    and merging the partial states must reproduce the unsplit result."""
    batch = _small_batch(7, [1, 3, 8, 1], [50, 19, 8, 3], Hq=4, Hkv=2, D=16, P=4)
    ref_out, ref_lse = oracle.sink_attention(batch)
    cuts = [0, 7, 21, 2**62]
    parts = [oracle.sink_attention(batch, kv_lo=cuts[c], kv_hi=cuts[c + 1], with_sink=(c == sink_part))
             for c in range(3)]
    out, lse = parts[0]
    for o, l in parts[1:]:
        out, lse = oracle.merge_states(out, lse, o, l)
    np.testing.assert_allclose(out, ref_out, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, rtol=0, atol=1e-12)


def test_merge_with_empty_state():
    """A state over no keys (lse = -inf) is the identity of the merge."""
    rng = np.random.default_rng(1)
    va = rng.standard_normal((5, 8))
    lsea = rng.standard_normal(5)
    vb = np.zeros((5, 8))
    lseb = np.full(5, -np.inf)
    vo, lo = oracle.merge_states(va, lsea, vb, lseb)
    np.testing.assert_array_equal(vo, va)
    np.testing.assert_array_equal(lo, lsea)
    vo, lo = oracle.merge_states(vb, lseb, vb, lseb)
    assert np.all(vo == 0) and np.all(lo == -np.inf)


def test_gqa_equals_repeated_heads():
    """Hkv = Hq with each KV head repeated G times equals the grouped result."""
    G = 3
    batch = _small_batch(8, [2, 1, 4], [9, 14, 6], Hq=6, Hkv=2, D=8, P=4)
    out_g, lse_g = oracle.sink_attention(batch)
    rep = syn.Batch(**{**batch.__dict__})
    rep.num_kv_heads = batch.num_qo_heads
    rep.kv_pool = np.repeat(batch.kv_pool, G, axis=2)
    out_r, lse_r = oracle.sink_attention(rep)
    np.testing.assert_array_equal(out_g, out_r)
    np.testing.assert_array_equal(lse_g, lse_r)


def test_score_shift_invariance():
    """Adding the same constant c to every score and to the sink leaves the
    output unchanged and adds c to lse; c = 1024 overflows a naive exp."""
    batch = _small_batch(9, [3, 1], [12, 26], Hq=2, Hkv=1, D=4, P=4)
    batch.q[..., 3] = 0
    batch.sinks = (np.round(batch.sinks * 64) / 64).astype(np.float32)   # so sink + c is exact
    out0, lse0 = oracle.sink_attention(batch)
    for t in (8.0, 2048.0):
        shifted = syn.Batch(**{**batch.__dict__})
        shifted.q = batch.q.copy()
        shifted.kv_pool = batch.kv_pool.copy()
        shifted.q[..., 3] = syn.bf16_bits(np.ones(1, np.float32))[0]
        keys = shifted.kv_pool[:, 0, :, :, 3]
        keys[keys != syn.BF16_NAN] = syn.bf16_bits(np.array([t], np.float32))[0]
        c = t * batch.sm_scale
        shifted.sinks = (batch.sinks.astype(np.float64) + c).astype(np.float32)
        assert np.all(shifted.sinks.astype(np.float64) - batch.sinks == c)   # exact shift
        out1, lse1 = oracle.sink_attention(shifted)
        np.testing.assert_allclose(out1, out0, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse1 - c, lse0, rtol=0, atol=1e-12)


def _decimal_reference(batch, row, h):
    """Brute force in 50-digit decimal arithmetic: softmax over the visible
    scores plus one sink column whose value vector is zero."""
    ctx = decimal.Context(prec=50)
    b = int(np.searchsorted(batch.qo_indptr, row, side="right") - 1)
    qo_len = int(batch.qo_lens[b])
    kv_len = int(batch.kv_lens[b])
    i = row - int(batch.qo_indptr[b])
    g = h // (batch.num_qo_heads // batch.num_kv_heads)
    k, v = _dense_kv(batch, b)
    q = syn.bf16_to_float(batch.q[row, h]).astype(np.float64)
    scale = decimal.Decimal(batch.sm_scale)
    last = kv_len - 1 if not batch.causal else min(kv_len - 1, kv_len - qo_len + i)
    weights, values = [], []
    for j in range(last + 1):
        dot = sum((decimal.Decimal(float(q[d])) * decimal.Decimal(float(k[j, g, d])) for d in range(len(q))),
                  decimal.Decimal(0))
        weights.append(ctx.exp(ctx.multiply(dot, scale)))
        values.append([decimal.Decimal(float(x)) for x in v[j, g]])
    if batch.sinks is not None:
        weights.append(ctx.exp(decimal.Decimal(float(batch.sinks[h]))))
        values.append([decimal.Decimal(0)] * len(q))
    den = sum(weights, decimal.Decimal(0))
    out = [float(sum((w * vv[d] for w, vv in zip(weights, values)), decimal.Decimal(0)) / den)
           for d in range(len(q))]
    return np.array(out), float(ctx.ln(den))


@pytest.mark.parametrize("seed", range(4))
def test_brute_force_decimal(seed):
    rng = np.random.default_rng(100 + seed)
    B = int(rng.integers(1, 4))
    kv = rng.integers(1, 6, size=B)
    qo = np.array([int(rng.integers(1, k + 1)) for k in kv])
    D = int(rng.integers(1, 5))
    P = int(rng.integers(1, 4))
    causal = bool(seed % 2 == 0)
    batch = _small_batch(seed, qo, kv, Hq=4, Hkv=2, D=D, P=P, sinks=(seed != 3), causal=causal)
    out, lse = oracle.sink_attention(batch)
    for row in range(batch.total_rows):
        for h in range(batch.num_qo_heads):
            ref_out, ref_lse = _decimal_reference(batch, row, h)
            np.testing.assert_allclose(out[row, h], ref_out, rtol=0, atol=1e-13)
            assert lse[row, h] == pytest.approx(ref_lse, abs=1e-13)


def test_selected_pairs_match_full():
    batch = _small_batch(10, [4, 1], [10, 21], Hq=4, Hkv=2, D=8, P=4)
    out, lse = oracle.sink_attention(batch)
    rows = np.array([0, 3, 4, 2])
    heads = np.array([1, 0, 3, 2])
    so, sl = oracle.sink_attention(batch, rows=rows, heads=heads)
    np.testing.assert_array_equal(so, out[rows, heads])
    np.testing.assert_array_equal(sl, lse[rows, heads])


def test_rejects_qo_longer_than_kv():
    batch = _small_batch(11, [1], [3])
    batch.qo_lens = np.array([5])
    batch.qo_indptr = np.array([0, 5], dtype=np.int32)
    batch.q = np.zeros((5, batch.num_qo_heads, batch.head_dim), dtype=np.uint16)
    with pytest.raises(ValueError):
        oracle.sink_attention(batch)


def test_request_without_queries_or_keys():
    """A request with qo_len = 0 (and even kv_len = 0) contributes no rows and
    does not disturb its neighbours."""
    a = _small_batch(12, [2, 0, 3], [5, 0, 7], Hq=2, Hkv=1, D=4, P=2)
    out, lse = oracle.sink_attention(a)
    assert out.shape[0] == 5 and np.all(np.isfinite(out)) and np.all(np.isfinite(lse))


# ---------------------------------------------------------------- KV append
# "Disaggregated prefill and decode", section "KV Messenger": the step's new
# tokens are appended to the KV cache before attention; the i-th forwarded row
# of a request is its cache position kv_len - qo_len + i.

def _literal_append_batch():
    """Hand-made batch: P = 4, Hkv = 2, D = 2, 4 pages.  Request 0 owns pages
    [3, 1] with 2 tokens on the last page (kv_len 6) and forwards 2 rows;
    request 1 owns page [0] with 3 tokens (kv_len 3) and forwards 1 row."""
    sentinel = np.uint16(0xAAAA)
    pool = np.full((4, 2, 2, 4, 2), sentinel, dtype=np.uint16)
    return syn.Batch(name="literal", num_qo_heads=2, num_kv_heads=2, head_dim=2, page_size=4, causal=True,
                     sm_scale=1.0, qo_lens=np.array([2, 1]), kv_lens=np.array([6, 3]),
                     qo_indptr=np.array([0, 2, 3], dtype=np.int32), kv_indptr=np.array([0, 2, 3], dtype=np.int32),
                     page_table=np.array([3, 1, 0], dtype=np.int32), last_page_len=np.array([2, 3], dtype=np.int32),
                     q=np.zeros((3, 2, 2), dtype=np.uint16), kv_pool=pool, sinks=None)


def test_append_literal_positions():
    b = _literal_append_batch()
    k = np.array([[[100 * r + 10 * g + d for d in range(2)] for g in range(2)] for r in range(3)], dtype=np.uint16)
    v = k + np.uint16(5000)
    pool, rc = oracle.append_kv(b, k, v)
    assert rc == 0
    expected = b.kv_pool.copy()
    # (row r, its page, row in page), listed by hand from the layout above:
    # request 0 rows 0, 1 -> positions 4, 5 -> second page (id 1), rows 0, 1;
    # request 1 row 2 -> position 2 -> page 0, row 2.
    for r, page, slot in ((0, 1, 0), (1, 1, 1), (2, 0, 2)):
        expected[page, 0, :, slot, :] = k[r]
        expected[page, 1, :, slot, :] = v[r]
    np.testing.assert_array_equal(pool, expected)
    assert b.kv_pool[0, 0, 0, 0, 0] == 0xAAAA          # the input pool is untouched


def test_append_then_attention_sees_new_rows_in_order():
    """A fresh prefill (qo_len == kv_len): after the append, the oracle's
    attention over the cache equals brute-force causal sink attention computed
    directly on the new rows -- ties the append's positions to the page walk."""
    batch = syn.make_batch("fresh", [5, 9], [5, 9], 4, 2, 8, 4, seed=21)
    k_new, v_new = syn.new_kv_rows(batch, seed=3)
    pool, rc = oracle.append_kv(batch, k_new, v_new)
    assert rc == 0
    batch.kv_pool = pool
    out, lse = oracle.sink_attention(batch)
    q = syn.bf16_to_float(batch.q).astype(np.float64)
    kf = syn.bf16_to_float(k_new).astype(np.float64)
    vf = syn.bf16_to_float(v_new).astype(np.float64)
    G = batch.num_qo_heads // batch.num_kv_heads
    for b in range(2):
        r0, n = int(batch.qo_indptr[b]), int(batch.qo_lens[b])
        for i in range(n):
            for h in range(batch.num_qo_heads):
                s = kf[r0:r0 + i + 1, h // G] @ q[r0 + i, h] * batch.sm_scale
                w = np.exp(np.append(s, batch.sinks[h]) - max(s.max(), batch.sinks[h]))
                ref = (w[:-1, None] * vf[r0:r0 + i + 1, h // G]).sum(0) / w.sum()
                np.testing.assert_allclose(out[r0 + i, h], ref, rtol=1e-12, atol=1e-12)


def test_append_bad_page_is_skipped():
    b = _literal_append_batch()
    b.page_table = np.array([3, 7, 0], dtype=np.int32)      # page 7 is outside the 4-page pool
    k = np.ones((3, 2, 2), dtype=np.uint16)
    pool, rc = oracle.append_kv(b, k, k)
    assert rc == 1
    assert np.all(pool[0, :, :, 2, :] == 1)                  # request 1's row still lands
    assert np.count_nonzero(pool != 0xAAAA) == 2 * 2 * 2     # and nothing else changed


# ------------------------------------------------------ head-slice pack / unpack
# "Disaggregated prefill and decode", section "Sharded KV transfer": HND keeps
# a page's head slice contiguous, so head-sharded pages are split and rebuilt
# from such slices.

def test_pack_literal():
    pool = np.arange(3 * 2 * 3 * 2 * 2, dtype=np.uint16).reshape(3, 2, 3, 2, 2)   # [pages, K/V, Hkv=3, P=2, D=2]
    buf, rc = oracle.pack_heads(pool, [2, 0], 1, 2)
    assert rc == 0
    # buf[i, kv, h, p, d] = pool[page_i, kv, 1 + h, p, d], written out for page 2 then page 0
    expected = np.stack([np.stack([pool[2, kv, 1:3] for kv in range(2)]),
                         np.stack([pool[0, kv, 1:3] for kv in range(2)])])
    np.testing.assert_array_equal(buf, expected)


def test_pack_all_heads_is_a_page_gather():
    rng = np.random.default_rng(5)
    pool = rng.integers(0, 65535, size=(9, 2, 4, 16, 8), dtype=np.uint16)
    ids = np.array([7, 2, 2, 0, 8], dtype=np.int32)
    buf, rc = oracle.pack_heads(pool, ids, 0, 4)
    assert rc == 0
    np.testing.assert_array_equal(buf, pool[ids])


def test_unpack_inverts_pack_and_touches_only_the_slice():
    rng = np.random.default_rng(6)
    pool = rng.integers(0, 65535, size=(6, 2, 4, 4, 8), dtype=np.uint16)
    ids = np.array([5, 1, 3], dtype=np.int32)
    buf, _ = oracle.pack_heads(pool, ids, 1, 2)
    zero = np.zeros_like(pool)
    rebuilt, rc = oracle.unpack_heads(zero, buf, ids, 1)
    assert rc == 0
    mask = np.zeros(pool.shape, dtype=bool)
    mask[ids[:, None], :, 1:3] = True
    np.testing.assert_array_equal(rebuilt[mask], pool[mask])
    assert np.all(rebuilt[~mask] == 0)
    # the two halves of a head-sharded page rebuild it exactly
    lo, _ = oracle.pack_heads(pool, ids, 0, 2)
    hi, _ = oracle.pack_heads(pool, ids, 2, 2)
    full, _ = oracle.unpack_heads(zero, lo, ids, 0)
    full, _ = oracle.unpack_heads(full, hi, ids, 2)
    np.testing.assert_array_equal(full[ids], pool[ids])


def test_pack_bad_page_is_skipped():
    pool = np.ones((2, 2, 2, 2, 2), dtype=np.uint16)
    buf, rc = oracle.pack_heads(pool, [1, -1], 0, 2)
    assert rc == 1 and np.all(buf[0] == 1) and np.all(buf[1] == 0)
