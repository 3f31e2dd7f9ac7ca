"""GPU parity of attn_merge_states (log-sum-exp merge of two attention states).

The merge is the step that the split of attention along the KV length in
"GPT-OSS on day 0", section "Sink Attention", implies; the sink must be
counted in exactly one of the two states."""
import numpy as np
import pytest
import torch

import oracle
from helpers import bf16_ulp, check_close, make_plan, syn, to_device

pytestmark = pytest.mark.gpu


def test_merge_random_states_matches_oracle():
    rng = np.random.default_rng(0)
    n, H, D = 333, 8, 64
    va = syn.bf16_bits(rng.standard_normal((n, H, D)).astype(np.float32))
    vb = syn.bf16_bits(rng.standard_normal((n, H, D)).astype(np.float32))
    la = (rng.standard_normal((n, H)) * 3).astype(np.float32)
    lb = (rng.standard_normal((n, H)) * 3).astype(np.float32)
    lb[:5] = -np.inf
    la[:2] = -np.inf
    dev = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()
    vout = torch.empty(n, H, D, dtype=torch.bfloat16, device="cuda")
    lout = torch.empty(n, H, device="cuda")
    from paged_kv_attention_sink_gb300 import binding
    binding.attn_merge_states(dev(va), torch.from_numpy(la).cuda(), dev(vb), torch.from_numpy(lb).cuda(),
                              vout, lout)
    ref_v, ref_l = oracle.merge_states(syn.bf16_to_float(va).astype(np.float64), la.astype(np.float64),
                                       syn.bf16_to_float(vb).astype(np.float64), lb.astype(np.float64))
    check_close(vout, lout, ref_v, ref_l, "merge")


def _subset_batch(batch, keep_pages, first):
    """Requests restricted to their first `keep_pages` pages (first=True) or to
    the remaining pages (first=False); same pool."""
    b2 = syn.Batch(**{**batch.__dict__})
    kv_indptr = [0]
    pt, lpl, kv = [], [], []
    P = batch.page_size
    for b in range(batch.batch_size):
        pages = batch.page_table[batch.kv_indptr[b]:batch.kv_indptr[b + 1]]
        k = keep_pages[b]
        sel = pages[:k] if first else pages[k:]
        pt.extend(sel)
        kv_indptr.append(len(pt))
        if first:
            lpl.append(P)
            kv.append(k * P)
        else:
            lpl.append(batch.last_page_len[b])
            kv.append(batch.kv_lens[b] - k * P)
    b2.page_table = np.asarray(pt, dtype=np.int32)
    b2.kv_indptr = np.asarray(kv_indptr, dtype=np.int32)
    b2.last_page_len = np.asarray(lpl, dtype=np.int32)
    b2.kv_lens = np.asarray(kv)
    return b2


def test_two_decodes_merged_equal_full_attention():
    """Attention over a prefix of pages (with the sink) merged with attention
    over the rest (no sink) equals attention over everything."""
    batch = syn.make_batch("cascade", [1] * 5, [64, 500, 1000, 2049, 16 * 40 + 3], 16, 2, 64, 16, seed=8)
    keep = [1, 10, 31, 64, 20]
    first = _subset_batch(batch, keep, True)
    rest = _subset_batch(batch, keep, False)
    q, kv, _, sk = to_device(batch)
    outs = []
    for part, sinks in ((first, sk), (rest, None)):
        pt = torch.from_numpy(part.page_table).cuda()
        plan = make_plan(part, pt)
        out = torch.empty_like(q)
        lse = torch.empty(batch.total_rows, batch.num_qo_heads, device="cuda")
        plan.decode(q, kv, sinks, out, lse)
        outs.append((out, lse, plan))
    from paged_kv_attention_sink_gb300 import binding
    vout, lout = binding.attn_merge_states(outs[0][0], outs[0][1], outs[1][0], outs[1][1],
                                           lseout=torch.empty_like(outs[0][1]))
    ref_out, ref_lse = oracle.sink_attention(batch)
    check_close(vout, lout, ref_out, ref_lse, "cascade merge")


def test_merge_f32_random_states_matches_oracle():
    """fp32 value states merge in fp32: against the fp64 merge of the same
    inputs, within fp32 rounding; the bf16 output within the bf16 tolerance."""
    rng = np.random.default_rng(1)
    n, H, D = 257, 8, 64
    va = rng.standard_normal((n, H, D)).astype(np.float32)
    vb = rng.standard_normal((n, H, D)).astype(np.float32)
    la = (rng.standard_normal((n, H)) * 3).astype(np.float32)
    lb = (rng.standard_normal((n, H)) * 3).astype(np.float32)
    lb[:5] = -np.inf
    la[:2] = -np.inf
    la[7, :] = lb[7, :] = -np.inf        # both empty: the identity
    ref_v, ref_l = oracle.merge_states(va.astype(np.float64), la.astype(np.float64),
                                       vb.astype(np.float64), lb.astype(np.float64))
    from paged_kv_attention_sink_gb300 import binding
    d = lambda a: torch.from_numpy(a).cuda()
    lout = torch.empty(n, H, device="cuda")
    v32, _ = binding.attn_merge_states_f32(d(va), d(la), d(vb), d(lb), lseout=lout)
    torch.cuda.synchronize()
    v32 = v32.cpu().numpy().astype(np.float64)
    assert np.abs(v32 - ref_v).max() <= 2e-6 * max(1.0, np.abs(ref_v).max())
    fin = np.isfinite(ref_l)
    assert np.array_equal(np.isfinite(lout.cpu().numpy()), fin)
    assert np.abs(lout.cpu().numpy()[fin] - ref_l[fin]).max() <= 2e-6 * max(1.0, np.abs(ref_l[fin]).max())
    # bf16 output: the fp32 result rounded once, so within one bf16 ulp of the
    # fp64 value everywhere (random N(0,1) states are larger than attention
    # outputs, so the attention tolerance is not the right bar here)
    vbf, _ = binding.attn_merge_states_f32(d(va), d(la), d(vb), d(lb), out_dtype=torch.bfloat16)
    vbf = vbf.double().cpu().numpy()
    assert np.all(np.abs(vbf - ref_v) <= bf16_ulp(ref_v))
    # in place into va
    va_d = d(va)
    binding.attn_merge_states_f32(va_d, d(la), d(vb), d(lb), vout=va_d)
    torch.cuda.synchronize()
    assert np.abs(va_d.cpu().numpy().astype(np.float64) - ref_v).max() <= 2e-6 * max(1.0, np.abs(ref_v).max())


def test_merge_f32_of_exact_partials_equals_full_attention():
    """Split-KV partial states (the oracle's own, in fp32, the sink in the
    first part only) merged on the GPU in fp32 give the unsplit attention to
    fp32 precision: the merge adds no bf16 rounding."""
    batch = syn.make_batch("split", [1] * 6, [64, 500, 1000, 2049, 700, 3000], 16, 2, 64, 16, seed=9)
    cut = 333
    oa, la = oracle.sink_attention(batch, kv_lo=0, kv_hi=cut, with_sink=True)
    ob, lb = oracle.sink_attention(batch, kv_lo=cut, with_sink=False)
    full_o, full_l = oracle.sink_attention(batch)
    from paged_kv_attention_sink_gb300 import binding
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()
    lout = torch.empty(batch.total_rows, batch.num_qo_heads, device="cuda")
    v, _ = binding.attn_merge_states_f32(d(oa), d(la), d(ob), d(lb), lseout=lout)
    torch.cuda.synchronize()
    assert np.abs(v.cpu().numpy() - full_o).max() <= 1e-5
    assert np.abs(lout.cpu().numpy() - full_l).max() <= 1e-5
