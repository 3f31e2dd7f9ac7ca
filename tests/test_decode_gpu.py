"""GPU parity of attn_decode against the fp64 oracle, through the C ABI.

Decode: one query token per request (qo_len = 1) against its whole paged KV
sequence, with the per-head sink in the softmax denominator ("GPT-OSS on day
0", section "Sink Attention").  Pool pages no request uses and the tail of
each last page hold NaN, so any stray read would poison the output.
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import check_close, decode_rows, make_plan, sample_pairs, syn, to_device

pytestmark = pytest.mark.gpu


def run_decode(batch, sinks="batch", num_sms=0, with_lse=True):
    q, kv, pt, sk = to_device(batch)
    if not isinstance(sinks, str):
        sk = None if sinks is None else torch.as_tensor(sinks, dtype=torch.float32, device="cuda")
    plan = make_plan(batch, pt, num_sms=num_sms)
    out = torch.full_like(q, float("nan"))
    lse = torch.full((batch.total_rows, batch.num_qo_heads), float("nan"), device="cuda") if with_lse else None
    plan.decode(q, kv, sk, out, lse)
    torch.cuda.synchronize()
    assert plan.device_error() == 0
    return out, lse, plan


@pytest.mark.parametrize("seed", range(5))
def test_tiny_decode(seed):
    batch = syn.tiny_decode(seed)
    out, lse, _ = run_decode(batch)
    ref_out, ref_lse = oracle.sink_attention(batch)
    check_close(out, lse, ref_out, ref_lse, "tiny")


@pytest.mark.parametrize("variant", ["null", "neg_inf", "huge"])
def test_tiny_decode_sink_variants(variant):
    batch = syn.tiny_decode(1)
    if variant == "null":
        sinks = None
    elif variant == "neg_inf":
        sinks = np.full(batch.num_qo_heads, -np.inf, dtype=np.float32)
    else:
        sinks = np.full(batch.num_qo_heads, 80.0, dtype=np.float32)
    out, lse, _ = run_decode(batch, sinks=sinks)
    ref_out, ref_lse = oracle.sink_attention(batch, sinks=sinks)
    check_close(out, lse, ref_out, ref_lse, variant)


def test_gptoss_decode_full():
    batch = syn.gptoss_decode(0)
    out, lse, plan = run_decode(batch)
    assert plan.info()["num_decode_groups_split"] > 0
    ref_out, ref_lse = oracle.sink_attention(batch)
    check_close(out, lse, ref_out, ref_lse, "gpt-oss decode")


def test_qwen_decode_full():
    """All 128 requests x 64 heads of the Qwen3-shaped long-context decode
    (kv_len log-uniform in [2048, 32768], no sinks) against the oracle."""
    batch = syn.qwen_decode(0)
    out, lse, _ = run_decode(batch)
    ref_out, ref_lse = oracle.sink_attention(batch)
    check_close(out, lse, ref_out, ref_lse, "qwen decode")


@pytest.mark.parametrize("Hq,Hkv,D,P", [
    (8, 8, 64, 16),      # G = 1
    (32, 2, 64, 32),     # G = 16
    (64, 2, 64, 16),     # G = 32: two head slices per KV head
    (24, 2, 128, 16),    # G = 12, D = 128
    (16, 1, 128, 128),   # G = 16, P = 128
    (12, 4, 64, 64),     # G = 3
])
def test_decode_shapes(Hq, Hkv, D, P):
    kv = [1, 15, 16, 17, P, P + 1, 3 * P - 1, 700, 2500]
    batch = syn.make_batch("shapes", [1] * len(kv), kv, Hq, Hkv, D, P, seed=Hq + D + P)
    out, lse, _ = run_decode(batch)
    ref_out, ref_lse = oracle.sink_attention(batch)
    check_close(out, lse, ref_out, ref_lse, f"{Hq}/{Hkv}/{D}/{P}")


@pytest.mark.parametrize("num_sms", [1, 7, 152, 1000])
def test_split_choices_agree(num_sms):
    """Different split-KV chunkings all match the oracle."""
    batch = syn.make_batch("split", [1] * 6, [33, 4000, 9000, 129, 16384, 2], 16, 2, 64, 16, seed=5)
    out, lse, plan = run_decode(batch, num_sms=num_sms)
    ref_out, ref_lse = oracle.sink_attention(batch)
    check_close(out, lse, ref_out, ref_lse, f"sms={num_sms}")


def test_identical_keys():
    """All keys equal: out = mean(V) * n / (n + exp(sink - s))."""
    batch = syn.make_batch("ident", [1, 1], [300, 45], 8, 2, 64, 16, seed=9)
    used = batch.kv_pool[:, 0] != syn.BF16_NAN
    one_key = syn.bf16_bits(np.random.default_rng(0).standard_normal(64).astype(np.float32))
    batch.kv_pool[:, 0][used] = np.broadcast_to(one_key, batch.kv_pool[:, 0].shape)[used]
    out, lse, _ = run_decode(batch)
    ref_out, ref_lse = oracle.sink_attention(batch)
    check_close(out, lse, ref_out, ref_lse, "identical keys")


def test_page_permutation_gives_identical_bits():
    batch = syn.make_batch("perm", [1] * 4, [700, 33, 1200, 16], 16, 2, 64, 16, pool_pages=200, seed=2)
    out_a, lse_a, _ = run_decode(batch)
    perm = np.random.default_rng(1).permutation(batch.num_pages)
    pool = np.empty_like(batch.kv_pool)
    pool[perm] = batch.kv_pool
    batch.kv_pool = pool
    batch.page_table = perm[batch.page_table].astype(np.int32)
    out_b, lse_b, _ = run_decode(batch)
    assert torch.equal(out_a.view(torch.int16), out_b.view(torch.int16))
    assert torch.equal(lse_a, lse_b)


def test_run_to_run_bitwise_deterministic():
    batch = syn.gptoss_decode(1, batch=16)
    q, kv, pt, sk = to_device(batch)
    plan = make_plan(batch, pt)
    outs = []
    for _ in range(3):
        out = torch.empty_like(q)
        lse = torch.empty(batch.total_rows, batch.num_qo_heads, device="cuda")
        plan.decode(q, kv, sk, out, lse)
        outs.append((out.view(torch.int16).clone(), lse.clone()))
    torch.cuda.synchronize()
    for o, l in outs[1:]:
        assert torch.equal(o, outs[0][0]) and torch.equal(l, outs[0][1])


def test_decode_leaves_prefill_rows_untouched():
    batch = syn.make_batch("mixed_small", [5, 1, 3, 1], [40, 77, 3, 1], 8, 2, 64, 16, seed=4)
    out, lse, _ = run_decode(batch)
    ref_out, ref_lse = oracle.sink_attention(batch)
    rows = decode_rows(batch)
    check_close(out[rows], lse[rows], ref_out[rows], ref_lse[rows], "decode rows")
    other = [r for r in range(batch.total_rows) if r not in rows]
    assert torch.isnan(out[other].float()).all() and torch.isnan(lse[other]).all()


def test_lse_optional():
    batch = syn.tiny_decode(2)
    out, _, _ = run_decode(batch, with_lse=False)
    ref_out, _ = oracle.sink_attention(batch)
    check_close(out, None, ref_out, None, "no lse")


def test_bad_page_id_is_flagged_not_faulted():
    """A page id outside the pool is caught by the kernel's own bounds check:
    the load is skipped and the device error word reports it."""
    batch = syn.tiny_decode(0)
    q, kv, pt, sk = to_device(batch)
    pt[3] = batch.num_pages + 5
    plan = make_plan(batch, pt)
    out = torch.empty_like(q)
    plan.decode(q, kv, sk, out, None)
    assert plan.device_error() & 1
    assert plan.device_error() == 0     # cleared by the read


def test_caller_workspace_reused_across_plans():
    """A caller-provided workspace, bound to a new plan per step (as a serving
    loop does once the previous step is done), gives the same bits as a plan
    with its own workspace; a too-small or misaligned one is not used."""
    from paged_kv_attention_sink_gb300 import binding
    b1, b2 = syn.gptoss_decode(seed=3, batch=24), syn.tiny_decode(1)
    ws = torch.empty(64 << 20, dtype=torch.uint8, device="cuda")
    for batch in (b1, b2, b1):
        q, kv, pt, sk = to_device(batch)
        own = make_plan(batch, pt)
        shared = binding.Plan(batch.qo_indptr, batch.kv_indptr, pt, batch.last_page_len, batch.num_qo_heads,
                              batch.num_kv_heads, batch.head_dim, batch.page_size, causal=batch.causal,
                              sm_scale=batch.sm_scale, num_pages=batch.num_pages, workspace=ws)
        assert shared.workspace.data_ptr() == ws.data_ptr()
        o1, o2 = torch.empty_like(q), torch.empty_like(q)
        l1 = torch.empty(batch.total_rows, batch.num_qo_heads, device="cuda")
        l2 = torch.empty_like(l1)
        own.decode(q, kv, sk, o1, l1)
        shared.decode(q, kv, sk, o2, l2)
        torch.cuda.synchronize()
        assert own.device_error() == 0 and shared.device_error() == 0
        assert torch.equal(o1.view(torch.int16), o2.view(torch.int16)) and torch.equal(l1, l2)
        del shared
    q, kv, pt, sk = to_device(b1)
    small = torch.empty(256, dtype=torch.uint8, device="cuda")
    p = binding.Plan(b1.qo_indptr, b1.kv_indptr, pt, b1.last_page_len, b1.num_qo_heads, b1.num_kv_heads,
                     b1.head_dim, b1.page_size, causal=b1.causal, sm_scale=b1.sm_scale, num_pages=b1.num_pages,
                     workspace=small)
    assert p.workspace.data_ptr() != small.data_ptr()
    p2 = binding.Plan(b1.qo_indptr, b1.kv_indptr, pt, b1.last_page_len, b1.num_qo_heads, b1.num_kv_heads,
                      b1.head_dim, b1.page_size, causal=b1.causal, sm_scale=b1.sm_scale, num_pages=b1.num_pages,
                      workspace=ws[16:])
    assert p2.workspace.data_ptr() != ws.data_ptr() + 16


def test_decode_many_short_requests():
    """1024 decode requests of 1..200 tokens: many more work units than CTA
    slots, most of them unsplit, several shorter than one 16-token block."""
    rng = np.random.default_rng(21)
    kv = rng.integers(1, 201, size=1024).tolist()
    batch = syn.make_batch("many", [1] * 1024, kv, 64, 8, 64, 16, seed=21)
    out, lse, _ = run_decode(batch)
    rows, heads = sample_pairs(batch, decode_rows(batch), 1024, seed=4)
    ref_out, ref_lse = oracle.sink_attention(batch, rows=rows, heads=heads)
    ri = torch.from_numpy(rows).cuda()
    hi = torch.from_numpy(heads).long().cuda()
    check_close(out[ri, hi], lse[ri, hi], ref_out, ref_lse, "1024 short decodes")
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()
