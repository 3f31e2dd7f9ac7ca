"""GPU parity of attn_prefill (tcgen05 tensor-core kernel) against the fp64
oracle, through the C ABI.

Prefill: qo_len > 1 query tokens per request, causal with bottom-right
alignment when a cached prefix precedes them, sink in the denominator ("GPT-OSS
on day 0", section "Sink Attention"; request model of "Disaggregated prefill
and decode", section "Prefill vs decode performance").
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import check_close, make_plan, prefill_rows, syn, to_device

pytestmark = pytest.mark.gpu


def run_prefill(batch, sinks="batch", with_lse=True):
    q, kv, pt, sk = to_device(batch)
    if not isinstance(sinks, str):
        sk = None if sinks is None else torch.as_tensor(sinks, dtype=torch.float32, device="cuda")
    plan = make_plan(batch, pt)
    out = torch.full_like(q, float("nan"))
    lse = torch.full((batch.total_rows, batch.num_qo_heads), float("nan"), device="cuda") if with_lse else None
    plan.prefill(q, kv, sk, out, lse)
    torch.cuda.synchronize()
    assert plan.device_error() == 0
    return out, lse, plan


def _check_rows(batch, out, lse, sinks="batch", what=""):
    ref_out, ref_lse = oracle.sink_attention(batch, sinks=sinks)
    rows = prefill_rows(batch)
    return check_close(out[rows], None if lse is None else lse[rows], ref_out[rows],
                       None if lse is None else ref_lse[rows], what)


@pytest.mark.parametrize("lens", [[200, 77], [128, 256, 2, 129], [300], [1000, 513]])
def test_prefill_causal_small(lens):
    batch = syn.make_batch("pf", lens, lens, 8, 2, 64, 16, seed=len(lens) + lens[0])
    out, lse, _ = run_prefill(batch)
    _check_rows(batch, out, lse, what=f"causal {lens}")


def test_prefill_with_cached_prefix():
    """qo_len < kv_len: rows are aligned to the end of the sequence."""
    qo = [64, 200, 130, 7]
    kv = [64, 2248, 4226, 100]
    batch = syn.make_batch("prefix", qo, kv, 8, 2, 64, 16, seed=3)
    out, lse, _ = run_prefill(batch)
    _check_rows(batch, out, lse, what="prefix")


def test_prefill_non_causal():
    batch = syn.make_batch("nc", [100, 260], [300, 260], 8, 2, 64, 16, causal=False, seed=4)
    out, lse, _ = run_prefill(batch)
    _check_rows(batch, out, lse, what="non-causal")


@pytest.mark.parametrize("Hq,Hkv,D,P", [
    (8, 8, 64, 16),     # G = 1: one head per CTA
    (12, 4, 64, 32),    # G = 3: a pair and a single
    (16, 2, 128, 64),   # D = 128
    (8, 2, 64, 128),    # one page per KV tile
    (4, 1, 128, 16),
])
def test_prefill_shapes(Hq, Hkv, D, P):
    qo = [300, 129, 64]
    kv = [300, 500, 64]
    batch = syn.make_batch("shapes", qo, kv, Hq, Hkv, D, P, seed=Hq * D + P)
    out, lse, _ = run_prefill(batch)
    _check_rows(batch, out, lse, what=f"{Hq}/{Hkv}/{D}/{P}")


@pytest.mark.parametrize("variant", ["null", "huge"])
def test_prefill_sink_variants(variant):
    batch = syn.make_batch("sinkvar", [150, 40], [150, 90], 8, 2, 64, 16, seed=6)
    sinks = None if variant == "null" else np.full(8, 80.0, dtype=np.float32)
    out, lse, _ = run_prefill(batch, sinks=sinks)
    _check_rows(batch, out, lse, sinks=sinks, what=variant)


def test_prefill_large_scores_rescale():
    """Scaled-up queries make the running max jump across tiles, exercising
    the lazy O rescale."""
    batch = syn.make_batch("scale", [700], [700], 4, 1, 64, 16, seed=7)
    q = syn.bf16_to_float(batch.q) * 6.0
    batch.q = syn.bf16_bits(q)
    out, lse, _ = run_prefill(batch)
    _check_rows(batch, out, lse, what="large scores")


def _scale_keys(batch, b, lo, hi, factor):
    """Multiply the K rows of keys [lo, hi) of request b by `factor`."""
    k = syn.bf16_to_float(batch.kv_pool)
    P = batch.page_size
    for t in range(lo, min(hi, int(batch.kv_lens[b]))):
        page = batch.page_table[batch.kv_indptr[b] + t // P]
        k[page, 0, :, t % P, :] *= factor
    batch.kv_pool = syn.bf16_bits(k)


@pytest.mark.parametrize("head_dim", [64, 128])
@pytest.mark.parametrize("causal", [True, False])
def test_prefill_max_jumps_mid_item(causal, head_dim):
    """Later key tiles score far above the first tile (by more than 64 in
    log2 units), so a tile's P row sum passes the limit and the tile is
    redone: S reloaded from TMEM, the running max raised mid-item and O
    rescaled -- twice."""
    batch = syn.make_batch("jump", [700], [700], 4, 1, head_dim, 16, causal=causal, seed=12)
    _scale_keys(batch, 0, 300, 500, 30.0)
    _scale_keys(batch, 0, 500, 700, 80.0)
    out, lse, _ = run_prefill(batch)
    _check_rows(batch, out, lse, what=f"max jump causal={causal} D={head_dim}")


@pytest.mark.parametrize("head_dim", [64, 128])
def test_prefill_huge_key_element_in_a_dimension_queries_zero(head_dim):
    """A key element of 3e4 in a dimension every query has zeroed leaves the
    scores as they were: the output must not see it."""
    batch = syn.make_batch("zerodim", [600], [600], 4, 1, head_dim, 16, seed=13)
    q = syn.bf16_to_float(batch.q)
    q[..., 5] = 0.0
    batch.q = syn.bf16_bits(q)
    k = syn.bf16_to_float(batch.kv_pool)
    P = batch.page_size
    for t in (200, 450):
        page = batch.page_table[batch.kv_indptr[0] + t // P]
        k[page, 0, :, t % P, 5] = 3.0e4
    batch.kv_pool = syn.bf16_bits(k)
    out, lse, _ = run_prefill(batch)
    _check_rows(batch, out, lse, what=f"huge key element D={head_dim}")


def test_gptoss_prefill_full():
    """Every row and head of the gpt-oss-shaped prefill (13,804 rows x 64
    heads, 3,584 work items over 152 persistent CTAs) against the oracle, in
    the launch configuration the benchmark times."""
    batch = syn.gptoss_prefill(0)
    out, lse, plan = run_prefill(batch)
    ref_out, ref_lse = oracle.sink_attention(batch)
    check_close(out, lse, ref_out, ref_lse, "gpt-oss prefill")


def test_mixed_batch_full():
    """One plan, prefill then decode on the same stream; every row and head
    (8,192 prefill rows and 256 decode rows x 64 heads) against the oracle."""
    batch = syn.mixed(0)
    q, kv, pt, sk = to_device(batch)
    plan = make_plan(batch, pt)
    out = torch.full_like(q, float("nan"))
    lse = torch.full((batch.total_rows, batch.num_qo_heads), float("nan"), device="cuda")
    plan.prefill(q, kv, sk, out, lse)
    plan.decode(q, kv, sk, out, lse)
    torch.cuda.synchronize()
    assert plan.device_error() == 0
    ref_out, ref_lse = oracle.sink_attention(batch)
    check_close(out, lse, ref_out, ref_lse, "mixed")


def test_prefill_bitwise_deterministic():
    batch = syn.make_batch("det", [400, 130], [400, 300], 8, 2, 64, 16, seed=8)
    q, kv, pt, sk = to_device(batch)
    plan = make_plan(batch, pt)
    res = []
    for _ in range(3):
        out = torch.empty_like(q)
        lse = torch.empty(batch.total_rows, batch.num_qo_heads, device="cuda")
        plan.prefill(q, kv, sk, out, lse)
        res.append((out.view(torch.int16).clone(), lse.clone()))
    torch.cuda.synchronize()
    for o, l in res[1:]:
        assert torch.equal(o, res[0][0]) and torch.equal(l, res[0][1])


@pytest.mark.parametrize("num_sms", [1, 3, 152])
def test_prefill_persistent_item_streams(num_sms):
    """Few CTAs walk long item lists (mixed head counts, ragged and full
    tiles), so barrier phases carry across many items per CTA."""
    batch = syn.make_batch("persist", [300, 129, 2, 700], [300, 400, 2, 900], 12, 4, 64, 16, seed=11)
    q, kv, pt, sk = to_device(batch)
    plan = make_plan(batch, pt, num_sms=num_sms)
    out = torch.full_like(q, float("nan"))
    lse = torch.full((batch.total_rows, batch.num_qo_heads), float("nan"), device="cuda")
    plan.prefill(q, kv, sk, out, lse)
    torch.cuda.synchronize()
    assert plan.device_error() == 0
    _check_rows(batch, out, lse, what=f"sms={num_sms}")


def test_prefill_long_sequence_full():
    """A 32K-token sequence whose last 8K tokens are the prefill rows (24K cached
    prefix), Qwen3-like D = 128 and P = 64: 256 KV tiles per item, so the
    running max is reused across many tiles and the item lists are long.
    Every row and head against the oracle."""
    batch = syn.make_batch("long", [8192, 300], [32768, 300], 16, 4, 128, 64, seed=13)
    out, lse, _ = run_prefill(batch)
    ref_out, ref_lse = oracle.sink_attention(batch)
    check_close(out, lse, ref_out, ref_lse, "long prefill")
