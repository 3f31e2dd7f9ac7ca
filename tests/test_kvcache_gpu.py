"""GPU parity of the KV-cache data movement around attention, through the C
ABI, against the oracle (bit-exact: these are copies).

attn_append_kv: the step's new K/V rows go to their cache positions before
attention ("Disaggregated prefill and decode", section "KV Messenger").
attn_pack_kv_heads / attn_unpack_kv_heads: head slices of HND pages to and
from a contiguous buffer (same page, section "Sharded KV transfer").
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import check_close, make_plan, sample_pairs, syn, to_device

pytestmark = pytest.mark.gpu


def _dev_bits(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()


def _host_bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _append(batch, seed=0):
    k_new, v_new = syn.new_kv_rows(batch, seed)
    q, kv, pt, sk = to_device(batch)
    plan = make_plan(batch, pt)
    plan.append_kv(_dev_bits(k_new), _dev_bits(v_new), kv)
    torch.cuda.synchronize()
    return plan, kv, k_new, v_new


@pytest.mark.parametrize("case", [
    dict(qo=[1, 1, 1], kv=[17, 1, 300], Hkv=2, D=64, P=16),          # decode rows, page-boundary positions
    dict(qo=[200, 7, 64], kv=[200, 71, 64], Hkv=2, D=64, P=16),       # prefill with and without a prefix
    dict(qo=[33, 1, 130], kv=[95, 64, 130], Hkv=4, D=128, P=64),      # D = 128, 64-token pages
    dict(qo=[5, 129], kv=[5, 300], Hkv=1, D=64, P=128),
    dict(qo=[3, 2], kv=[40, 2], Hkv=8, D=64, P=32),
])
def test_append_matches_oracle(case):
    batch = syn.make_batch("app", case["qo"], case["kv"], 2 * case["Hkv"], case["Hkv"], case["D"], case["P"],
                           seed=sum(case["kv"]))
    plan, kv, k_new, v_new = _append(batch, seed=1)
    assert plan.device_error() == 0
    ref, rc = oracle.append_kv(batch, k_new, v_new)
    assert rc == 0
    np.testing.assert_array_equal(_host_bits(kv), ref)


def test_append_gptoss_prefill_full():
    batch = syn.gptoss_prefill(0)
    plan, kv, k_new, v_new = _append(batch, seed=2)
    assert plan.device_error() == 0
    ref, _ = oracle.append_kv(batch, k_new, v_new)
    np.testing.assert_array_equal(_host_bits(kv), ref)


def test_append_mixed_then_attention():
    """Append the step's rows, then prefill + decode read them: outputs match
    the oracle's attention over the oracle-appended cache."""
    batch = syn.mixed(0, n_decode=24)
    plan, kv, k_new, v_new = _append(batch, seed=3)
    ref_pool, _ = oracle.append_kv(batch, k_new, v_new)
    np.testing.assert_array_equal(_host_bits(kv), ref_pool)
    batch.kv_pool = ref_pool
    q, _, pt, sk = to_device(batch)
    out = torch.full_like(q, float("nan"))
    lse = torch.full((batch.total_rows, batch.num_qo_heads), float("nan"), device="cuda")
    plan.prefill(q, kv, sk, out, lse)
    plan.decode(q, kv, sk, out, lse)
    torch.cuda.synchronize()
    assert plan.device_error() == 0
    rows, heads = sample_pairs(batch, list(range(batch.total_rows)), 600, seed=4)
    ref_out, ref_lse = oracle.sink_attention(batch, rows=rows, heads=heads)
    ri = torch.from_numpy(rows).cuda()
    hi = torch.from_numpy(heads).long().cuda()
    check_close(out[ri, hi], lse[ri, hi], ref_out, ref_lse, "append + attention")


def test_append_bad_page_sets_error_and_skips_row():
    batch = syn.make_batch("bad", [2, 1], [40, 9], 4, 2, 64, 16, seed=9)
    k_new, v_new = syn.new_kv_rows(batch, 0)
    q, kv, pt, sk = to_device(batch)
    plan = make_plan(batch, pt)
    bad = batch.page_table.copy()
    bad[batch.kv_indptr[1] - 1] = batch.num_pages + 5          # request 0's last page id out of range
    pt.copy_(torch.from_numpy(bad))
    plan.append_kv(_dev_bits(k_new), _dev_bits(v_new), kv)
    assert plan.device_error() == 1                            # ATTN_DEVICE_ERR_PAGE_ID
    batch.page_table = bad
    ref, rc = oracle.append_kv(batch, k_new, v_new)
    assert rc == 1
    np.testing.assert_array_equal(_host_bits(kv), ref)


@pytest.mark.parametrize("Hkv,P,D,h0,nh", [(8, 16, 64, 0, 4), (8, 16, 64, 4, 4), (8, 16, 64, 3, 1),
                                           (4, 64, 128, 1, 2), (2, 128, 64, 0, 2)])
def test_pack_unpack_match_oracle(Hkv, P, D, h0, nh):
    rng = np.random.default_rng(Hkv * P + h0)
    n_pool = 300
    pool = rng.integers(0, 65535, size=(n_pool, 2, Hkv, P, D), dtype=np.uint16)
    ids = rng.choice(n_pool, size=97, replace=False).astype(np.int32)
    kv = _dev_bits(pool)
    ids_d = torch.from_numpy(ids).cuda()
    from paged_kv_attention_sink_gb300 import binding
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    buf = binding.attn_pack_kv_heads(kv, ids_d, h0, nh, device_error=err)
    ref_buf, _ = oracle.pack_heads(pool, ids, h0, nh)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(_host_bits(buf), ref_buf)
    # unpack a different buffer into a copy of the pool
    other = rng.integers(0, 65535, size=ref_buf.shape, dtype=np.uint16)
    binding.attn_unpack_kv_heads(_dev_bits(other), ids_d, h0, kv, device_error=err)
    ref_pool, _ = oracle.unpack_heads(pool, other, ids, h0)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(_host_bits(kv), ref_pool)
    assert int(err.item()) == 0


def test_pack_bad_page_sets_error():
    pool = np.arange(4 * 2 * 2 * 16 * 64, dtype=np.uint16).reshape(4, 2, 2, 16, 64)
    ids = np.array([3, 9, 0], dtype=np.int32)
    from paged_kv_attention_sink_gb300 import binding
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    buf = torch.zeros((3, 2, 1, 16, 64), dtype=torch.bfloat16, device="cuda")
    binding.attn_pack_kv_heads(_dev_bits(pool), torch.from_numpy(ids).cuda(), 1, 1, buf=buf, device_error=err)
    ref, rc = oracle.pack_heads(pool, ids, 1, 1)
    torch.cuda.synchronize()
    assert rc == 1 and int(err.item()) == 1
    np.testing.assert_array_equal(_host_bits(buf), ref)
