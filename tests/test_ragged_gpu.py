"""GPU parity of the ragged, non-paged prefill (attn_plan_ragged +
attn_prefill_ragged) against the fp64 oracle, through the C ABI.

No KV cache: K and V are contiguous [tokens, Hkv, D] arrays with a token CSR
("Fast embeddings on GPUs", section "ROSE": embedding serving skips the KV
cache and uses attention kernels that take ragged inputs, so nothing is
padded).  The inputs are the paged synthetic batches with each request's K/V
rows gathered into one contiguous array, so the oracle runs on the paged form.
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import check_close, sample_pairs, syn

pytestmark = pytest.mark.gpu


def ragged_inputs(batch):
    """Contiguous K, V bits [sum kv_len, Hkv, D] and the token CSR."""
    P = batch.page_size
    ks, vs = [], []
    for b in range(batch.batch_size):
        n = int(batch.kv_lens[b])
        t = np.arange(n)
        pages = batch.page_table[batch.kv_indptr[b] + t // P]
        ks.append(batch.kv_pool[pages, 0, :, t % P, :])
        vs.append(batch.kv_pool[pages, 1, :, t % P, :])
    kv_indptr = np.concatenate([[0], np.cumsum(batch.kv_lens)]).astype(np.int32)
    return np.concatenate(ks), np.concatenate(vs), kv_indptr


def _dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def run_ragged(batch, num_sms=0):
    from paged_kv_attention_sink_gb300 import binding
    k, v, kv_indptr = ragged_inputs(batch)
    plan = binding.RaggedPlan(batch.qo_indptr, kv_indptr, batch.num_qo_heads, batch.num_kv_heads, batch.head_dim,
                              causal=batch.causal, sm_scale=batch.sm_scale, num_sms=num_sms)
    q = _dev(batch.q)
    sk = None if batch.sinks is None else torch.from_numpy(batch.sinks).cuda()
    out = torch.full_like(q, float("nan"))
    lse = torch.full((batch.total_rows, batch.num_qo_heads), float("nan"), device="cuda")
    plan.prefill(q, _dev(k), _dev(v), sk, out, lse)
    torch.cuda.synchronize()
    assert plan.device_error() == 0
    return out, lse, plan


@pytest.mark.parametrize("qo,kv,causal", [
    ([300, 77, 1, 129], [300, 77, 1, 129], True),      # self-attention, causal, a 1-token request
    ([300, 77, 1, 129], [300, 77, 1, 129], False),     # bidirectional (embedding models)
    ([64, 200, 3], [100, 2248, 3], True),              # queries aligned to the end of longer keys
    ([40, 1000], [513, 1000], False),
])
def test_ragged_matches_oracle(qo, kv, causal):
    batch = syn.make_batch("rag", qo, kv, 8, 2, 64, 16, causal=causal, seed=sum(kv) + int(causal))
    out, lse, _ = run_ragged(batch)
    ref_out, ref_lse = oracle.sink_attention(batch)
    check_close(out, lse, ref_out, ref_lse, f"ragged {qo}/{kv} causal={causal}")


@pytest.mark.parametrize("Hq,Hkv,D", [(16, 2, 128), (12, 4, 64), (4, 4, 64)])
def test_ragged_shapes(Hq, Hkv, D):
    batch = syn.make_batch("ragshape", [129, 260, 5], [129, 300, 5], Hq, Hkv, D, 32, seed=Hq + D)
    out, lse, _ = run_ragged(batch, num_sms=3)
    ref_out, ref_lse = oracle.sink_attention(batch)
    check_close(out, lse, ref_out, ref_lse, f"ragged {Hq}/{Hkv}/{D}")


def test_ragged_no_sinks():
    batch = syn.make_batch("ragns", [200, 31], [200, 31], 8, 2, 64, 16, with_sinks=False, seed=5)
    out, lse, _ = run_ragged(batch)
    ref_out, ref_lse = oracle.sink_attention(batch)
    check_close(out, lse, ref_out, ref_lse, "ragged without sinks")


def test_ragged_gptoss_prefill_sampled():
    batch = syn.gptoss_prefill(1)
    out, lse, _ = run_ragged(batch)
    rows, heads = sample_pairs(batch, list(range(batch.total_rows)), 512, seed=6)
    ref_out, ref_lse = oracle.sink_attention(batch, rows=rows, heads=heads)
    ri = torch.from_numpy(rows).cuda()
    hi = torch.from_numpy(heads).long().cuda()
    check_close(out[ri, hi], lse[ri, hi], ref_out, ref_lse, "ragged gpt-oss prefill")
    assert torch.isfinite(out.float()).all()


def test_ragged_plan_rejects_paged_calls():
    from paged_kv_attention_sink_gb300 import binding
    plan = binding.RaggedPlan(np.array([0, 2]), np.array([0, 5]), 4, 2, 64)
    lib = binding.load_library()
    import ctypes
    p = ctypes.c_void_p(plan.workspace.data_ptr())
    assert lib.attn_prefill(plan.handle, p, p, None, p, None, None) == 1      # paged entry refuses a ragged plan
    assert lib.attn_append_kv(plan.handle, p, p, p, None) == 1
