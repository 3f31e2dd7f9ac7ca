"""attn_decode_noalloc: decode for callers that cannot allocate device memory
while they run attention (for example a step replayed from a captured CUDA
graph, or an engine that reserves its memory budget up front).  Its scratch
is a static array inside the library instead of a caller workspace.

The results must match attn_decode on the same plan and inputs, call after
call: the static scratch keeps the previous call's contents, so a second call
(with the same or another plan) must not be disturbed by the first.  This file
is collected last on purpose and passes both alone and after the other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

from helpers import LSE_ABS, MAX_ABS, MEAN_ABS, make_plan, syn, to_device

pytestmark = pytest.mark.gpu

WORKSPACE_TOO_SMALL = 3


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _decode_both(batch):
    from paged_kv_attention_sink_gb300 import binding
    lib = binding.load_library()
    q, kv, pt, sk = to_device(batch)
    plan = make_plan(batch, pt)
    ref_out = torch.empty_like(q)
    ref_lse = torch.empty(batch.total_rows, batch.num_qo_heads, device="cuda")
    plan.decode(q, kv, sk, ref_out, ref_lse)
    out = torch.full_like(q, float("nan"))
    lse = torch.full_like(ref_lse, float("nan"))
    status = lib.attn_decode_noalloc(plan.handle, _p(q), _p(kv), _p(sk), _p(out), _p(lse), _stream())
    assert status == 0
    torch.cuda.synchronize()
    return ref_out, ref_lse, out, lse


def _assert_same(ref_out, ref_lse, out, lse):
    err = (out.float() - ref_out.float()).abs()
    assert torch.isfinite(out.float()).all()
    assert err.max().item() <= MAX_ABS and err.mean().item() <= MEAN_ABS
    assert (lse - ref_lse).abs().max().item() <= LSE_ABS


def test_noalloc_matches_decode_on_consecutive_calls():
    batches = [syn.gptoss_decode(3, batch=24), syn.tiny_decode(1), syn.gptoss_decode(3, batch=24)]
    for batch in batches:       # three calls in a row, the second with another plan
        _assert_same(*_decode_both(batch))


def test_noalloc_rejects_plans_larger_than_its_scratch():
    """A plan whose workspace exceeds the static scratch is refused up front."""
    from paged_kv_attention_sink_gb300 import binding
    lib = binding.load_library()
    B, P, kv = 64, 16, 16384
    pages = kv // P
    pt = torch.arange(B * pages, dtype=torch.int32, device="cuda")
    plan = binding.Plan(np.arange(B + 1), np.arange(B + 1) * pages, pt, np.full(B, P), 64, 8, 128, P,
                        num_pages=B * pages, num_sms=2000)
    assert plan.info()["workspace_bytes"] > 16 << 20
    dummy = torch.zeros(1024, dtype=torch.bfloat16, device="cuda")
    status = lib.attn_decode_noalloc(plan.handle, _p(dummy), _p(dummy), None, _p(dummy), None, _stream())
    assert status == WORKSPACE_TOO_SMALL
