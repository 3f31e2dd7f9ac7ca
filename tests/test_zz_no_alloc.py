"""attn_decode_noalloc: decode for callers that cannot allocate device memory
while they serve (an engine that reserves its memory budget up front and
forbids cudaMalloc, whose implicit device synchronisation would also stall
its other streams).  Its scratch is a static array inside the library
instead of a caller workspace.

It runs the same decode kernel on the same work list as attn_decode, so the
results must be bitwise equal to attn_decode's, call after call: the static
scratch keeps the previous call's contents, so a second call (with the same
or another plan) must not be disturbed by the first.  They must also match
the fp64 oracle.  This file is collected last on purpose and passes both
alone and after the other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from helpers import check_close, make_plan, syn, to_device

pytestmark = pytest.mark.gpu

INVALID_ARG, WORKSPACE_TOO_SMALL, DEVICE_ERR = 1, 3, 6


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _lib():
    from paged_kv_attention_sink_gb300 import binding
    return binding.load_library()


def _decode_both(batch):
    lib = _lib()
    q, kv, pt, sk = to_device(batch)
    plan = make_plan(batch, pt)
    ref_out = torch.empty_like(q)
    ref_lse = torch.empty(batch.total_rows, batch.num_qo_heads, device="cuda")
    plan.decode(q, kv, sk, ref_out, ref_lse)
    out = torch.full_like(q, float("nan"))
    lse = torch.full_like(ref_lse, float("nan"))
    status = lib.attn_decode_noalloc(plan.handle, _p(q), _p(kv), _p(sk), _p(out), _p(lse), _stream())
    assert status == 0
    code = ctypes.c_int32(-1)
    assert lib.attn_decode_noalloc_device_error(plan.handle, ctypes.byref(code), _stream()) == 0
    assert code.value == 0
    torch.cuda.synchronize()
    return plan, ref_out, ref_lse, out, lse


def _assert_bitwise(ref_out, ref_lse, out, lse):
    assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))
    assert torch.equal(lse.view(torch.int32), ref_lse.view(torch.int32))


def test_noalloc_matches_decode_bitwise_on_consecutive_calls():
    batches = [syn.gptoss_decode(3, batch=24), syn.tiny_decode(1), syn.gptoss_decode(3, batch=24)]
    for batch in batches:       # three calls in a row, the second with another plan
        plan, ref_out, ref_lse, out, lse = _decode_both(batch)
        _assert_bitwise(ref_out, ref_lse, out, lse)


def test_noalloc_matches_oracle_on_a_split_batch():
    batch = syn.gptoss_decode(4, batch=24)
    plan, ref_out, ref_lse, out, lse = _decode_both(batch)
    assert plan.info()["num_decode_partials"] > 0   # the batch is split across SMs
    want_out, want_lse = oracle.sink_attention(batch)
    check_close(out, lse, want_out, want_lse, "noalloc split batch")


def test_noalloc_calls_allocate_nothing():
    batch = syn.gptoss_decode(5, batch=16)
    lib = _lib()
    q, kv, pt, sk = to_device(batch)
    plan = make_plan(batch, pt)
    out = torch.empty_like(q)
    lse = torch.empty(batch.total_rows, batch.num_qo_heads, device="cuda")
    args = (plan.handle, _p(q), _p(kv), _p(sk), _p(out), _p(lse), _stream())
    assert lib.attn_decode_noalloc(*args) == 0       # the first call may load the module
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(5):
        assert lib.attn_decode_noalloc(*args) == 0
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0


def test_noalloc_reports_bad_page_ids():
    """An out-of-pool page id is skipped by the kernel's bounds check and its
    bit lands in the static array's error word, read back (and cleared) by
    attn_decode_noalloc_device_error."""
    batch = syn.tiny_decode(0)
    lib = _lib()
    q, kv, pt, sk = to_device(batch)
    pt[3] = batch.num_pages + 5
    plan = make_plan(batch, pt)
    out = torch.empty_like(q)
    assert lib.attn_decode_noalloc(plan.handle, _p(q), _p(kv), _p(sk), _p(out), None, _stream()) == 0
    code = ctypes.c_int32(0)
    assert lib.attn_decode_noalloc_device_error(plan.handle, ctypes.byref(code), _stream()) == DEVICE_ERR
    assert code.value & 1
    assert lib.attn_decode_noalloc_device_error(plan.handle, ctypes.byref(code), _stream()) == 0
    assert code.value == 0


def test_noalloc_rejects_graph_plans():
    from paged_kv_attention_sink_gb300 import binding
    batch = syn.tiny_decode(0)
    q, kv, pt, sk = to_device(batch)
    gplan = binding.GraphPlan(batch.batch_size, batch.num_qo_heads, batch.num_kv_heads, batch.head_dim,
                              batch.page_size, pt, batch.num_pages, sm_scale=batch.sm_scale)
    out = torch.full_like(q, float("nan"))
    status = _lib().attn_decode_noalloc(gplan.handle, _p(q), _p(kv), _p(sk), _p(out), None, _stream())
    assert status == INVALID_ARG
    torch.cuda.synchronize()
    assert torch.isnan(out.float()).all()          # nothing was launched


def test_noalloc_rejects_plans_larger_than_its_scratch():
    """A plan whose workspace exceeds the static scratch is refused up front."""
    from paged_kv_attention_sink_gb300 import binding
    lib = _lib()
    B, P, kv = 64, 16, 16384
    pages = kv // P
    pt = torch.arange(B * pages, dtype=torch.int32, device="cuda")
    plan = binding.Plan(np.arange(B + 1), np.arange(B + 1) * pages, pt, np.full(B, P), 64, 8, 128, P,
                        num_pages=B * pages, num_sms=2000)
    assert plan.info()["workspace_bytes"] > 16 << 20
    dummy = torch.zeros(1024, dtype=torch.bfloat16, device="cuda")
    status = lib.attn_decode_noalloc(plan.handle, _p(dummy), _p(dummy), None, _p(dummy), None, _stream())
    assert status == WORKSPACE_TOO_SMALL
