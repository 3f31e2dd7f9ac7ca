"""GPU check of the kernels' failure detection without a fault: a wait that
nothing completes must end, with the timeout bit recorded for the host, and
leave the context usable for the next launch."""
import pytest
import torch

import oracle
from helpers import check_close, decode_rows, make_plan, syn, to_device

pytestmark = pytest.mark.gpu

ATTN_DEVICE_ERR_TIMEOUT = 2


def test_bounded_wait_gives_up_and_context_stays_usable():
    from paged_kv_attention_sink_gb300 import binding
    res = binding.attn_selftest_bounded_wait()
    torch.cuda.synchronize()
    status, waited_ns = (int(x) for x in res.cpu())
    assert status == ATTN_DEVICE_ERR_TIMEOUT
    assert 2.0e9 <= waited_ns < 6.0e9            # the 2 s limit, plus a sleep-hint period or so
    # the same context runs attention afterwards
    b = syn.tiny_decode(0)
    q, kv, pt, sk = to_device(b)
    plan = make_plan(b, pt)
    out = torch.full_like(q, float("nan"))
    lse = torch.full((b.total_rows, b.num_qo_heads), float("nan"), device="cuda")
    plan.decode(q, kv, sk, out, lse)
    torch.cuda.synchronize()
    assert plan.device_error() == 0
    rows = decode_rows(b)
    ref_out, ref_lse = oracle.sink_attention(b)
    check_close(out[rows], lse[rows], ref_out[rows], ref_lse[rows], "decode after a timed-out wait")
