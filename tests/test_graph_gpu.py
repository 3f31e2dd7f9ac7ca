"""GPU tests of the CUDA-graph decode path (attn_graph_plan + attn_decode_graph):
the work list is built on the device from device-resident request metadata,
so one captured graph replays for new batches ("Fast embeddings on GPUs",
section "Managing CUDA graphs": kernels configured from dynamic host inputs
prevent full CUDA graphs).  Parity is against the fp64 oracle; the device
planner is also checked unit for unit against the host planner.
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import check_close, make_plan, sample_pairs, syn, to_device

pytestmark = pytest.mark.gpu


class Buffers:
    """Fixed device buffers a captured graph reads; each batch is copied in."""

    def __init__(self, max_batch, Hq, Hkv, D, P, max_pages, max_slots):
        dev = "cuda"
        self.q = torch.zeros((max_batch, Hq, D), dtype=torch.bfloat16, device=dev)
        self.out = torch.zeros_like(self.q)
        self.lse = torch.zeros((max_batch, Hq), dtype=torch.float32, device=dev)
        self.kv = torch.zeros((max_pages, 2, Hkv, P, D), dtype=torch.bfloat16, device=dev)
        self.pt = torch.zeros(max_slots, dtype=torch.int32, device=dev)
        self.kv_indptr = torch.zeros(max_batch + 1, dtype=torch.int32, device=dev)
        self.lpl = torch.zeros(max_batch, dtype=torch.int32, device=dev)
        self.batch = torch.zeros(1, dtype=torch.int32, device=dev)
        self.sinks = torch.zeros(Hq, dtype=torch.float32, device=dev)

    def load(self, b):
        B = b.batch_size
        q, kv, pt, sk = to_device(b)
        self.q[:B].copy_(q)
        self.kv[:b.num_pages].copy_(kv)
        self.pt[:len(b.page_table)].copy_(pt)
        self.kv_indptr[:B + 1].copy_(torch.from_numpy(b.kv_indptr))
        self.lpl[:B].copy_(torch.from_numpy(b.last_page_len))
        self.batch.fill_(B)
        self.sinks.copy_(sk)
        self.out.fill_(float("nan"))
        self.lse.fill_(float("nan"))


def _graph_plan(buf, max_batch, b, **kw):
    from paged_kv_attention_sink_gb300 import binding
    return binding.GraphPlan(max_batch, b.num_qo_heads, b.num_kv_heads, b.head_dim, b.page_size, buf.pt,
                             buf.kv.shape[0], sm_scale=b.sm_scale, **kw)


def _decode(plan, buf):
    return plan.decode(buf.q, buf.kv, buf.kv_indptr, buf.lpl, buf.batch, buf.sinks, buf.out, buf.lse)


def _check(b, buf, n=600, seed=0, what=""):
    rows, heads = sample_pairs(b, list(range(b.batch_size)), n, seed=seed)
    ref_out, ref_lse = oracle.sink_attention(b, rows=rows, heads=heads)
    ri = torch.from_numpy(rows).cuda()
    hi = torch.from_numpy(heads).long().cuda()
    check_close(buf.out[ri, hi], buf.lse[ri, hi], ref_out, ref_lse, what)


@pytest.mark.parametrize("which", ["gptoss", "300_requests"])
def test_device_plan_equals_host_plan(which):
    """The gpt-oss batch (64 requests, capacity 96) and 300 requests of up to
    3K tokens (capacity 600)."""
    if which == "gptoss":
        b, max_batch = syn.gptoss_decode(0), 96
    else:
        kv = np.random.default_rng(15).integers(1, 3000, size=300).tolist()
        b, max_batch = syn.make_batch("r300", [1] * 300, kv, 64, 8, 64, 16, seed=15), 600
    buf = Buffers(max_batch, 64, 8, 64, 16, b.num_pages, len(b.page_table))
    buf.load(b)
    plan = _graph_plan(buf, max_batch, b)
    _decode(plan, buf)
    dev_units = plan.device_units()
    q, kv, pt, sk = to_device(b)
    host_units = make_plan(b, pt).decode_units()
    # Same chunks (request, heads, token range, chunk index / count) ...
    key = lambda u: tuple(int(x) for x in u[:9])
    assert sorted(map(key, dev_units)) == sorted(map(key, host_units))
    # ... ordered longest first like the host's ...
    lens = dev_units[:, 6] - dev_units[:, 5]
    assert np.all(np.diff(lens) <= 16)            # chunks of one request differ by at most one block
    # ... and a consistent numbering of split groups and partial slots (the two
    # planners number them in different orders).
    groups, slots = {}, set()
    for u in dev_units:
        q_row, kv_head, head0, chunk, n_chunks, group, partial0 = (int(u[i]) for i in (0, 2, 3, 7, 8, 9, 10))
        if n_chunks == 1:
            assert group == -1
            continue
        assert groups.setdefault((q_row, kv_head, head0), (group, partial0)) == (group, partial0)
        assert partial0 + chunk not in slots
        slots.add(partial0 + chunk)
    assert len(set(groups.values())) == len(groups)
    assert plan.device_error() == 0


def test_in_grid_plan_equals_planner_kernel_plan():
    """Plans of up to 128 requests are built inside the persistent decode grid
    (every CTA plans for itself), larger ones by the planner kernel: the same
    batch under a 128-request and a 129-request plan gives the same units and
    the same output, bit for bit."""
    kv = np.random.default_rng(16).integers(1, 5000, size=100).tolist()
    b = syn.make_batch("r100", [1] * 100, kv, 64, 8, 64, 16, seed=16)
    res = []
    for max_batch in (128, 129):
        buf = Buffers(max_batch, 64, 8, 64, 16, b.num_pages, len(b.page_table))
        buf.load(b)
        plan = _graph_plan(buf, max_batch, b)
        _decode(plan, buf)
        torch.cuda.synchronize()
        assert plan.device_error() == 0
        key = lambda u: tuple(int(x) for x in u[:9])
        res.append((sorted(map(key, plan.device_units())), buf.out[:b.batch_size].clone(), buf.lse[:b.batch_size].clone()))
    assert res[0][0] == res[1][0]
    assert torch.equal(res[0][1].view(torch.int16), res[1][1].view(torch.int16))
    assert torch.equal(res[0][2], res[1][2])
    _check(b, buf, what="graph decode, 100 requests")


@pytest.mark.parametrize("which", ["gptoss", "tiny", "long"])
def test_graph_decode_matches_oracle(which):
    if which == "gptoss":
        b = syn.gptoss_decode(3)
    elif which == "tiny":
        b = syn.tiny_decode(0)
    else:
        b = syn.make_batch("long", [1, 1], [70000, 33], 16, 2, 128, 64, seed=5)
    buf = Buffers(b.batch_size + 7, b.num_qo_heads, b.num_kv_heads, b.head_dim, b.page_size, b.num_pages,
                  len(b.page_table))
    buf.load(b)
    plan = _graph_plan(buf, b.batch_size + 7, b)
    _decode(plan, buf)
    torch.cuda.synchronize()
    assert plan.device_error() == 0
    _check(b, buf, what=f"graph decode {which}")
    assert torch.isnan(buf.out[b.batch_size:].float()).all()      # rows past the batch are not touched


def test_cuda_graph_capture_replays_new_batches():
    """Capture once, replay for three batches of different sizes and lengths."""
    batches = [syn.gptoss_decode(seed=7, batch=40), syn.gptoss_decode(seed=8, batch=64),
               syn.make_batch("short", [1] * 9, [5, 17, 300, 1, 16, 64, 2000, 9000, 33], 64, 8, 64, 16, seed=9)]
    max_pages = max(b.num_pages for b in batches)
    max_slots = max(len(b.page_table) for b in batches)
    max_tokens = max(int(b.kv_lens.sum()) for b in batches)
    buf = Buffers(64, 64, 8, 64, 16, max_pages, max_slots)
    buf.load(batches[0])
    plan = _graph_plan(buf, 64, batches[0], max_kv_tokens=max_tokens)
    _decode(plan, buf)                         # uncaptured call: builds the TMA descriptor
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            _decode(plan, buf)
    torch.cuda.current_stream().wait_stream(s)
    for k, b in enumerate(batches):
        buf.load(b)
        g.replay()
        torch.cuda.synchronize()
        assert plan.device_error() == 0
        _check(b, buf, n=400, seed=k, what=f"replay {k}")


@pytest.mark.parametrize("max_batch", [128, 200])
def test_graph_empty_and_full_batches(max_batch):
    """B = 0 leaves every row untouched and records no error; B = max_batch
    fills the plan (128: the most the in-grid plan takes; 200: the planner
    kernel).  Both paths, one plan, one after the other."""
    kv = np.random.default_rng(17).integers(1, 1200, size=max_batch).tolist()
    b = syn.make_batch("full", [1] * max_batch, kv, 16, 2, 64, 16, seed=17)
    buf = Buffers(max_batch, 16, 2, 64, 16, b.num_pages, len(b.page_table))
    buf.load(b)
    plan = _graph_plan(buf, max_batch, b)
    buf.batch.fill_(0)
    _decode(plan, buf)
    torch.cuda.synchronize()
    assert plan.device_error() == 0
    assert len(plan.device_units()) == 0
    assert torch.isnan(buf.out.float()).all()
    buf.batch.fill_(max_batch)
    _decode(plan, buf)
    torch.cuda.synchronize()
    assert plan.device_error() == 0
    _check(b, buf, n=500, seed=3, what=f"graph decode, {max_batch} of {max_batch} requests")
    assert torch.isfinite(buf.out.float()).all()


def test_graph_malformed_request_sets_plan_error():
    b = syn.make_batch("bad", [1, 1, 1], [40, 90, 7], 8, 2, 64, 16, seed=11)
    buf = Buffers(4, 8, 2, 64, 16, b.num_pages, len(b.page_table))
    buf.load(b)
    buf.lpl[1] = 0                              # request 1: last page length out of range
    plan = _graph_plan(buf, 4, b)
    _decode(plan, buf)
    assert plan.device_error() == 4             # ATTN_DEVICE_ERR_PLAN
    rows = np.array([0, 0, 2, 2]), np.array([0, 5, 1, 7], dtype=np.int32)
    ref_out, ref_lse = oracle.sink_attention(b, rows=rows[0], heads=rows[1])
    ri = torch.from_numpy(rows[0]).cuda()
    hi = torch.from_numpy(rows[1]).long().cuda()
    check_close(buf.out[ri, hi], buf.lse[ri, hi], ref_out, ref_lse, "graph decode around a bad request")
    assert torch.isnan(buf.out[1].float()).all()


def test_graph_batch_beyond_capacity_sets_plan_error():
    b = syn.make_batch("cap", [1, 1], [40, 90], 8, 2, 64, 16, seed=12)
    buf = Buffers(2, 8, 2, 64, 16, b.num_pages, len(b.page_table))
    buf.load(b)
    buf.batch.fill_(3)                          # more requests than the plan's max_batch
    plan = _graph_plan(buf, 2, b)
    _decode(plan, buf)
    assert plan.device_error() == 4


def test_graph_decode_at_planner_capacity():
    """4096 requests, the most one device-planned replay can order."""
    rng = np.random.default_rng(22)
    kv = rng.integers(1, 300, size=4096).tolist()
    b = syn.make_batch("cap4096", [1] * 4096, kv, 16, 2, 64, 16, seed=22)
    buf = Buffers(4096, 16, 2, 64, 16, b.num_pages, len(b.page_table))
    buf.load(b)
    plan = _graph_plan(buf, 4096, b)
    _decode(plan, buf)
    torch.cuda.synchronize()
    assert plan.device_error() == 0
    _check(b, buf, n=1024, seed=5, what="graph decode, 4096 requests")
    assert torch.isfinite(buf.out.float()).all()


def test_graph_kv_beyond_plan_capacity_sets_plan_error():
    """A batch holding more KV than the plan was sized for is refused on the
    device (no units, error word set) instead of overrunning the work list."""
    b = syn.make_batch("kvcap", [1, 1], [40, 90], 8, 2, 64, 16, seed=14)
    buf = Buffers(2, 8, 2, 64, 16, b.num_pages, len(b.page_table))
    buf.load(b)
    plan = _graph_plan(buf, 2, b, max_kv_tokens=64)   # 9 blocks needed, 64 / 16 + 2 = 6 allowed
    _decode(plan, buf)
    torch.cuda.synchronize()
    assert plan.device_error() == 4
    assert len(plan.device_units()) == 0
    assert torch.isnan(buf.out.float()).all()
