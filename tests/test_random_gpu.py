"""GPU parity on random mixed batches: decode requests, prefills on cached
prefixes and requests without queries in one plan, over random head counts,
head dims, page sizes, causal flags and sink settings.  Prefill then decode
run on one stream with the same plan ("GPT-OSS on day 0", section "Sink
Attention"; request model of "Disaggregated prefill and decode", section
"Prefill vs decode performance").  Sampled (row, head) pairs against the fp64
oracle; rows of requests without queries do not exist, and every row is
written exactly once, so the output is finite everywhere."""
import numpy as np
import pytest
import torch

import oracle
from helpers import check_close, make_plan, sample_pairs, syn, to_device

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("seed", range(24))
def test_random_mixed_batch_matches_oracle(seed):
    rng = np.random.default_rng(900 + seed)
    Hkv = int(rng.choice([1, 2, 4, 8]))
    G = int(rng.choice([1, 2, 3, 8, 12, 20]))
    D = int(rng.choice([64, 128]))
    P = int(rng.choice([16, 32, 64, 128]))
    B = int(rng.integers(1, 12))
    kv = rng.integers(1, 3000, size=B)
    kinds = rng.integers(0, 3, size=B)               # 0: decode, 1: prefill, 2: no queries
    qo = np.where(kinds == 0, 1, np.where(kinds == 1, rng.integers(2, 300, size=B), 0))
    qo = np.minimum(qo, kv)
    if qo.sum() == 0:
        qo[0] = 1
    causal = bool(rng.integers(0, 2))
    batch = syn.make_batch(f"rand{seed}", qo.tolist(), kv.tolist(), Hkv * G, Hkv, D, P, causal=causal,
                           with_sinks=bool(rng.integers(0, 4) > 0), seed=900 + seed)
    q, pool, pt, sk = to_device(batch)
    plan = make_plan(batch, pt)
    out = torch.full_like(q, float("nan"))
    lse = torch.full((batch.total_rows, batch.num_qo_heads), float("nan"), device="cuda")
    plan.prefill(q, pool, sk, out, lse)
    plan.decode(q, pool, sk, out, lse)
    torch.cuda.synchronize()
    assert plan.device_error() == 0
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()
    rows, heads = sample_pairs(batch, list(range(batch.total_rows)), 400, seed=seed)
    ref_out, ref_lse = oracle.sink_attention(batch, rows=rows, heads=heads)
    ri = torch.from_numpy(rows).cuda()
    hi = torch.from_numpy(heads).long().cuda()
    check_close(out[ri, hi], lse[ri, hi], ref_out, ref_lse,
                f"random batch {seed}: Hq {Hkv * G}, Hkv {Hkv}, D {D}, P {P}, causal {causal}, qo {qo.tolist()}")
