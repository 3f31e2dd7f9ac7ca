"""CPU checks of the benchmark's accounting: the algorithmic byte and flop
counts it divides by, and the traffic table it reports.

Decode bytes count K and V of every valid token of the decode requests once
(kv_len * Hkv * D * 2 values * 2 bytes); prefill flops count 4 * D per
visible (query, key) pair per query head, the causal mask aligned
bottom-right (query i of a request sees keys j <= kv_len - qo_len + i).
"""
import hashlib
import json
import os

import numpy as np
import pytest

import bench
from helpers import syn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_kv_bytes_counts_decode_tokens_only():
    b = syn.make_batch("mix", [1, 5, 1, 0], [40, 9, 300, 7], 8, 2, 64, 16, seed=3)
    want = (40 + 300) * 2 * 64 * 2 * 2          # decode rows only: K and V, bf16
    assert bench.kv_bytes(b) == want


def test_kv_bytes_headline_batch():
    b = syn.gptoss_decode(0, fill_pool=False)   # same lengths as the timed batch
    assert bench.kv_bytes(b) == int(b.kv_lens.sum()) * 8 * 64 * 4
    assert bench.kv_bytes(b) == 613208064        # the bytes the summaries quote


@pytest.mark.parametrize("causal", [True, False])
def test_prefill_flops_equal_brute_force_pairs(causal):
    qo, kv = [3, 1, 7, 4], [5, 6, 7, 10]
    b = syn.make_batch("pf", qo, kv, 4, 2, 64, 16, causal=causal, seed=1)
    pairs = 0
    for q_len, k_len in zip(qo, kv):
        if q_len <= 1:
            continue                               # decode rows are not prefill work
        for i in range(q_len):
            for j in range(k_len):
                if not causal or j <= k_len - q_len + i:
                    pairs += 1
    assert bench.prefill_flops(b) == pairs * 4 * 4 * 64


def test_job_throughput_single_rank():
    assert bench.job_throughput(1e9, 10, 2.0, 1) == pytest.approx(5.0)


def test_traffic_table_is_keyed_to_the_current_sources():
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        table = json.load(f)
    for key, src in (("decode_gptoss", "decode.cu"), ("prefill_gptoss", "prefill.cu")):
        entry = table[key]
        assert entry["dram_bytes_per_launch"] > 0
        with open(os.path.join(ROOT, "paged_kv_attention_sink_gb300", "csrc", src), "rb") as f:
            sha = hashlib.sha256(f.read()).hexdigest()
        # bench reports the entry only while the kernel source is the one captured
        assert (bench.traffic_for(src, key) is not None) == (sha == entry["source_sha256"])
    # DRAM reads of the decode capture stay within 1% of the algorithmic bytes
    # (every KV byte read once); reads plus writes (partial states, out, lse)
    # within 2%
    d = table["decode_gptoss"]
    assert d["dram_read_bytes_per_launch"] <= 1.01 * d["algorithmic_bytes_per_launch"]
    assert d["dram_bytes_per_launch"] <= 1.02 * d["algorithmic_bytes_per_launch"]


def test_sample_prefill_flops_over_all_rows_equals_total():
    """The CPU baseline's prefill sample is counted row by row; over every
    row it must give the whole launch's algorithmic flops."""
    for batch in (syn.make_batch("cnt", [40, 7, 300], [40, 100, 1000], 4, 2, 64, 16, seed=2),
                  syn.mixed(0, fill_pool=False)):
        rows = np.arange(batch.total_rows)
        prefill = [r for r in rows if batch.qo_lens[np.searchsorted(batch.qo_indptr, r, side="right") - 1] > 1]
        assert bench.sample_prefill_flops(batch, prefill) == bench.prefill_flops(batch)
