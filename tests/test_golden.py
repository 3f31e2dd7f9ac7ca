"""Regression pin: the seeded generator and the oracle still produce the values
stored by tests/golden/make_golden.py for the tiny decode workload."""
import json
import os

import numpy as np

import oracle
from paged_kv_attention_sink_gb300 import synthetic as syn

HERE = os.path.dirname(os.path.abspath(__file__))


def test_tiny_decode_golden():
    import hashlib
    with open(os.path.join(HERE, "golden", "tiny_decode_seed0.json")) as f:
        gold = json.load(f)
    batch = syn.tiny_decode(0)
    for name, digest in gold["checksums"].items():
        assert hashlib.sha256(getattr(batch, name).tobytes()).hexdigest() == digest, name
    out, lse = oracle.sink_attention(batch)
    for r, h, d, v in gold["out"]:
        assert abs(out[r, h, d] - v) <= 1e-12
    for r, h, v in gold["lse"]:
        assert abs(lse[r, h] - v) <= 1e-12
    assert np.all(np.isfinite(out))
