"""Writes tests/golden/tiny_decode_seed0.json.

Regression fixture for the seeded input generator and the fp64 oracle on the
two-request tiny decode workload (kv_len 256 and 97, Hq 8 / Hkv 2, D 64,
16-token pages in a 64-page pool).  Every stored value comes from
``paged_kv_attention_sink_gb300.synthetic`` (input checksums) or from
``oracle`` (outputs); nothing here comes from the CUDA path.

Run from the repository root:  python tests/golden/make_golden.py
"""
import hashlib
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from paged_kv_attention_sink_gb300 import synthetic as syn  # noqa: E402


def checksums(batch):
    return {name: hashlib.sha256(getattr(batch, name).tobytes()).hexdigest()
            for name in ("q", "kv_pool", "page_table", "last_page_len", "sinks")}


def main():
    batch = syn.tiny_decode(0)
    out, lse = oracle.sink_attention(batch)
    picks = [(0, 0, 0), (0, 3, 17), (0, 7, 63), (1, 0, 5), (1, 4, 40), (1, 6, 62)]
    data = {
        "workload": "tiny_decode seed 0",
        "definition": "sink attention as in 'GPT-OSS on day 0' (Perplexity), section 'Sink Attention'",
        "checksums": checksums(batch),
        "out": [[r, h, d, float(out[r, h, d])] for r, h, d in picks],
        "lse": [[r, h, float(lse[r, h])] for r in range(2) for h in range(8)],
    }
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_decode_seed0.json")
    with open(path, "w") as f:
        json.dump(data, f, indent=1)
        f.write("\n")


if __name__ == "__main__":
    main()
