"""The multi-rank bench path on CPU: two gloo ranks, as torchrun would start
them.  The attention path shards by request with no exchange (replicas), so
the only collectives are the bench's barrier and the max over ranks of the
timed region; these tests run them for real on world_size 2.
"""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out_q):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "WORLD_SIZE": str(world),
                       "RANK": str(rank), "LOCAL_RANK": str(rank)})
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    w, r, _ = bench.dist_setup("reference")           # gloo
    bench.barrier(w)
    slowest = bench.max_over_ranks(1.0 + r, w)        # rank 1 is the slow one
    gbs = bench.job_throughput(1e9, 10, 2.0 + r, w)   # 2 ranks x 10 steps x 1 GB over 3 s
    from paged_kv_attention_sink_gb300 import synthetic as syn
    b = syn.gptoss_decode(seed=r, batch=4)            # replicas draw different batches
    out_q.put((r, w, slowest, gbs, int(b.kv_lens.sum())))
    bench.barrier(w)
    dist.destroy_process_group()


def test_two_gloo_ranks_barrier_and_max():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[0] for r in res] == [0, 1] and all(r[1] == 2 for r in res)
    assert all(r[2] == pytest.approx(2.0) for r in res)        # max over ranks, seen by both
    assert all(r[3] == pytest.approx(2 * 10 * 1e9 / 3.0 / 1e9) for r in res)
    assert res[0][4] != res[1][4]                              # seed = rank


def test_reference_arm_runs_on_rank_zero_only(tmp_path):
    """`bench.py --impl reference` under a 2-rank launch: rank 0 prints the
    reference line, the other rank exits without work."""
    import json
    import subprocess
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", f"--master-port={port}", os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle"
