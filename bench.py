#!/usr/bin/env python
"""Benchmark of the paged sink-attention hot path on GB300.

Headline (`value`): decode attention on the gpt-oss-120b-shaped batch (64
requests, kv_len ~ U[1024, 8192], Hq 64 / Hkv 8, head_dim 64, 16-token HND
pages, split-KV), reported as algorithmic KV bytes read per second (GB/s):
sum over requests of kv_len * Hkv * head_dim * 2 (K and V) * 2 bytes, divided
by the device time of one attn_decode launch (which includes the split-KV
merge).  Inputs are resident in HBM; the KV pool (about 750 MB) is larger
than L2, and L2 is also flushed before every timed step, outside the timed
events: a 256 MB memset, then a read of another 256 MB buffer, so that the
timed kernel starts with a cold L2 that holds no dirty lines (otherwise the
write-back of the memset's ~129 MB of dirty lines lands inside the timed
kernel and is charged to it).  The prefill leg (gpt-oss-120b-shaped ragged causal
prefill) is reported in TFLOP/s of visible (query, key) pairs x 4 * head_dim.
`value` and `ms_per_step` use the total of the K timed steps (the mean);
`ms_per_step_median` gives the median step beside it.

One step = one pass of the hot path over one batch: the plan is built once
per batch (host), then attn_decode runs (and attn_prefill for the prefill
leg).  `e2e` times the same decode through the public API from pinned host
buffers: H2D of q and the page table, planning and work-list upload, the
launch, and D2H of out and lse, every step, with up to three steps in
flight (the host plans step k while the GPU runs the steps before it) and the
copies on their own streams (they overlap the neighbouring steps' decodes).

Multi-GPU: the path shards by request with no exchange, so N ranks run N
independent replicas ("scaling": "weak"); value = all ranks' bytes / max
rank time.  `--impl reference` times the CPU fp64 oracle instead.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "decode attn KV-read GB/s vs ~8 TB/s HBM; prefill attn TFLOP/s vs bf16 peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def kv_bytes(batch, rows_only=None):
    """Algorithmic KV bytes of the decode requests (K and V of every valid token)."""
    per_tok = batch.num_kv_heads * batch.head_dim * 2 * 2
    kv = batch.kv_lens[batch.qo_lens == 1] if rows_only is None else rows_only
    return int(np.sum(kv)) * per_tok


def sample_prefill_flops(batch, rows):
    """Algorithmic flops of the given query rows (all heads): 4 * D per
    visible (query, key) pair per head, as prefill_flops counts them."""
    pairs = 0
    for r in rows:
        b = int(np.searchsorted(batch.qo_indptr, r, side="right") - 1)
        qo, kv = int(batch.qo_lens[b]), int(batch.kv_lens[b])
        i = int(r - batch.qo_indptr[b])
        pairs += min(kv, kv - qo + i + 1) if batch.causal else kv
    return pairs * batch.num_qo_heads * 4 * batch.head_dim


def prefill_flops(batch):
    pairs = 0
    for b in range(batch.batch_size):
        qo, kv = int(batch.qo_lens[b]), int(batch.kv_lens[b])
        if qo > 1:
            prefix = kv - qo
            pairs += qo * prefix + qo * (qo + 1) // 2 if batch.causal else qo * kv
    return pairs * batch.num_qo_heads * 4 * batch.head_dim


# ----------------------------------------------------------------- clocks
class NvmlSampler:
    """Samples the SM clock, its maximum, the board power and the active
    clock-event reasons every few ms from a thread, through NVML (read-only
    queries on the driver's libnvidia-ml), so that even a short timed region
    gets samples.  Falls back to an nvidia-smi loop if NVML is unavailable."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, uuid: str, period_s: float = 0.0005):
        self.uuid, self.period = uuid, period_s
        self.samples, self.thread, self.stop_flag = [], None, False
        self.nvml = self.handle = None
        self.fallback = None

    def _open(self):
        import ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        h = ctypes.c_void_p()
        if lib.nvmlDeviceGetHandleByUUID(self.uuid.encode(), ctypes.byref(h)) != 0:
            raise RuntimeError("no NVML handle for " + self.uuid)
        self.nvml, self.handle = lib, h
        self.reason_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")

    def _poll(self):
        import ctypes
        clk, mx, mw, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        while not self.stop_flag:
            ok = (self.nvml.nvmlDeviceGetClockInfo(self.handle, 1, ctypes.byref(clk)) == 0 and
                  self.nvml.nvmlDeviceGetMaxClockInfo(self.handle, 1, ctypes.byref(mx)) == 0)
            if ok:
                p = mw.value / 1000.0 if self.nvml.nvmlDeviceGetPowerUsage(self.handle, ctypes.byref(mw)) == 0 else None
                r = rs.value if self.reason_fn(self.handle, ctypes.byref(rs)) == 0 else 0
                self.samples.append((float(clk.value), float(mx.value), p, int(r)))
            time.sleep(self.period)

    def start(self):
        import threading
        try:
            self._open()
        except Exception:
            self.fallback = ClockSampler(self.uuid)
            self.fallback.start()
            return
        self.thread = threading.Thread(target=self._poll, daemon=True)
        self.thread.start()

    def stop(self):
        if self.fallback is not None:
            return self.fallback.stop()
        self.stop_flag = True
        self.thread.join(timeout=5)
        try:
            self.nvml.nvmlShutdown()
        except Exception:
            pass
        sm = [x[0] for x in self.samples]
        smax = [x[1] for x in self.samples]
        pw = [x[2] for x in self.samples if x[2] is not None]
        reasons = sorted({name for x in self.samples for bit, name in self.REASONS.items() if x[3] & bit})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "sm_min_mhz": min(sm) if sm else None, "power_w_median": statistics.median(pw) if pw else None,
                "reasons": reasons, "samples": len(sm), "source": "nvml"}


class ClockSampler:
    """nvidia-smi loop (fallback sampler)."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = [l.strip().split(", ") for l in self.file.read().splitlines() if l.strip()]
        os.unlink(self.file.name)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[0]))
                smax.append(float(r[1]))
                for name, v in zip(names, r[4:8]):
                    if v.strip().lower() == "active":
                        reasons.add(name)
            except (ValueError, IndexError):
                continue
        busy = [s for s in sm if smax and s > 0.5 * max(smax)] or sm
        return {"sm_mhz": statistics.median(busy) if busy else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm), "source": "nvidia-smi"}


# -------------------------------------------------------------- distributed
def dist_setup(impl):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        backend = "nccl" if impl == "ours" else "gloo"
        if backend == "nccl":
            import torch
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    """Max of a per-rank scalar over all ranks (the job's time is its slowest rank's)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    device = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(bytes_per_rank_step, steps, rank_seconds, world):
    """Whole-job throughput of N replicas (GB/s): the units all ranks processed
    over the slowest rank's time.  Collective when world > 1."""
    return world * bytes_per_rank_step * steps / max_over_ranks(rank_seconds, world) / 1e9


def headline_config(batch, world):
    """The headline workload, as both arms report it (static: no timings)."""
    return {"workload": "gptoss_decode", "batch": batch.batch_size, "kv_len": "U[1024,8192]",
            "Hq": batch.num_qo_heads, "Hkv": batch.num_kv_heads, "head_dim": batch.head_dim,
            "page_size": batch.page_size, "split_kv": True, "sinks": batch.sinks is not None,
            "kv_bytes_per_step": kv_bytes(batch),
            "l2": "flushed before every timed step (256 MB memset, then a 256 MB read: cold L2, no dirty lines)",
            "parallelism": f"replicas x{world}"}


# ----------------------------------------------------------- reference arm
def run_reference(args, world, rank):
    if rank != 0:
        return
    import oracle
    from paged_kv_attention_sink_gb300 import synthetic as syn
    oracle.build()
    batch = syn.gptoss_decode(0)
    cores = os.cpu_count() or 1
    # Each step: the oracle over a fixed sample of 8 requests (all 64 heads).
    rows = np.arange(8, dtype=np.int64)
    rr = np.repeat(rows, batch.num_qo_heads)
    hh = np.tile(np.arange(batch.num_qo_heads, dtype=np.int32), len(rows))
    sample_bytes = kv_bytes(batch, rows_only=batch.kv_lens[:8])
    for _ in range(args.warmup):
        oracle.sink_attention(batch, rows=rr, heads=hh, n_threads=cores)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.sink_attention(batch, rows=rr, heads=hh, n_threads=cores)
    dt = time.perf_counter() - t0
    value = sample_bytes * args.steps / dt / 1e9
    sample = "gptoss_decode seed 0, requests 0-7 (all 64 query heads), fp64 C oracle per step"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": headline_config(batch, world),
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


# ---------------------------------------------------------------- our arm
_cudart = None


def cudart():
    """The CUDA runtime libattn.so links, for the end-to-end loop's copies,
    events and stream waits (ctypes signatures set once)."""
    global _cudart
    if _cudart is None:
        import ctypes.util
        rt = None
        for name in ("libcudart.so.13", "libcudart.so.12", ctypes.util.find_library("cudart")):
            if not name:
                continue
            try:
                rt = ctypes.CDLL(name)
                break
            except OSError:
                continue
        if rt is None:
            raise RuntimeError("the CUDA runtime library was not found")
        vp, sz = ctypes.c_void_p, ctypes.c_size_t
        for fn, args in (("cudaMemcpyAsync", [vp, vp, sz, ctypes.c_int, vp]), ("cudaEventRecord", [vp, vp]),
                         ("cudaStreamWaitEvent", [vp, vp, ctypes.c_uint]), ("cudaEventSynchronize", [vp]),
                         ("cudaEventCreateWithFlags", [ctypes.POINTER(vp), ctypes.c_uint]),
                         ("cudaEventDestroy", [vp]), ("cudaGetLastError", [])):
            f = getattr(rt, fn)
            f.argtypes, f.restype = args, ctypes.c_int
        _cudart = rt
    return _cudart


def rt_check(status, what):
    if status != 0:
        raise RuntimeError(f"{what}: CUDA error {status}")


def traffic_for(kernel_file, key):
    """DRAM bytes per launch from a committed ncu summary, if the kernel source
    is unchanged since the capture (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        table = json.load(f)
    entry = table.get(key)
    if not entry:
        return None
    src = os.path.join(ROOT, "paged_kv_attention_sink_gb300", "csrc", kernel_file)
    with open(src, "rb") as f:
        sha = hashlib.sha256(f.read()).hexdigest()
    return entry["dram_bytes_per_launch"] if entry.get("source_sha256") == sha else None


class L2Flush:
    """Evicts L2 between timed steps: a 256 MB memset (writes) followed by a
    read of a second 256 MB buffer, so the lines left in L2 are clean."""

    def __init__(self, dev):
        import torch
        self.w = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
        self.r = torch.ones(64 * 1024 * 1024, dtype=torch.float32, device=dev)

    def __call__(self):
        self.w.zero_()
        self.r.sum()



def leg_steps(args):
    """Launches timed by each side leg: at least 50, whatever --steps says."""
    return max(50, args.steps // 10)


def timed_leg(fn, steps, flush, stream, gpu_id):
    """time_device with an NVML clock record of its own."""
    sampler = NvmlSampler(gpu_id)
    sampler.start()
    times = time_device(fn, steps, flush, stream)
    return times, sampler.stop()


def time_device(fn, steps, flush, stream):
    import torch
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for i in range(steps):
        flush()
        starts[i].record(stream)
        fn()
        ends[i].record(stream)
    torch.cuda.synchronize()
    return [s.elapsed_time(e) for s, e in zip(starts, ends)]


def run_ours(args, world, rank, local):
    import torch
    from paged_kv_attention_sink_gb300 import build as libbuild
    libbuild.build()
    from paged_kv_attention_sink_gb300 import binding, synthetic as syn

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    peaks, peak_src = load_peaks()

    def to_dev(batch):
        q = torch.from_numpy(batch.q.view(np.int16)).view(torch.bfloat16).to(dev)
        kv = torch.from_numpy(batch.kv_pool.view(np.int16)).view(torch.bfloat16).to(dev)
        pt = torch.from_numpy(batch.page_table).to(dev)
        sk = None if batch.sinks is None else torch.from_numpy(batch.sinks).to(dev)
        return q, kv, pt, sk

    def plan_of(batch, pt, workspace=None, stream=None):
        return binding.Plan(batch.qo_indptr, batch.kv_indptr, pt, batch.last_page_len,
                            batch.num_qo_heads, batch.num_kv_heads, batch.head_dim, batch.page_size,
                            causal=batch.causal, sm_scale=batch.sm_scale, num_pages=batch.num_pages,
                            workspace=workspace, stream=stream)

    flush = L2Flush(dev)
    props = torch.cuda.get_device_properties(dev)
    gpu_id = getattr(props, "uuid", None)
    gpu_id = ("GPU-" + str(gpu_id)) if gpu_id is not None and not str(gpu_id).startswith("GPU-") else str(gpu_id or local)

    # ---- decode (headline)
    batch = syn.gptoss_decode(seed=rank)
    q, kv, pt, sinks = to_dev(batch)
    t0 = time.perf_counter()
    plan = plan_of(batch, pt)
    plan_first_us = (time.perf_counter() - t0) * 1e6   # includes the workspace allocation
    # Steady state: re-plan into the same workspace (host planning + the work
    # list's upload), as a serving loop does every step.
    plan_times = []
    for _ in range(50):
        t0 = time.perf_counter()
        plan_of(batch, pt, plan.workspace)
        plan_times.append((time.perf_counter() - t0) * 1e6)
    plan_us = statistics.median(plan_times)
    out = torch.empty_like(q)
    lse = torch.empty(batch.total_rows, batch.num_qo_heads, device=dev)
    dec = lambda: plan.decode(q, kv, sinks, out, lse)
    for _ in range(args.warmup):
        flush()
        dec()
    torch.cuda.synchronize()
    if plan.device_error():
        raise RuntimeError("decode kernel recorded a device error")

    sampler = NvmlSampler(gpu_id)
    sampler.start()
    barrier(world)
    torch.cuda.synchronize()
    times = time_device(dec, args.steps, flush, stream)
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop()
    total_ms = max_over_ranks(sum(times), world)
    bytes_step = kv_bytes(batch)
    value = world * bytes_step * args.steps / (total_ms / 1e3) / 1e9   # = job_throughput(...)
    mean_s = sum(times) / len(times) / 1e3
    achieved = bytes_step / mean_s / 1e9
    peak = float(peaks["hbm_gbs"])
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "traffic": traffic_for("decode.cu", "decode_gptoss"),
                "kernel": "decode_sink_attn_kernel<64,false>", "peak_source": peak_src,
                "frac_of_nominal_8TBps": achieved / 8000.0}

    # ---- the same decode as one replay of a captured CUDA graph (device-built
    # work list + persistent decode over it), inputs resident
    graph = None
    try:
        gplan = binding.GraphPlan(batch.batch_size, batch.num_qo_heads, batch.num_kv_heads, batch.head_dim,
                                  batch.page_size, pt, batch.num_pages, sm_scale=batch.sm_scale)
        g_indptr = torch.from_numpy(batch.kv_indptr).to(dev)
        g_lpl = torch.from_numpy(batch.last_page_len).to(dev)
        g_b = torch.tensor([batch.batch_size], dtype=torch.int32, device=dev)
        gdec = lambda: gplan.decode(q, kv, g_indptr, g_lpl, g_b, sinks, out, lse)
        gdec()
        torch.cuda.synchronize()
        cg = torch.cuda.CUDAGraph()
        cs = torch.cuda.Stream()
        cs.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(cs):
            with torch.cuda.graph(cg, stream=cs):
                gdec()
        torch.cuda.current_stream().wait_stream(cs)
        for _ in range(args.warmup):
            cg.replay()
        gsteps = leg_steps(args)
        gtimes, gclocks = timed_leg(cg.replay, gsteps, flush, stream, gpu_id)
        gmean = sum(gtimes) / len(gtimes) / 1e3
        if gplan.device_error():
            raise RuntimeError("graph decode recorded a device error")
        # Plans for up to 128 requests are built inside the persistent decode
        # grid (one kernel per replay); larger ones by a planner kernel first.
        per_replay = 1 if batch.batch_size <= 128 else 2
        graph = {"workload": "gptoss_decode, one CUDA-graph replay (device-built work list + persistent decode)",
                 "value": bytes_step / gmean / 1e9, "unit": "GB/s", "ms_per_step": gmean * 1e3,
                 "frac_of_hbm_peak": bytes_step / gmean / 1e9 / float(peaks["hbm_gbs"]),
                 "steps": gsteps, "launches": per_replay * gsteps, "clocks": gclocks}
    except binding.AttnError as e:
        graph = {"unavailable": str(e)}

    # ---- e2e through the public API from pinned host buffers.  Up to three
    # steps are in flight, as a serving loop would run them: the host plans and
    # launches step k (H2D of its q and page table, attn_plan + workspace
    # upload, attn_decode, D2H of its out and lse) while the GPU still runs the
    # steps before it, and waits for a step's read-back before reusing its
    # buffers (three slots, so host-side jitter of one step does not stall
    # the GPU).  The
    # uploads run on one copy stream and the read-backs on another, ordered
    # against the decode on the compute stream by events, so a step's copies
    # overlap its neighbours' decodes.
    # q and the page table share one pinned host buffer and one device buffer
    # per slot (one upload); out and lse likewise (one read-back).  The copies,
    # events and stream waits go straight to the CUDA runtime the library
    # links (ctypes), as a serving loop in C would make them: torch's stream
    # switching and copy dispatch cost more host time per step than the
    # planner itself, and with three steps in flight the host loop, not the
    # GPU, then set the pace.
    q_bytes, pt_bytes = q.numel() * 2, pt.numel() * 4
    out_bytes, lse_bytes = out.numel() * 2, lse.numel() * 4
    in_h = torch.empty(q_bytes + pt_bytes, dtype=torch.uint8).pin_memory()
    in_h[:q_bytes].copy_(torch.from_numpy(batch.q.view(np.uint8).reshape(-1)))
    in_h[q_bytes:].copy_(torch.from_numpy(batch.page_table.view(np.uint8).reshape(-1)))
    e2e_slots = []
    for _ in range(3):
        d_in = torch.empty(q_bytes + pt_bytes, dtype=torch.uint8, device=dev)
        d_res = torch.empty(out_bytes + lse_bytes, dtype=torch.uint8, device=dev)
        e2e_slots.append({
            "in": d_in, "q": d_in[:q_bytes].view(torch.bfloat16).view(q.shape),
            "pt": d_in[q_bytes:].view(torch.int32),
            "res": d_res, "out": d_res[:out_bytes].view(torch.bfloat16).view(out.shape),
            "lse": d_res[out_bytes:].view(torch.float32).view(lse.shape),
            "res_h": torch.empty(out_bytes + lse_bytes, dtype=torch.uint8).pin_memory(),
            "plan": None, "ws": torch.empty(plan.info()["workspace_bytes"], dtype=torch.uint8, device=dev)})
    # A fixed 500 steps (about 50 ms), whatever --steps says: with three steps
    # in flight, a short region is dominated by filling and draining the
    # pipeline.
    e2e_steps = 500
    up_stream, down_stream = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    rt = cudart()
    s_up, s_down, s_main = (ctypes.c_void_p(x.cuda_stream) for x in (up_stream, down_stream, stream))
    for sl in e2e_slots:
        for name in ("ev", "uploaded", "decoded"):
            ev = ctypes.c_void_p()
            rt_check(rt.cudaEventCreateWithFlags(ctypes.byref(ev), 2), "cudaEventCreateWithFlags")   # no timing
            sl[name] = ev
        sl["in_p"], sl["res_p"] = ctypes.c_void_p(sl["in"].data_ptr()), ctypes.c_void_p(sl["res"].data_ptr())
        sl["res_h_p"] = ctypes.c_void_p(sl["res_h"].data_ptr())
    in_h_p, n_in, n_res = ctypes.c_void_p(in_h.data_ptr()), in_h.numel(), e2e_slots[0]["res_h"].numel()
    torch.cuda.synchronize()   # the slots' buffers exist before other streams touch them

    def e2e_step(k):
        sl = e2e_slots[k % 3]
        if sl["plan"] is not None:
            rt.cudaEventSynchronize(sl["ev"])   # step k-3's result is on the host; its buffers are free
        rt.cudaMemcpyAsync(sl["in_p"], in_h_p, n_in, 1, s_up)              # host to device
        sl["plan"] = plan_of(batch, sl["pt"], sl["ws"], stream=up_stream)  # binds: the work list goes up on up_stream
        rt.cudaEventRecord(sl["uploaded"], s_up)
        rt.cudaStreamWaitEvent(s_main, sl["uploaded"], 0)
        sl["plan"].decode(sl["q"], kv, sinks, sl["out"], sl["lse"], stream=stream)
        rt.cudaEventRecord(sl["decoded"], s_main)
        rt.cudaStreamWaitEvent(s_down, sl["decoded"], 0)
        rt.cudaMemcpyAsync(sl["res_h_p"], sl["res_p"], n_res, 2, s_down)  # device to host
        rt.cudaEventRecord(sl["ev"], s_down)

    for k in range(3):
        e2e_step(k)
    torch.cuda.synchronize()
    barrier(world)
    t0 = time.perf_counter()
    for k in range(e2e_steps):
        e2e_step(k)
    torch.cuda.synchronize()
    e2e_s = max_over_ranks(time.perf_counter() - t0, world)
    rt_check(rt.cudaGetLastError(), "e2e loop")
    for sl in e2e_slots:
        for name in ("ev", "uploaded", "decoded"):
            rt.cudaEventDestroy(sl[name])
    if not torch.equal(e2e_slots[0]["res_h"], e2e_slots[1]["res_h"]):
        raise RuntimeError("end-to-end decode steps on the same batch disagree")
    units = plan.info()["num_decode_units"]
    h2d = in_h.numel() + units * 48
    d2h = e2e_slots[0]["res_h"].numel()
    e2e = {"value": world * bytes_step * e2e_steps / e2e_s / 1e9, "unit": "GB/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
           "ms_per_step": e2e_s * 1e3 / e2e_steps, "steps_in_flight": 3,
           "streams": "uploads, decode and read-backs on three streams, ordered by events"}

    # ---- prefill leg (TFLOP/s), if the kernel is available
    prefill = None
    launches = args.steps + (graph.get("launches", 0) if graph else 0)
    if not args.no_prefill:
        pbatch = syn.gptoss_prefill(seed=rank)
        pq, pkv, ppt, psk = to_dev(pbatch)
        pplan = plan_of(pbatch, ppt)
        pout = torch.empty_like(pq)
        plse = torch.empty(pbatch.total_rows, pbatch.num_qo_heads, device=dev)
        pre = lambda: pplan.prefill(pq, pkv, psk, pout, plse)
        try:
            pre()
            torch.cuda.synchronize()
        except binding.AttnError as e:
            prefill = {"unavailable": str(e)}
        if prefill is None:
            for _ in range(args.warmup):
                pre()
            torch.cuda.synchronize()
            psteps = leg_steps(args)
            ptimes, pclocks = timed_leg(pre, psteps, flush, stream, gpu_id)
            pmean = sum(ptimes) / len(ptimes) / 1e3
            flops = prefill_flops(pbatch)
            tf = flops / pmean / 1e12
            ppeak = float(peaks["bf16_tflops"])
            mhz = pclocks.get("sm_mhz")
            prefill = {"workload": "gptoss_prefill", "value": tf, "unit": "TFLOP/s",
                       "ms_per_step": pmean * 1e3, "steps": psteps, "clocks": pclocks,
                       # time x median SM clock: the launch in SM cycles, comparable across clocks
                       "sm_cycles_per_step": pmean * mhz * 1e6 if mhz else None,
                       "flops": flops,
                       "roofline": {"bound": "tensor", "achieved": tf, "peak": ppeak,
                                    "unit": "TFLOP/s", "frac": tf / ppeak,
                                    "traffic": traffic_for("prefill.cu", "prefill_gptoss"),
                                    "peak_source": peak_src}}
            launches += psteps

    # ---- ragged (non-paged) prefill on the same batch: contiguous K / V
    ragged = None
    if not args.no_prefill and prefill is not None and "unavailable" not in prefill:
        P = pbatch.page_size
        ks, vs = [], []
        for b in range(pbatch.batch_size):
            t = np.arange(int(pbatch.kv_lens[b]))
            pages = pbatch.page_table[pbatch.kv_indptr[b] + t // P]
            ks.append(pbatch.kv_pool[pages, 0, :, t % P, :])
            vs.append(pbatch.kv_pool[pages, 1, :, t % P, :])
        rk = torch.from_numpy(np.concatenate(ks).view(np.int16)).view(torch.bfloat16).to(dev)
        rv = torch.from_numpy(np.concatenate(vs).view(np.int16)).view(torch.bfloat16).to(dev)
        rplan = binding.RaggedPlan(pbatch.qo_indptr, np.concatenate([[0], np.cumsum(pbatch.kv_lens)]),
                                   pbatch.num_qo_heads, pbatch.num_kv_heads, pbatch.head_dim,
                                   causal=pbatch.causal, sm_scale=pbatch.sm_scale, device=dev)
        rag = lambda: rplan.prefill(pq, rk, rv, psk, pout, plse)
        for _ in range(args.warmup):
            rag()
        rsteps = leg_steps(args)
        rtimes, rclocks = timed_leg(rag, rsteps, flush, stream, gpu_id)
        rmean = sum(rtimes) / len(rtimes) / 1e3
        rtf = prefill_flops(pbatch) / rmean / 1e12
        ragged = {"workload": "gptoss_prefill, contiguous K/V (no cache)", "value": rtf, "unit": "TFLOP/s",
                  "ms_per_step": rmean * 1e3, "frac_of_bf16_peak": rtf / float(peaks["bf16_tflops"]),
                  "steps": rsteps, "clocks": rclocks}
        launches += rsteps

    # ---- KV-cache legs (HBM copies): the step's append on the prefill batch,
    # and a head-slice pack of half the heads of every page of the decode pool.
    kvcache = None
    if not args.no_prefill and prefill is not None and "unavailable" not in prefill:
        k_new, v_new = syn.new_kv_rows(pbatch, seed=rank)
        kd = torch.from_numpy(k_new.view(np.int16)).view(torch.bfloat16).to(dev)
        vd = torch.from_numpy(v_new.view(np.int16)).view(torch.bfloat16).to(dev)
        app = lambda: pplan.append_kv(kd, vd, pkv)
        for _ in range(args.warmup):
            app()
        asteps = leg_steps(args)
        atimes, aclocks = timed_leg(app, asteps, flush, stream, gpu_id)
        amean = sum(atimes) / len(atimes) / 1e3
        abytes = 2 * 2 * kd.numel() * 2                       # K and V rows, read once + written once
        ids = torch.from_numpy(np.unique(batch.page_table)).to(dev)
        nh = batch.num_kv_heads // 2
        buf = torch.empty((ids.numel(), 2, nh, batch.page_size, batch.head_dim), dtype=torch.bfloat16, device=dev)
        pk = lambda: binding.attn_pack_kv_heads(kv, ids, 0, nh, buf=buf)
        for _ in range(args.warmup):
            pk()
        ktimes, kclocks = timed_leg(pk, asteps, flush, stream, gpu_id)
        kmean = sum(ktimes) / len(ktimes) / 1e3
        kbytes = 2 * buf.numel() * 2                           # slice read once + buffer written once
        peak = float(peaks["hbm_gbs"])
        kvcache = {
            "append": {"workload": "gptoss_prefill rows (new K/V of every query row)", "bytes": abytes,
                       "us": amean * 1e6, "value": abytes / amean / 1e9, "unit": "GB/s",
                       "frac_of_hbm_peak": abytes / amean / 1e9 / peak, "steps": asteps, "clocks": aclocks},
            "pack_heads": {"workload": f"gptoss_decode pool, heads [0,{nh}) of {ids.numel()} pages",
                           "bytes": kbytes, "us": kmean * 1e6, "value": kbytes / kmean / 1e9, "unit": "GB/s",
                           "frac_of_hbm_peak": kbytes / kmean / 1e9 / peak, "steps": asteps,
                           "clocks": kclocks},
        }
        launches += 2 * asteps

    # ---- the other serving shapes: Qwen3-shaped long-context decode (no
    # sinks) and the mixed batch (chunked prefill on cached prefixes + 256
    # decode requests, one plan, prefill then decode on one stream).
    others = None
    if not args.no_prefill and prefill is not None and "unavailable" not in prefill:
        others = {}
        hbm = float(peaks["hbm_gbs"])
        tc = float(peaks["bf16_tflops"])
        osteps = leg_steps(args)
        def pool_on_device(b_):
            # N(0,1) bf16, drawn on the GPU (seeded): these legs only time kernels
            g = torch.Generator(device=dev)
            g.manual_seed(1000 + rank)
            pool = torch.empty((b_.num_pages, 2, b_.num_kv_heads, b_.page_size, b_.head_dim), dtype=torch.bfloat16,
                               device=dev)
            flat = pool.view(-1)
            for s0 in range(0, flat.numel(), 1 << 28):
                n = min(1 << 28, flat.numel() - s0)
                flat[s0:s0 + n] = torch.randn(n, generator=g, device=dev, dtype=torch.float32).to(torch.bfloat16)
            return pool

        def to_dev_gen(b_):
            q_ = torch.from_numpy(b_.q.view(np.int16)).view(torch.bfloat16).to(dev)
            pt_ = torch.from_numpy(b_.page_table).to(dev)
            sk_ = None if b_.sinks is None else torch.from_numpy(b_.sinks).to(dev)
            return q_, pool_on_device(b_), pt_, sk_

        qb = syn.qwen_decode(seed=rank, fill_pool=False)
        qq, qkv, qpt, qsk = to_dev_gen(qb)
        qplan = plan_of(qb, qpt)
        qout = torch.empty_like(qq)
        qlse = torch.empty(qb.total_rows, qb.num_qo_heads, device=dev)
        qdec = lambda: qplan.decode(qq, qkv, qsk, qout, qlse)
        for _ in range(args.warmup):
            qdec()
        qtimes, qclocks = timed_leg(qdec, osteps, flush, stream, gpu_id)
        qmean = sum(qtimes) / len(qtimes) / 1e3
        qbytes = kv_bytes(qb)
        others["qwen_decode"] = {
            "workload": "qwen_decode: 128 requests, kv_len log-U[2048,32768], Hq 64, Hkv 4, D 128, P 64, no sinks"
                        " (KV pool drawn on the GPU)",
            "bytes": qbytes, "ms_per_step": qmean * 1e3, "value": qbytes / qmean / 1e9, "unit": "GB/s",
            "frac_of_hbm_peak": qbytes / qmean / 1e9 / hbm, "steps": osteps, "clocks": qclocks}
        launches += osteps
        del qq, qkv, qpt, qout, qlse, qplan
        mb = syn.mixed(seed=rank, fill_pool=False)
        mq, mkv, mpt, msk = to_dev_gen(mb)
        mplan = plan_of(mb, mpt)
        mout = torch.empty_like(mq)
        mlse = torch.empty(mb.total_rows, mb.num_qo_heads, device=dev)
        mpre = lambda: mplan.prefill(mq, mkv, msk, mout, mlse)
        mdec = lambda: mplan.decode(mq, mkv, msk, mout, mlse)
        for _ in range(args.warmup):
            mpre()
            mdec()
        mp, mpclocks = timed_leg(mpre, osteps, flush, stream, gpu_id)
        md, mdclocks = timed_leg(mdec, osteps, flush, stream, gpu_id)
        mboth, mbclocks = timed_leg(lambda: (mpre(), mdec()), osteps, flush, stream, gpu_id)
        mp_s, md_s, mb_s = (sum(t) / len(t) / 1e3 for t in (mp, md, mboth))
        mflops, mbytes = prefill_flops(mb), kv_bytes(mb)
        ideal = mflops / (tc * 1e12) + mbytes / (hbm * 1e9)
        others["mixed"] = {
            "workload": "mixed: 4 prefills (qo 2048 on prefixes 0/2048/4096/8192) + 256 decodes (kv U[512,16384])"
                        " (KV pool drawn on the GPU)",
            "prefill_tflops": mflops / mp_s / 1e12, "prefill_frac_of_bf16_peak": mflops / mp_s / 1e12 / tc,
            "decode_gbs": mbytes / md_s / 1e9, "decode_frac_of_hbm_peak": mbytes / md_s / 1e9 / hbm,
            "both_ms": mb_s * 1e3, "combined_frac_of_ideal": ideal / mb_s, "steps": osteps,
            "clocks": {"prefill": mpclocks, "decode": mdclocks, "both": mbclocks}}
        launches += 4 * osteps
        del mq, mkv, mpt, mout, mlse, mplan

    # ---- CPU baseline: the oracle on a bounded sample (rank 0, N = 1 only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        cores = os.cpu_count() or 1
        rows = np.arange(batch.batch_size, dtype=np.int64)
        rr = np.repeat(rows, batch.num_qo_heads)
        hh = np.tile(np.arange(batch.num_qo_heads, dtype=np.int32), len(rows))
        t0 = time.perf_counter()
        oracle.sink_attention(batch, rows=rr, heads=hh, n_threads=cores)
        dt = time.perf_counter() - t0
        cpu = {"value": bytes_step / dt / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
               "sample": f"the whole gptoss_decode batch (seed 0), fp64 C oracle, {dt:.2f} s"}
        # One core: the tiny decode whole, and 1/64 of the headline batch
        # (request 0, all 64 heads).
        tiny = syn.tiny_decode(0)
        t0 = time.perf_counter()
        oracle.sink_attention(tiny, n_threads=1)
        dt_tiny = time.perf_counter() - t0
        r1, h1 = np.zeros(batch.num_qo_heads, dtype=np.int64), np.arange(batch.num_qo_heads, dtype=np.int32)
        t0 = time.perf_counter()
        oracle.sink_attention(batch, rows=r1, heads=h1, n_threads=1)
        dt_one = time.perf_counter() - t0
        cpu["single_core"] = {
            "tiny_decode": {"value": kv_bytes(tiny) / dt_tiny / 1e9, "unit": "GB/s", "seconds": dt_tiny},
            "gptoss_decode_1_64": {"value": kv_bytes(batch, rows_only=batch.kv_lens[:1]) / dt_one / 1e9,
                                   "unit": "GB/s", "seconds": dt_one,
                                   "sample": "request 0 of the gptoss_decode batch, all 64 heads"}}
        # Prefill: every 64th query row of the gpt-oss prefill, all heads, on
        # all cores; the throughput of that sample estimates the whole run.
        if not args.no_prefill and prefill is not None and "unavailable" not in prefill:
            prow = np.arange(0, pbatch.total_rows, 64, dtype=np.int64)
            pr = np.repeat(prow, pbatch.num_qo_heads)
            ph = np.tile(np.arange(pbatch.num_qo_heads, dtype=np.int32), len(prow))
            t0 = time.perf_counter()
            oracle.sink_attention(pbatch, rows=pr, heads=ph, n_threads=cores)
            dt_p = time.perf_counter() - t0
            sflops = sample_prefill_flops(pbatch, prow)
            cpu["prefill"] = {"value": sflops / dt_p / 1e9, "unit": "GFLOP/s", "cores": cores, "kind": "oracle",
                              "sample": f"every 64th row of gptoss_prefill ({len(prow)} rows x 64 heads), "
                                        f"{dt_p:.2f} s; scaled: the sample's throughput stands for the whole run",
                              "scaled_full_run_s": prefill_flops(pbatch) / (sflops / dt_p)}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": total_ms / args.steps, "ms_per_step_median": statistics.median(times),
            "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": headline_config(batch, world),
            "plan": {"plan_us": plan_us, "plan_first_us": plan_first_us, "decode_units": units},
            "roofline": roofline, "e2e": e2e, "gpu_launches": launches,
            "clocks": clocks, "cpu_baseline": cpu, "decode_graph": graph, "prefill": prefill, "prefill_ragged": ragged, "kv_cache": kvcache,
            "other_shapes": others,
        }
        print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_setup(args.impl)
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
