"""Shared helpers for the GPU parity tests (device copies of seeded inputs,
plan construction, and the tolerance check against the fp64 oracle)."""
import numpy as np
import torch

from paged_kv_attention_sink_gb300 import synthetic as syn

# Tolerances on bf16 outputs and fp32 lse against the fp64 oracle.
MAX_ABS = 1e-2
MEAN_ABS = 1e-3
LSE_ABS = 1e-3


def to_device(batch, device="cuda"):
    q = torch.from_numpy(batch.q.view(np.int16)).view(torch.bfloat16).to(device)
    kv = torch.from_numpy(batch.kv_pool.view(np.int16)).view(torch.bfloat16).to(device)
    pt = torch.from_numpy(batch.page_table).to(device)
    sinks = None if batch.sinks is None else torch.from_numpy(batch.sinks).to(device)
    return q, kv, pt, sinks


def make_plan(batch, page_table, **kw):
    from paged_kv_attention_sink_gb300 import binding
    return binding.Plan(batch.qo_indptr, batch.kv_indptr, page_table, batch.last_page_len,
                        batch.num_qo_heads, batch.num_kv_heads, batch.head_dim, batch.page_size,
                        causal=batch.causal, sm_scale=batch.sm_scale, num_pages=batch.num_pages, **kw)


def bf16_ulp(x):
    """Spacing of bf16 numbers at |x| (8 significant bits)."""
    ax = np.maximum(np.abs(x), np.finfo(np.float32).tiny)
    return 2.0 ** (np.floor(np.log2(ax)) - 7)


def check_close(out_gpu, lse_gpu, ref_out, ref_lse, what=""):
    """Spec tolerance: max-abs <= 1e-2 and mean-abs <= 1e-3 on the bf16
    outputs, lse within 1e-3.  Where |ref| >= 4, one bf16 ulp already exceeds
    1e-2, so those elements are held to 1 ulp instead (counted and reported)."""
    out = out_gpu.double().cpu().numpy() if isinstance(out_gpu, torch.Tensor) else out_gpu
    assert out.shape == ref_out.shape, (out.shape, ref_out.shape)
    assert np.all(np.isfinite(out)), f"{what}: non-finite output"
    err = np.abs(out - ref_out)
    big = np.abs(ref_out) >= 4.0
    assert np.all(err[big] <= bf16_ulp(ref_out[big])), f"{what}: >1 ulp where |ref| >= 4"
    small_err = err[~big]
    assert small_err.size == 0 or small_err.max() <= MAX_ABS, f"{what}: max abs err {small_err.max():.3e}"
    assert err.mean() <= MEAN_ABS, f"{what}: mean abs err {err.mean():.3e}"
    if lse_gpu is not None:
        lse = lse_gpu.double().cpu().numpy() if isinstance(lse_gpu, torch.Tensor) else lse_gpu
        fin = np.isfinite(ref_lse)
        assert np.array_equal(np.isfinite(lse), fin), f"{what}: lse finiteness differs"
        if fin.any():
            lerr = np.abs(lse[fin] - ref_lse[fin])
            assert lerr.max() <= LSE_ABS, f"{what}: lse max abs err {lerr.max():.3e}"
    return float(err.max()), float(err.mean()), int(big.sum())


def sample_pairs(batch, rows, n, seed=0):
    """n random (row, head) pairs drawn from the given rows."""
    rng = np.random.default_rng(seed)
    r = rng.choice(np.asarray(rows), size=n)
    h = rng.integers(0, batch.num_qo_heads, size=n)
    return r.astype(np.int64), h.astype(np.int32)


def decode_rows(batch):
    return [int(batch.qo_indptr[b]) for b in range(batch.batch_size) if batch.qo_lens[b] == 1]


def prefill_rows(batch):
    rows = []
    for b in range(batch.batch_size):
        if batch.qo_lens[b] > 1:
            rows.extend(range(int(batch.qo_indptr[b]), int(batch.qo_indptr[b + 1])))
    return rows


__all__ = ["syn", "to_device", "make_plan", "check_close", "sample_pairs", "decode_rows",
           "prefill_rows", "MAX_ABS", "MEAN_ABS", "LSE_ABS"]
