"""Seeded synthetic inputs for paged sink attention.

This module only draws random inputs and lays them out; it holds none of the
attention arithmetic, so that both the CUDA library and the CPU oracle can be
fed the very same bytes.  Everything is numpy; nothing here touches a GPU.

Recipe (the same for every workload):

* generator: ``numpy.random.Generator(PCG64(seed))``;
* Q, K, V: N(0, 1) drawn in float32 and rounded to bf16 (round to nearest,
  ties to even); arrays hold bf16 bit patterns as ``uint16``;
* sinks: N(0, 1) float32 per query head, or None (no sink, i.e. -inf);
* page table: the request's pages are a random subset, in random order, of a
  pool holding ``pool_factor`` times the pages needed (or an explicit pool
  size); pages no request uses, and the unused tail of each request's last
  page, are filled with bf16 NaN so that any stray read shows up in results;
* KV layout HND: pool[page][0=K,1=V][kv_head][token_in_page][dim];
* Q / output layout: [total_qo_rows][Hq][D], rows of request b at
  qo_indptr[b] .. qo_indptr[b+1];
* sm_scale = 1 / sqrt(D).

The named workloads mirror the serving shapes the pages talk about (gpt-oss
with 64 query / 8 KV heads of dim 64 and 16-token pages; Qwen3-235B with 64
query / 4 KV heads of dim 128), with lengths drawn as stated per function.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import numpy as np

BF16_NAN = np.uint16(0x7FC0)
_CHUNK_ELEMS = 1 << 24   # pool values are drawn in fixed-size chunks (deterministic)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_to_float(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float32 (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclasses.dataclass
class Batch:
    name: str
    num_qo_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    causal: bool
    sm_scale: float
    qo_lens: np.ndarray        # [B] int64
    kv_lens: np.ndarray        # [B] int64
    qo_indptr: np.ndarray      # [B+1] int32
    kv_indptr: np.ndarray      # [B+1] int32 (CSR into page_table)
    page_table: np.ndarray     # [kv_indptr[B]] int32
    last_page_len: np.ndarray  # [B] int32
    q: np.ndarray              # [rows, Hq, D] uint16 (bf16 bits)
    kv_pool: Optional[np.ndarray]  # [num_pages, 2, Hkv, P, D] uint16 (bf16 bits); None if not drawn
    sinks: Optional[np.ndarray]  # [Hq] float32 or None
    pool_pages: int = 0        # pages in the pool (also when kv_pool is None)

    @property
    def batch_size(self) -> int:
        return len(self.qo_lens)

    @property
    def num_pages(self) -> int:
        return self.kv_pool.shape[0] if self.kv_pool is not None else self.pool_pages

    @property
    def total_rows(self) -> int:
        return int(self.qo_indptr[-1])


def _normal_bf16(rng: np.random.Generator, n: int) -> np.ndarray:
    out = np.empty(n, dtype=np.uint16)
    for s in range(0, n, _CHUNK_ELEMS):
        e = min(n, s + _CHUNK_ELEMS)
        out[s:e] = bf16_bits(rng.standard_normal(e - s, dtype=np.float32))
    return out


def make_batch(name: str, qo_lens: Sequence[int], kv_lens: Sequence[int], num_qo_heads: int,
               num_kv_heads: int, head_dim: int, page_size: int, *, causal: bool = True,
               with_sinks: bool = True, pool_pages: Optional[int] = None,
               pool_factor: float = 1.25, rng: Optional[np.random.Generator] = None,
               seed: int = 0, fill_pool: bool = True) -> Batch:
    """Lay out one ragged batch (see the module docstring for the recipe).
    fill_pool=False leaves kv_pool as None (a caller that only times kernels
    draws the pool on the device itself)."""
    if rng is None:
        rng = np.random.Generator(np.random.PCG64(seed))
    qo = np.asarray(qo_lens, dtype=np.int64)
    kv = np.asarray(kv_lens, dtype=np.int64)
    B = len(qo)
    P, D, Hq, Hkv = page_size, head_dim, num_qo_heads, num_kv_heads
    n_pages = (kv + P - 1) // P
    total = int(n_pages.sum())
    pool = pool_pages if pool_pages is not None else max(total, int(math.ceil(total * pool_factor)))
    if pool < total:
        raise ValueError("pool smaller than the pages the batch needs")
    qo_indptr = np.zeros(B + 1, dtype=np.int32)
    qo_indptr[1:] = np.cumsum(qo)
    kv_indptr = np.zeros(B + 1, dtype=np.int32)
    kv_indptr[1:] = np.cumsum(n_pages)
    page_table = rng.permutation(pool)[:total].astype(np.int32)
    last_page_len = np.where(n_pages > 0, kv - (n_pages - 1) * P, 0).astype(np.int32)

    q = _normal_bf16(rng, int(qo.sum()) * Hq * D).reshape(int(qo.sum()), Hq, D)
    kv_pool = None
    if fill_pool:
        kv_pool = _normal_bf16(rng, pool * 2 * Hkv * P * D).reshape(pool, 2, Hkv, P, D)
        used = np.zeros(pool, dtype=bool)
        used[page_table] = True
        kv_pool[~used] = BF16_NAN
        for b in range(B):
            if n_pages[b] > 0 and last_page_len[b] < P:
                last = page_table[kv_indptr[b + 1] - 1]
                kv_pool[last, :, :, last_page_len[b]:, :] = BF16_NAN
    sinks = rng.standard_normal(Hq, dtype=np.float32) if with_sinks else None
    return Batch(name=name, num_qo_heads=Hq, num_kv_heads=Hkv, head_dim=D, page_size=P,
                 causal=causal, sm_scale=1.0 / math.sqrt(D), qo_lens=qo, kv_lens=kv,
                 qo_indptr=qo_indptr, kv_indptr=kv_indptr, page_table=page_table,
                 last_page_len=last_page_len, q=q, kv_pool=kv_pool, sinks=sinks, pool_pages=pool)


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def tiny_decode(seed: int = 0) -> Batch:
    """Two decode requests, kv_len 256 and 97, Hq 8 / Hkv 2, D 64, 16-token
    pages scattered over a 64-page pool."""
    rng = _rng(seed)
    return make_batch("tiny_decode", [1, 1], [256, 97], 8, 2, 64, 16, pool_pages=64, rng=rng)


def gptoss_decode(seed: int = 0, batch: int = 64, fill_pool: bool = True) -> Batch:
    """gpt-oss-120b-shaped decode: kv_len ~ U[1024, 8192], Hq 64 / Hkv 8, D 64, P 16."""
    rng = _rng(seed)
    kv = rng.integers(1024, 8192, size=batch, endpoint=True)
    return make_batch("gptoss_decode", [1] * batch, kv, 64, 8, 64, 16, rng=rng, fill_pool=fill_pool)


def gptoss_prefill(seed: int = 0, n_seq: int = 8) -> Batch:
    """gpt-oss-120b-shaped ragged causal prefill: qo_len = kv_len ~ U[512, 4096]."""
    rng = _rng(seed)
    L = rng.integers(512, 4096, size=n_seq, endpoint=True)
    return make_batch("gptoss_prefill", L, L, 64, 8, 64, 16, causal=True, rng=rng)


def qwen_decode(seed: int = 0, batch: int = 128, fill_pool: bool = True) -> Batch:
    """Qwen3-235B-shaped long-context decode without sinks: kv_len log-uniform in
    [2048, 32768], Hq 64 / Hkv 4, D 128, 64-token pages."""
    rng = _rng(seed)
    kv = np.exp(rng.uniform(math.log(2048), math.log(32768), size=batch))
    kv = np.clip(np.rint(kv), 2048, 32768).astype(np.int64)
    return make_batch("qwen_decode", [1] * batch, kv, 64, 4, 128, 64, with_sinks=False, rng=rng,
                      fill_pool=fill_pool)


def mixed(seed: int = 0, n_decode: int = 256, fill_pool: bool = True) -> Batch:
    """Mixed serving batch: 4 chunked-prefill requests (qo_len 2048 on cached
    prefixes of 0 / 2048 / 4096 / 8192 tokens, causal) followed by decode
    requests with kv_len ~ U[512, 16384]; Hq 64 / Hkv 8, D 64, P 16."""
    rng = _rng(seed)
    prefix = np.array([0, 2048, 4096, 8192])
    dec_kv = rng.integers(512, 16384, size=n_decode, endpoint=True)
    qo = np.concatenate([np.full(4, 2048), np.ones(n_decode, dtype=np.int64)])
    kv = np.concatenate([prefix + 2048, dec_kv])
    return make_batch("mixed", qo, kv, 64, 8, 64, 16, causal=True, rng=rng, fill_pool=fill_pool)


WORKLOADS = {
    "tiny_decode": tiny_decode,
    "gptoss_decode": gptoss_decode,
    "gptoss_prefill": gptoss_prefill,
    "qwen_decode": qwen_decode,
    "mixed": mixed,
}


def new_kv_rows(batch: Batch, seed: int = 0):
    """The step's new K and V rows, one per query row of the batch: bf16 bits
    [rows, Hkv, D] each, ~N(0, 1), seeded (the input of the KV append)."""
    rng = _rng(1000003 + seed)
    n = batch.total_rows * batch.num_kv_heads * batch.head_dim
    shape = (batch.total_rows, batch.num_kv_heads, batch.head_dim)
    return _normal_bf16(rng, n).reshape(shape), _normal_bf16(rng, n).reshape(shape)
