"""Oracle for paged sink attention: a plain fp64 CPU implementation.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The product library (``paged_kv_attention_sink_gb300``) never imports
it, and the two share no code; both only consume the seeded inputs from
``paged_kv_attention_sink_gb300.synthetic``.

The arithmetic lives in ``oracle.c`` (see its header for the definition and the
passages of "GPT-OSS on day 0", "Hosting Qwen on Blackwell" and "Disaggregated
prefill and decode" that it follows).  This module compiles it with gcc and
wraps it with ctypes; it adds no arithmetic of its own.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (gcc, fp64, OpenMP, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", _SRC, "-o", _LIB, "-lm"]
        subprocess.run(cmd, check=True)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        p = ctypes.c_void_p
        i32, i64, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
        lib.oracle_sink_attention.restype = ctypes.c_int
        lib.oracle_sink_attention.argtypes = [
            i32, p, p, p, p, p, p, p, i32, i32, i32, i32, i32, f64, i64, i64, i32,
            i64, p, p, i32, p, p]
        lib.oracle_merge_states.restype = None
        lib.oracle_merge_states.argtypes = [i64, i32, p, p, p, p, p, p]
        lib.oracle_append_kv.restype = ctypes.c_int
        lib.oracle_append_kv.argtypes = [i32, p, p, p, p, i32, i32, i32, i64, p, p, p]
        for name in ("oracle_pack_heads", "oracle_unpack_heads"):
            f = getattr(lib, name)
            f.restype = ctypes.c_int
            f.argtypes = [p, i64, i32, i32, i32, p, i64, i32, i32, p]
        _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def sink_attention(batch, sm_scale=None, causal=None, kv_lo=0, kv_hi=2**62, with_sink=True,
                   rows=None, heads=None, n_threads=0, sinks="batch"):
    """Run the oracle on a ``synthetic.Batch``.

    Returns (out, lse) as float64 arrays: [rows, Hq, D] and [rows, Hq] for all
    pairs, or [n, D] and [n] when ``rows``/``heads`` select n (row, head) pairs.
    ``sinks`` may be overridden with an explicit float32 array or None.
    """
    lib = _load()
    b = batch
    sm_scale = b.sm_scale if sm_scale is None else sm_scale
    causal = b.causal if causal is None else causal
    sk = b.sinks if isinstance(sinks, str) else sinks
    sk = None if sk is None else np.ascontiguousarray(sk, dtype=np.float32)
    qo = np.ascontiguousarray(b.qo_indptr, dtype=np.int32)
    kvp = np.ascontiguousarray(b.kv_indptr, dtype=np.int32)
    pt = np.ascontiguousarray(b.page_table, dtype=np.int32)
    lpl = np.ascontiguousarray(b.last_page_len, dtype=np.int32)
    q = np.ascontiguousarray(b.q)
    kv = np.ascontiguousarray(b.kv_pool)
    total_rows = int(qo[-1]) if len(qo) else 0
    if rows is None:
        n_sel = -1
        out = np.empty((total_rows, b.num_qo_heads, b.head_dim), dtype=np.float64)
        lse = np.empty((total_rows, b.num_qo_heads), dtype=np.float64)
        sel_r = sel_h = None
    else:
        sel_r = np.ascontiguousarray(rows, dtype=np.int64)
        sel_h = np.ascontiguousarray(heads, dtype=np.int32)
        n_sel = len(sel_r)
        out = np.empty((n_sel, b.head_dim), dtype=np.float64)
        lse = np.empty((n_sel,), dtype=np.float64)
    rc = lib.oracle_sink_attention(
        b.batch_size, _ptr(qo), _ptr(kvp), _ptr(pt), _ptr(lpl), _ptr(q), _ptr(kv), _ptr(sk),
        b.num_qo_heads, b.num_kv_heads, b.head_dim, b.page_size, int(bool(causal)),
        float(sm_scale), int(kv_lo), int(kv_hi), int(bool(with_sink)), n_sel, _ptr(sel_r),
        _ptr(sel_h), int(n_threads), _ptr(out), _ptr(lse))
    if rc != 0:
        raise ValueError(f"oracle_sink_attention rejected its input (code {rc})")
    return out, lse


def merge_states(va, lsea, vb, lseb):
    """Merge two fp64 attention states (out [..., D], lse [...]) by log-sum-exp."""
    lib = _load()
    va = np.ascontiguousarray(va, dtype=np.float64)
    vb = np.ascontiguousarray(vb, dtype=np.float64)
    lsea = np.ascontiguousarray(lsea, dtype=np.float64)
    lseb = np.ascontiguousarray(lseb, dtype=np.float64)
    D = va.shape[-1]
    n = lsea.size
    vout = np.empty_like(va)
    lseout = np.empty_like(lsea)
    lib.oracle_merge_states(n, D, _ptr(va), _ptr(lsea), _ptr(vb), _ptr(lseb), _ptr(vout),
                            _ptr(lseout))
    return vout, lseout


def append_kv(batch, k_new, v_new):
    """Return (pool after appending k_new / v_new [rows, Hkv, D] bf16 bits,
    status); the batch's pool is not modified."""
    lib = _load()
    pool = np.array(batch.kv_pool, dtype=np.uint16, copy=True)
    k_new = np.ascontiguousarray(k_new, dtype=np.uint16)
    v_new = np.ascontiguousarray(v_new, dtype=np.uint16)
    rc = lib.oracle_append_kv(batch.batch_size, _ptr(batch.qo_indptr), _ptr(batch.kv_indptr),
                              _ptr(batch.page_table), _ptr(batch.last_page_len), batch.num_kv_heads,
                              batch.head_dim, batch.page_size, batch.num_pages, _ptr(k_new),
                              _ptr(v_new), _ptr(pool))
    return pool, rc


def pack_heads(pool, page_ids, h0, nh):
    """Heads [h0, h0+nh) of the given pages of pool [pages, 2, Hkv, P, D] ->
    (buf [n, 2, nh, P, D], status)."""
    lib = _load()
    pool = np.ascontiguousarray(pool, dtype=np.uint16)
    ids = np.ascontiguousarray(page_ids, dtype=np.int32)
    n_pages, _, Hkv, P, D = pool.shape
    buf = np.zeros((len(ids), 2, nh, P, D), dtype=np.uint16)
    rc = lib.oracle_pack_heads(_ptr(pool), n_pages, Hkv, P, D, _ptr(ids), len(ids), h0, nh, _ptr(buf))
    return buf, rc


def unpack_heads(pool, buf, page_ids, h0):
    """Return (pool with buf [n, 2, nh, P, D] written into heads [h0, h0+nh)
    of the given pages, status); the input pool is not modified."""
    lib = _load()
    out = np.array(pool, dtype=np.uint16, copy=True)
    buf = np.ascontiguousarray(buf, dtype=np.uint16)
    ids = np.ascontiguousarray(page_ids, dtype=np.int32)
    n_pages, _, Hkv, P, D = out.shape
    rc = lib.oracle_unpack_heads(_ptr(buf), n_pages, Hkv, P, D, _ptr(ids), len(ids), h0, buf.shape[2],
                                 _ptr(out))
    return out, rc
