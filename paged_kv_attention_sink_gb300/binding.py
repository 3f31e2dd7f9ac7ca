"""ctypes binding of libattn.so (argument marshalling only).

Every step of the attention runs inside the library's CUDA kernels; this
module checks tensor shapes / dtypes / devices, passes raw pointers and the
current torch CUDA stream through the C ABI declared in ``include/attn.h``,
and turns non-zero status codes into ``AttnError``.  There is no fallback:
if the library is missing, importing this module raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libattn.so")

_STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported shape", 3: "workspace too small",
           4: "CUDA error", 5: "workspace not bound", 6: "device-side error recorded"}


class AttnError(RuntimeError):
    def __init__(self, fn: str, status: int, extra: str = ""):
        self.status = status
        super().__init__(f"{fn} failed: {_STATUS.get(status, status)}{extra}")


class PlanInfo(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("total_qo_rows", ctypes.c_int32),
                ("num_decode_requests", ctypes.c_int32), ("num_prefill_requests", ctypes.c_int32),
                ("num_decode_units", ctypes.c_int32), ("num_decode_groups_split", ctypes.c_int32),
                ("num_decode_partials", ctypes.c_int32), ("decode_chunk_blocks", ctypes.c_int32),
                ("num_prefill_items", ctypes.c_int32), ("num_sms", ctypes.c_int32),
                ("decode_kv_tokens", ctypes.c_int64), ("prefill_pairs", ctypes.c_int64),
                ("workspace_bytes", ctypes.c_size_t)]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_}


def library_path() -> str:
    return _LIB_PATH


def _declare(lib):
    p, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
    st = ctypes.c_int
    sig = {
        "attn_plan": (st, [p, p, p, p, i32, i32, i32, i32, i32, i32, f32, i32, i32, p, p]),
        "attn_plan_bind_workspace": (st, [p, p, ctypes.c_size_t, p]),
        "attn_decode": (st, [p, p, p, p, p, p, p]),
        "attn_prefill": (st, [p, p, p, p, p, p, p]),
        "attn_decode_noalloc": (st, [p, p, p, p, p, p, p]),
        "attn_decode_noalloc_device_error": (st, [p, p, p]),
        "attn_merge_states": (st, [p, p, p, p, p, p, i32, i32, i32, p]),
        "attn_merge_states_f32": (st, [p, p, p, p, p, i32, p, i32, i32, i32, p]),
        "attn_append_kv": (st, [p, p, p, p, p]),
        "attn_plan_ragged": (st, [p, p, i32, i32, i32, i32, i32, f32, i32, p, p]),
        "attn_graph_plan": (st, [i32, i32, i32, i32, i32, f32, i32, i64, p, i32, p, p]),
        "attn_decode_graph": (st, [p, p, p, p, p, p, p, p, p, p]),
        "attn_graph_plan_read_units": (st, [p, p, i64, p, p]),
        "attn_prefill_ragged": (st, [p, p, p, p, p, p, p, p]),
        "attn_pack_kv_heads": (st, [p, i64, i32, i32, i32, p, i64, i32, i32, p, p, p]),
        "attn_unpack_kv_heads": (st, [p, i64, i32, i32, i32, p, i64, i32, i32, p, p, p]),
        "attn_plan_get_info": (st, [p, p]),
        "attn_plan_get_decode_units": (st, [p, p, i64]),
        "attn_plan_get_prefill_items": (st, [p, p, i64]),
        "attn_plan_device_error": (st, [p, p, p]),
        "attn_plan_destroy": (None, [p]),
        "attn_status_string": (ctypes.c_char_p, [st]),
        "attn_selftest_bounded_wait": (st, [p, p]),
        "attn_selftest_exp2": (st, [p, p, p, i64, f32, f32, p]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib = None


def load_library():
    """Load libattn.so (raises ImportError if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise ImportError(f"{_LIB_PATH} is missing: build it with "
                              "`python -c 'import __graft_entry__ as g; g.build()'`")
        _lib = _declare(ctypes.CDLL(_LIB_PATH))
    return _lib


load_library()


def _check(fn: str, status: int, extra: str = ""):
    if status != 0:
        raise AttnError(fn, status, extra)


def _i32_host(a) -> np.ndarray:
    if isinstance(a, torch.Tensor):
        a = a.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(a), dtype=np.int32)


def _ptr(t: Optional[torch.Tensor]):
    # A plain int: ctypes converts it for the c_void_p parameter (cheaper than
    # building a c_void_p object on every call).
    return None if t is None else t.data_ptr()


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream_ptr(stream=None):
    if stream is not None:
        return stream.cuda_stream
    if _raw_stream is not None:   # the current stream's handle without building a Stream object
        return _raw_stream(torch.cuda.current_device())
    return torch.cuda.current_stream().cuda_stream


class Plan:
    """A planned batch: host work lists inside the library plus the device
    workspace (a torch uint8 buffer) they were uploaded to.

    qo_indptr, kv_indptr, last_page_len: host int arrays (or CPU tensors).
    page_table: int32 CUDA tensor; kept referenced by the plan.
    workspace: optional uint8 CUDA tensor to bind instead of allocating one
    (used when it holds at least the plan's workspace_bytes and starts on a
    256-byte boundary); a serving loop can reuse one per step in flight, as
    long as no launch of an older plan bound to it is still running.
    """

    def __init__(self, qo_indptr, kv_indptr, page_table: torch.Tensor, last_page_len,
                 num_qo_heads: int, num_kv_heads: int, head_dim: int, page_size: int,
                 causal: bool = True, sm_scale: Optional[float] = None,
                 num_pages: Optional[int] = None, num_sms: int = 0, stream=None,
                 workspace: Optional[torch.Tensor] = None):
        lib = load_library()
        self._handle = None
        qo = _i32_host(qo_indptr)
        kv = _i32_host(kv_indptr)
        lpl = _i32_host(last_page_len)
        if not (isinstance(page_table, torch.Tensor) and page_table.is_cuda and
                page_table.dtype == torch.int32 and page_table.is_contiguous()):
            raise TypeError("page_table must be a contiguous int32 CUDA tensor")
        if num_pages is None:
            raise ValueError("num_pages (pages in the KV pool) is required")
        self.page_table = page_table
        self.batch = len(qo) - 1
        self.num_qo_heads, self.num_kv_heads = num_qo_heads, num_kv_heads
        self.head_dim, self.page_size, self.num_pages = head_dim, page_size, num_pages
        self.causal = bool(causal)
        self.sm_scale = float(sm_scale) if sm_scale is not None else head_dim ** -0.5
        self.total_rows = int(qo[-1]) if len(qo) else 0
        handle = ctypes.c_void_p()
        ws_bytes = ctypes.c_size_t()
        _check("attn_plan", lib.attn_plan(
            qo.ctypes.data, kv.ctypes.data, _ptr(page_table), lpl.ctypes.data, self.batch, num_qo_heads,
            num_kv_heads, head_dim, page_size, int(self.causal), self.sm_scale, int(num_pages),
            int(num_sms), ctypes.byref(handle), ctypes.byref(ws_bytes)))
        self._handle = handle
        need = max(int(ws_bytes.value), 256)
        if (workspace is not None and workspace.is_cuda and workspace.dtype == torch.uint8
                and workspace.numel() >= need and workspace.data_ptr() % 256 == 0):
            self.workspace = workspace
        else:
            self.workspace = torch.empty(need, dtype=torch.uint8, device=page_table.device)
        _check("attn_plan_bind_workspace", lib.attn_plan_bind_workspace(
            self._handle, _ptr(self.workspace), self.workspace.numel(), _stream_ptr(stream)))

    def __del__(self):
        if getattr(self, "_handle", None) is not None and _lib is not None:
            _lib.attn_plan_destroy(self._handle)
            self._handle = None

    @property
    def handle(self):
        return self._handle

    def info(self) -> dict:
        info = PlanInfo()
        _check("attn_plan_get_info", load_library().attn_plan_get_info(self._handle, ctypes.byref(info)))
        return info.as_dict()

    def decode_units(self) -> np.ndarray:
        n = self.info()["num_decode_units"]
        out = np.zeros((n, 12), dtype=np.int32)
        _check("attn_plan_get_decode_units", load_library().attn_plan_get_decode_units(
            self._handle, out.ctypes.data_as(ctypes.c_void_p), n))
        return out

    def prefill_items(self) -> np.ndarray:
        n = self.info()["num_prefill_items"]
        out = np.zeros((n, 12), dtype=np.int32)
        _check("attn_plan_get_prefill_items", load_library().attn_plan_get_prefill_items(
            self._handle, out.ctypes.data_as(ctypes.c_void_p), n))
        return out

    def device_error(self, stream=None) -> int:
        code = ctypes.c_int32()
        status = load_library().attn_plan_device_error(self._handle, ctypes.byref(code), _stream_ptr(stream))
        if status not in (0, 6):
            _check("attn_plan_device_error", status)
        return int(code.value)

    # -- launches ---------------------------------------------------------
    def _check_tensors(self, q, kv_cache, sinks, out, lse):
        H, D = self.num_qo_heads, self.head_dim
        for name, t, dt in (("q", q, torch.bfloat16), ("kv_cache", kv_cache, torch.bfloat16),
                            ("out", out, torch.bfloat16)):
            if not (isinstance(t, torch.Tensor) and t.is_cuda and t.dtype == dt and t.is_contiguous()):
                raise TypeError(f"{name} must be a contiguous {dt} CUDA tensor")
        if tuple(q.shape) != (self.total_rows, H, D) or tuple(out.shape) != (self.total_rows, H, D):
            raise ValueError(f"q / out must be [{self.total_rows}, {H}, {D}]")
        if tuple(kv_cache.shape) != (self.num_pages, 2, self.num_kv_heads, self.page_size, D):
            raise ValueError("kv_cache must be [num_pages, 2, Hkv, page_size, head_dim]")
        if sinks is not None and not (sinks.is_cuda and sinks.dtype == torch.float32 and
                                      sinks.is_contiguous() and sinks.numel() == H):
            raise TypeError("sinks must be a contiguous float32 CUDA tensor of num_qo_heads values")
        if lse is not None and not (lse.is_cuda and lse.dtype == torch.float32 and lse.is_contiguous()
                                    and tuple(lse.shape) == (self.total_rows, H)):
            raise TypeError("lse must be a contiguous float32 CUDA tensor [rows, Hq]")

    def _launch(self, fn_name, q, kv_cache, sinks, out, lse, stream):
        self._check_tensors(q, kv_cache, sinks, out, lse)
        fn = getattr(load_library(), fn_name)
        _check(fn_name, fn(self._handle, _ptr(q), _ptr(kv_cache), _ptr(sinks), _ptr(out), _ptr(lse),
                           _stream_ptr(stream)))
        return out, lse

    def decode(self, q, kv_cache, sinks=None, out=None, lse=None, stream=None):
        out = torch.empty_like(q) if out is None else out
        return self._launch("attn_decode", q, kv_cache, sinks, out, lse, stream)

    def prefill(self, q, kv_cache, sinks=None, out=None, lse=None, stream=None):
        out = torch.empty_like(q) if out is None else out
        return self._launch("attn_prefill", q, kv_cache, sinks, out, lse, stream)

    def append_kv(self, k_new, v_new, kv_cache, stream=None):
        """Write the new K/V rows ([rows, Hkv, D] bf16, one per query row) into
        their cache positions in kv_cache (in place)."""
        shape = (self.total_rows, self.num_kv_heads, self.head_dim)
        for name, t in (("k_new", k_new), ("v_new", v_new), ("kv_cache", kv_cache)):
            if not (isinstance(t, torch.Tensor) and t.is_cuda and t.dtype == torch.bfloat16 and t.is_contiguous()):
                raise TypeError(f"{name} must be a contiguous bfloat16 CUDA tensor")
        if tuple(k_new.shape) != shape or tuple(v_new.shape) != shape:
            raise ValueError(f"k_new / v_new must be {list(shape)}")
        if tuple(kv_cache.shape) != (self.num_pages, 2, self.num_kv_heads, self.page_size, self.head_dim):
            raise ValueError("kv_cache must be [num_pages, 2, Hkv, page_size, head_dim]")
        _check("attn_append_kv", load_library().attn_append_kv(
            self._handle, _ptr(k_new), _ptr(v_new), _ptr(kv_cache), _stream_ptr(stream)))
        return kv_cache


class RaggedPlan(Plan):
    """A planned batch over contiguous K / V (no KV cache): every request runs
    on the prefill kernel.  qo_indptr, kv_indptr: host int arrays (token CSR)."""

    def __init__(self, qo_indptr, kv_indptr, num_qo_heads: int, num_kv_heads: int, head_dim: int,
                 causal: bool = True, sm_scale: Optional[float] = None, num_sms: int = 0, device="cuda",
                 stream=None):
        lib = load_library()
        self._handle = None
        qo = _i32_host(qo_indptr)
        kv = _i32_host(kv_indptr)
        self.batch = len(qo) - 1
        self.num_qo_heads, self.num_kv_heads, self.head_dim = num_qo_heads, num_kv_heads, head_dim
        self.causal = bool(causal)
        self.sm_scale = float(sm_scale) if sm_scale is not None else head_dim ** -0.5
        self.total_rows = int(qo[-1]) if len(qo) else 0
        self.kv_tokens = int(kv[-1]) if len(kv) else 0
        handle = ctypes.c_void_p()
        ws_bytes = ctypes.c_size_t()
        _check("attn_plan_ragged", lib.attn_plan_ragged(
            qo.ctypes.data_as(ctypes.c_void_p), kv.ctypes.data_as(ctypes.c_void_p), self.batch, num_qo_heads,
            num_kv_heads, head_dim, int(self.causal), self.sm_scale, int(num_sms), ctypes.byref(handle),
            ctypes.byref(ws_bytes)))
        self._handle = handle
        self.workspace = torch.empty(max(int(ws_bytes.value), 256), dtype=torch.uint8, device=device)
        _check("attn_plan_bind_workspace", lib.attn_plan_bind_workspace(
            self._handle, _ptr(self.workspace), self.workspace.numel(), _stream_ptr(stream)))

    def prefill(self, q, k, v, sinks=None, out=None, lse=None, stream=None):
        H, Hkv, D = self.num_qo_heads, self.num_kv_heads, self.head_dim
        out = torch.empty_like(q) if out is None else out
        for name, t in (("q", q), ("k", k), ("v", v), ("out", out)):
            if not (isinstance(t, torch.Tensor) and t.is_cuda and t.dtype == torch.bfloat16 and t.is_contiguous()):
                raise TypeError(f"{name} must be a contiguous bfloat16 CUDA tensor")
        if tuple(q.shape) != (self.total_rows, H, D) or tuple(out.shape) != (self.total_rows, H, D):
            raise ValueError(f"q / out must be [{self.total_rows}, {H}, {D}]")
        if tuple(k.shape) != (self.kv_tokens, Hkv, D) or tuple(v.shape) != (self.kv_tokens, Hkv, D):
            raise ValueError(f"k / v must be [{self.kv_tokens}, {Hkv}, {D}]")
        if sinks is not None and not (sinks.is_cuda and sinks.dtype == torch.float32 and
                                      sinks.is_contiguous() and sinks.numel() == H):
            raise TypeError("sinks must be a contiguous float32 CUDA tensor of num_qo_heads values")
        if lse is not None and not (lse.is_cuda and lse.dtype == torch.float32 and lse.is_contiguous()
                                    and tuple(lse.shape) == (self.total_rows, H)):
            raise TypeError("lse must be a contiguous float32 CUDA tensor [rows, Hq]")
        _check("attn_prefill_ragged", load_library().attn_prefill_ragged(
            self._handle, _ptr(q), _ptr(k), _ptr(v), _ptr(sinks), _ptr(out), _ptr(lse), _stream_ptr(stream)))
        return out, lse

    def decode(self, *args, **kwargs):
        raise TypeError("a ragged plan has no KV cache; use prefill(q, k, v, ...)")

    def append_kv(self, *args, **kwargs):
        raise TypeError("a ragged plan has no KV cache")


class GraphPlan(Plan):
    """Decode plan for CUDA-graph capture: the work list is built on the device
    at every call from device-resident request metadata (see attn_decode_graph).
    q / out are [max_batch, Hq, D]; lse [max_batch, Hq]."""

    def __init__(self, max_batch: int, num_qo_heads: int, num_kv_heads: int, head_dim: int, page_size: int,
                 page_table: torch.Tensor, num_pages: int, sm_scale: Optional[float] = None,
                 max_kv_tokens: int = 0, num_sms: int = 0, stream=None):
        lib = load_library()
        self._handle = None
        if not (isinstance(page_table, torch.Tensor) and page_table.is_cuda and
                page_table.dtype == torch.int32 and page_table.is_contiguous()):
            raise TypeError("page_table must be a contiguous int32 CUDA tensor")
        self.page_table = page_table
        self.batch = self.total_rows = int(max_batch)
        self.num_qo_heads, self.num_kv_heads = num_qo_heads, num_kv_heads
        self.head_dim, self.page_size, self.num_pages = head_dim, page_size, num_pages
        self.sm_scale = float(sm_scale) if sm_scale is not None else head_dim ** -0.5
        handle = ctypes.c_void_p()
        ws_bytes = ctypes.c_size_t()
        _check("attn_graph_plan", lib.attn_graph_plan(
            int(max_batch), num_qo_heads, num_kv_heads, head_dim, page_size, self.sm_scale, int(num_pages),
            int(max_kv_tokens), _ptr(page_table), int(num_sms), ctypes.byref(handle), ctypes.byref(ws_bytes)))
        self._handle = handle
        self.workspace = torch.empty(max(int(ws_bytes.value), 256), dtype=torch.uint8, device=page_table.device)
        _check("attn_plan_bind_workspace", lib.attn_plan_bind_workspace(
            self._handle, _ptr(self.workspace), self.workspace.numel(), _stream_ptr(stream)))

    def decode(self, q, kv_cache, kv_indptr, last_page_len, batch, sinks=None, out=None, lse=None, stream=None):
        """kv_indptr [>= B+1], last_page_len [>= B], batch [1]: int32 CUDA tensors read on the device."""
        for name, t in (("kv_indptr", kv_indptr), ("last_page_len", last_page_len), ("batch", batch)):
            if not (isinstance(t, torch.Tensor) and t.is_cuda and t.dtype == torch.int32 and t.is_contiguous()):
                raise TypeError(f"{name} must be a contiguous int32 CUDA tensor")
        out = torch.empty_like(q) if out is None else out
        self._check_tensors(q, kv_cache, sinks, out, lse)
        _check("attn_decode_graph", load_library().attn_decode_graph(
            self._handle, _ptr(kv_indptr), _ptr(last_page_len), _ptr(batch), _ptr(q), _ptr(kv_cache), _ptr(sinks),
            _ptr(out), _ptr(lse), _stream_ptr(stream)))
        return out, lse

    def device_units(self, stream=None) -> np.ndarray:
        cap = self.info()["num_decode_partials"]
        out = np.zeros((cap, 12), dtype=np.int32)
        n = ctypes.c_int64()
        _check("attn_graph_plan_read_units", load_library().attn_graph_plan_read_units(
            self._handle, out.ctypes.data_as(ctypes.c_void_p), cap, ctypes.byref(n), _stream_ptr(stream)))
        return out[:n.value]

    def prefill(self, *args, **kwargs):
        raise TypeError("a graph plan only decodes")

    def append_kv(self, *args, **kwargs):
        raise TypeError("a graph plan only decodes")


def attn_plan(qo_indptr, kv_indptr, page_table, last_page_len, num_qo_heads, num_kv_heads,
              head_dim, page_size, causal=True, sm_scale=None, num_pages=None, num_sms=0,
              stream=None) -> Plan:
    return Plan(qo_indptr, kv_indptr, page_table, last_page_len, num_qo_heads, num_kv_heads,
                head_dim, page_size, causal=causal, sm_scale=sm_scale, num_pages=num_pages,
                num_sms=num_sms, stream=stream)


def attn_decode(plan: Plan, q, kv_cache, sinks=None, out=None, lse=None, stream=None):
    return plan.decode(q, kv_cache, sinks, out, lse, stream)


def attn_prefill(plan: Plan, q, kv_cache, sinks=None, out=None, lse=None, stream=None):
    return plan.prefill(q, kv_cache, sinks, out, lse, stream)


def attn_merge_states(va, lsea, vb, lseb, vout=None, lseout=None, stream=None):
    """Merge two (bf16 [n, H, D], fp32 [n, H]) attention states by log-sum-exp."""
    for name, t, dt in (("va", va, torch.bfloat16), ("vb", vb, torch.bfloat16),
                        ("lsea", lsea, torch.float32), ("lseb", lseb, torch.float32)):
        if not (isinstance(t, torch.Tensor) and t.is_cuda and t.dtype == dt and t.is_contiguous()):
            raise TypeError(f"{name} must be a contiguous {dt} CUDA tensor")
    n, H, D = va.shape
    if vb.shape != va.shape or lsea.shape != (n, H) or lseb.shape != (n, H):
        raise ValueError("state shapes disagree")
    vout = torch.empty_like(va) if vout is None else vout
    _check("attn_merge_states", load_library().attn_merge_states(
        _ptr(va), _ptr(lsea), _ptr(vb), _ptr(lseb), _ptr(vout), _ptr(lseout), n, H, D,
        _stream_ptr(stream)))
    return vout, lseout


def attn_merge_states_f32(va, lsea, vb, lseb, vout=None, lseout=None, out_dtype=torch.float32, stream=None):
    """Merge two (fp32 [n, H, D], fp32 [n, H]) attention states by log-sum-exp;
    the merged values are fp32 or bf16 (out_dtype, or vout's dtype)."""
    for name, t in (("va", va), ("vb", vb), ("lsea", lsea), ("lseb", lseb)):
        if not (isinstance(t, torch.Tensor) and t.is_cuda and t.dtype == torch.float32 and t.is_contiguous()):
            raise TypeError(f"{name} must be a contiguous float32 CUDA tensor")
    n, H, D = va.shape
    if vb.shape != va.shape or lsea.shape != (n, H) or lseb.shape != (n, H):
        raise ValueError("state shapes disagree")
    if vout is None:
        vout = torch.empty(n, H, D, dtype=out_dtype, device=va.device)
    if vout.dtype not in (torch.float32, torch.bfloat16) or vout.shape != va.shape or not vout.is_contiguous():
        raise TypeError("vout must be a contiguous float32 or bfloat16 tensor shaped like va")
    _check("attn_merge_states_f32", load_library().attn_merge_states_f32(
        _ptr(va), _ptr(lsea), _ptr(vb), _ptr(lseb), _ptr(vout), int(vout.dtype == torch.bfloat16), _ptr(lseout),
        n, H, D, _stream_ptr(stream)))
    return vout, lseout


def _head_slice(fn_name, kv_cache, page_ids, head_begin, n_heads, buf, device_error, stream):
    for name, t in (("kv_cache", kv_cache), ("buf", buf)):
        if not (isinstance(t, torch.Tensor) and t.is_cuda and t.dtype == torch.bfloat16 and t.is_contiguous()):
            raise TypeError(f"{name} must be a contiguous bfloat16 CUDA tensor")
    if not (isinstance(page_ids, torch.Tensor) and page_ids.is_cuda and page_ids.dtype == torch.int32
            and page_ids.is_contiguous()):
        raise TypeError("page_ids must be a contiguous int32 CUDA tensor")
    num_pages, two, hkv, P, D = kv_cache.shape
    if two != 2 or tuple(buf.shape) != (page_ids.numel(), 2, n_heads, P, D):
        raise ValueError("buf must be [n_pages, 2, n_heads, page_size, head_dim] for the pool's page shape")
    _check(fn_name, getattr(load_library(), fn_name)(
        _ptr(kv_cache) if fn_name == "attn_pack_kv_heads" else _ptr(buf), num_pages, hkv, P, D, _ptr(page_ids),
        page_ids.numel(), head_begin, n_heads,
        _ptr(buf) if fn_name == "attn_pack_kv_heads" else _ptr(kv_cache), _ptr(device_error),
        _stream_ptr(stream)))


def attn_pack_kv_heads(kv_cache, page_ids, head_begin, n_heads, buf=None, device_error=None, stream=None):
    """Heads [head_begin, head_begin + n_heads) of pages page_ids of the HND
    pool -> buf [n_pages, 2, n_heads, page_size, head_dim]."""
    if buf is None:
        buf = torch.empty((page_ids.numel(), 2, n_heads, kv_cache.shape[3], kv_cache.shape[4]),
                          dtype=kv_cache.dtype, device=kv_cache.device)
    _head_slice("attn_pack_kv_heads", kv_cache, page_ids, head_begin, n_heads, buf, device_error, stream)
    return buf


def attn_unpack_kv_heads(buf, page_ids, head_begin, kv_cache, device_error=None, stream=None):
    """Write buf [n_pages, 2, n_heads, page_size, head_dim] into heads
    [head_begin, head_begin + n_heads) of pages page_ids of the pool (in place)."""
    _head_slice("attn_unpack_kv_heads", kv_cache, page_ids, head_begin, buf.shape[2], buf, device_error, stream)
    return kv_cache


def attn_selftest_bounded_wait(result=None, stream=None):
    """Run the library's bounded-wait diagnostic (one warp waits on an mbarrier
    nothing arrives on).  Returns the device int64 [2] result: the
    ATTN_DEVICE_ERR_* bit the kernel recorded and the nanoseconds it waited."""
    if result is None:
        result = torch.full((2,), -1, dtype=torch.int64, device="cuda")
    if not (isinstance(result, torch.Tensor) and result.is_cuda and result.dtype == torch.int64
            and result.numel() >= 2 and result.is_contiguous()):
        raise TypeError("result must be a contiguous int64 CUDA tensor of at least 2 elements")
    _check("attn_selftest_bounded_wait", load_library().attn_selftest_bounded_wait(_ptr(result),
                                                                                   _stream_ptr(stream)))
    return result


def attn_selftest_exp2(x, scale_log2=1.0, m=0.0, stream=None):
    """Evaluate the prefill softmax's FMA-pipe 2^(x * scale_log2 - m) and the
    MUFU's ex2.approx on the same fp32 CUDA tensor; returns (y_poly, y_mufu)."""
    if not (isinstance(x, torch.Tensor) and x.is_cuda and x.dtype == torch.float32 and x.is_contiguous()):
        raise TypeError("x must be a contiguous float32 CUDA tensor")
    y_poly = torch.empty_like(x)
    y_mufu = torch.empty_like(x)
    _check("attn_selftest_exp2", load_library().attn_selftest_exp2(
        _ptr(x), _ptr(y_poly), _ptr(y_mufu), x.numel(), float(scale_log2), float(m), _stream_ptr(stream)))
    return y_poly, y_mufu
