"""Paged GQA attention with per-head sink logits for GB300 (sm_103a).

The compute lives in ``libattn.so`` (hand-written CUDA behind a C ABI declared
in ``include/attn.h``); ``binding`` marshals torch tensors into that ABI.  The
binding is imported lazily so that ``synthetic`` (seeded inputs) can be used on
machines without the built library; any use of the API without the library
raises immediately -- there is no CPU fallback.
"""
_API = ("Plan", "RaggedPlan", "GraphPlan", "attn_plan", "attn_prefill", "attn_decode", "attn_merge_states",
        "attn_pack_kv_heads", "attn_unpack_kv_heads", "load_library", "library_path", "AttnError")


def __getattr__(name):
    if name in _API:
        from . import binding
        return getattr(binding, name)
    raise AttributeError(name)
