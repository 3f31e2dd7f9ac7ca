"""CPU checks of the C ABI: the library loads, exports every symbol that
include/attn.h declares, and the host planner builds correct work lists and
rejects malformed input with status codes (no GPU needed: attn_plan never
touches the device when num_sms is given, and never reads page_table)."""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn.h")

OK, INVALID, UNSUPPORTED = 0, 1, 2


@pytest.fixture(scope="module")
def lib():
    from paged_kv_attention_sink_gb300 import build
    build.build()
    from paged_kv_attention_sink_gb300 import binding
    return binding.load_library()


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"ATTN_API\s+[\w\s\*]+?\b(attn_\w+)\s*\(", text)


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 11
    for name in names:
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code in range(7):
        assert lib.attn_status_string(code)
    assert lib.attn_status_string(0) == b"ok"


FAKE_PT = ctypes.c_void_p(0x1000)   # never dereferenced by the planner


def plan(lib, qo, kv_pages, last, Hq=64, Hkv=8, D=64, P=16, causal=1, pool=100000, sms=152):
    qo_indptr = np.concatenate([[0], np.cumsum(qo)]).astype(np.int32)
    kv_indptr = np.concatenate([[0], np.cumsum(kv_pages)]).astype(np.int32)
    last = np.asarray(last, dtype=np.int32)
    handle = ctypes.c_void_p()
    ws = ctypes.c_size_t()
    st = lib.attn_plan(qo_indptr.ctypes.data_as(ctypes.c_void_p), kv_indptr.ctypes.data_as(ctypes.c_void_p),
                       FAKE_PT, last.ctypes.data_as(ctypes.c_void_p), len(qo), Hq, Hkv, D, P, causal,
                       D ** -0.5, pool, sms, ctypes.byref(handle), ctypes.byref(ws))
    return st, handle, ws.value


def units_of(lib, handle):
    from paged_kv_attention_sink_gb300.binding import PlanInfo
    info = PlanInfo()
    assert lib.attn_plan_get_info(handle, ctypes.byref(info)) == OK
    u = np.zeros((info.num_decode_units, 12), dtype=np.int32)
    assert lib.attn_plan_get_decode_units(handle, u.ctypes.data_as(ctypes.c_void_p), len(u)) == OK
    it = np.zeros((info.num_prefill_items, 12), dtype=np.int32)
    assert lib.attn_plan_get_prefill_items(handle, it.ctypes.data_as(ctypes.c_void_p), len(it)) == OK
    return info, u, it


@pytest.mark.parametrize("Hq,Hkv,P", [(64, 8, 16), (64, 4, 64), (8, 2, 16), (48, 1, 32), (20, 20, 128)])
def test_decode_units_cover_every_token_once(lib, Hq, Hkv, P):
    rng = np.random.default_rng(Hq + P)
    kv = rng.integers(1, 20000, size=37)
    pages = (kv + P - 1) // P
    last = kv - (pages - 1) * P
    st, h, ws = plan(lib, [1] * len(kv), pages, last, Hq=Hq, Hkv=Hkv, P=P)
    assert st == OK and ws > 0
    info, u, _ = units_of(lib, h)
    G = Hq // Hkv
    cover = {}
    for (q_row, page_base, g, head0, nh, t0, t1, chunk, nch, group, part0, _) in u:
        assert t0 % 16 == 0 and t0 < t1 and nh >= 1 and nh <= 16
        assert head0 >= g * G and head0 + nh <= (g + 1) * G
        assert (t1 - t0) <= 512 * 16
        assert (group >= 0) == (nch > 1)
        for hh in range(head0, head0 + nh):
            cover.setdefault((q_row, hh), []).append((t0, t1, chunk, nch))
    assert len(cover) == len(kv) * Hq
    for b in range(len(kv)):
        for hh in range(Hq):
            parts = sorted(cover[(b, hh)])
            assert parts[0][0] == 0 and parts[-1][1] == kv[b]
            for a, c in zip(parts, parts[1:]):
                assert a[1] == c[0]                       # contiguous, no overlap
            assert sorted(p[2] for p in parts) == list(range(parts[0][3]))
            assert sum(1 for p in parts if p[2] == 0) == 1   # sink in exactly one chunk
    # partial slots are disjoint per group
    slots = set()
    for row in u:
        if row[8] > 1:
            s = (row[10] + row[7])
            assert s not in slots
            slots.add(s)
    assert len(slots) == info.num_decode_partials
    lib.attn_plan_destroy(h)


def test_decode_units_sorted_longest_first(lib):
    kv = np.array([100, 5000, 17, 9000, 3000])
    pages = (kv + 15) // 16
    st, h, _ = plan(lib, [1] * 5, pages, kv - (pages - 1) * 16)
    _, u, _ = units_of(lib, h)
    lens = u[:, 6] - u[:, 5]
    assert np.all(np.diff(lens) <= 0)
    lib.attn_plan_destroy(h)


@pytest.mark.parametrize("causal", [1, 0])
def test_prefill_items_cover_rows_heads(lib, causal):
    qo = np.array([300, 1, 2048, 129, 0, 5])
    kv = np.array([300, 40, 4096, 1000, 7, 5])
    pages = (kv + 15) // 16
    last = kv - (pages - 1) * 16
    st, h, _ = plan(lib, qo, pages, last, causal=causal)
    assert st == OK
    info, u, it = units_of(lib, h)
    assert info.num_decode_requests == 1 and info.num_prefill_requests == 4
    qo_indptr = np.concatenate([[0], np.cumsum(qo)])
    seen = {}
    for (row0, nrows, page_base, kv_len, pos0, g, head0, nh, ntiles, key_end, _, _) in it:
        b = int(np.searchsorted(qo_indptr, row0, side="right") - 1)
        assert kv_len == kv[b] and 1 <= nrows <= 128 and nh in (1, 2)
        assert pos0 == kv[b] - qo[b] + (row0 - qo_indptr[b])
        exp_end = min(kv[b], pos0 + nrows) if causal else kv[b]
        assert key_end == exp_end and ntiles == -(-exp_end // 128)
        for hh in range(head0, head0 + nh):
            assert hh // 8 == g
            for r in range(row0, row0 + nrows):
                seen[(r, hh)] = seen.get((r, hh), 0) + 1
    expected = {(r, hh) for b in range(len(qo)) if qo[b] > 1
                for r in range(qo_indptr[b], qo_indptr[b + 1]) for hh in range(64)}
    assert set(seen) == expected and all(v == 1 for v in seen.values())
    pairs = sum((kv[b] - qo[b] + i + 1) if causal else kv[b]
                for b in range(len(qo)) if qo[b] > 1 for i in range(qo[b]))
    assert info.prefill_pairs == pairs
    lib.attn_plan_destroy(h)


def test_split_balances_small_batches(lib):
    """Two long sequences on 152 SMs are split into many chunks."""
    kv = np.array([32768, 32768])
    pages = kv // 16
    st, h, _ = plan(lib, [1, 1], pages, np.full(2, 16))
    info, u, _ = units_of(lib, h)
    assert info.num_decode_units >= 152
    lib.attn_plan_destroy(h)


@pytest.mark.parametrize("case", [
    dict(qo=[2], kv_pages=[0], last=[0]),            # qo_len > kv_len
    dict(qo=[1], kv_pages=[2], last=[0]),            # last_page_len out of range
    dict(qo=[1], kv_pages=[2], last=[17]),
    dict(qo=[1], kv_pages=[1], last=[4], Hq=6, Hkv=4),
    dict(qo=[1], kv_pages=[1], last=[4], causal=2),
])
def test_plan_rejects_malformed(lib, case):
    st, h, _ = plan(lib, **case)
    assert st == INVALID


@pytest.mark.parametrize("case", [dict(D=96), dict(P=8), dict(D=256)])
def test_plan_rejects_unsupported(lib, case):
    st, h, _ = plan(lib, [1], [1], [4], **case)
    assert st == UNSUPPORTED


def test_plan_null_and_negative_indptr(lib):
    handle = ctypes.c_void_p()
    ws = ctypes.c_size_t()
    assert lib.attn_plan(None, None, None, None, 1, 8, 2, 64, 16, 1, 0.125, 10, 152,
                         ctypes.byref(handle), ctypes.byref(ws)) == INVALID
    st, h, _ = plan(lib, [3, -2], [1, 1], [4, 4])
    assert st == INVALID


def test_empty_batch_plan(lib):
    st, h, ws = plan(lib, [], [], [])
    assert st == OK
    info, u, it = units_of(lib, h)
    assert info.num_decode_units == 0 and info.num_prefill_items == 0
    lib.attn_plan_destroy(h)


def test_launch_without_workspace_is_rejected(lib):
    st, h, _ = plan(lib, [1], [1], [4])
    dummy = ctypes.c_void_p(0x10000)
    assert lib.attn_decode(h, dummy, dummy, None, dummy, None, None) == 5   # not bound
    assert lib.attn_plan_bind_workspace(h, ctypes.c_void_p(0x10001), 1 << 20, None) == INVALID
    assert lib.attn_plan_bind_workspace(h, ctypes.c_void_p(0x10000), 1, None) == 3
    lib.attn_plan_destroy(h)


def test_noalloc_decode_refuses_graph_plans(lib):
    """A graph plan's work list is built on the device, so its host list is
    empty; the no-alloc decode must refuse it rather than report an empty
    batch as done.  Neither call reaches the device here."""
    h = ctypes.c_void_p()
    ws = ctypes.c_size_t()
    assert lib.attn_graph_plan(8, 16, 2, 64, 16, ctypes.c_float(0.125), 1024, 8 * 4096, ctypes.c_void_p(0x10000),
                               152, ctypes.byref(h), ctypes.byref(ws)) == OK
    dummy = ctypes.c_void_p(0x10000)
    assert lib.attn_decode_noalloc(h, dummy, dummy, None, dummy, None, None) == INVALID
    code = ctypes.c_int32(-1)
    assert lib.attn_decode_noalloc_device_error(h, ctypes.byref(code), None) == INVALID
    assert lib.attn_decode_noalloc(None, dummy, dummy, None, dummy, None, None) == INVALID
    assert lib.attn_decode_noalloc_device_error(None, ctypes.byref(code), None) == INVALID
    lib.attn_plan_destroy(h)


def test_merge_states_argument_checks(lib):
    p = ctypes.c_void_p(0x10000)
    assert lib.attn_merge_states(p, p, p, p, p, None, 4, 2, 6, None) == INVALID   # D % 4
    assert lib.attn_merge_states(p, p, p, p, p, None, -1, 2, 8, None) == INVALID
    assert lib.attn_merge_states(None, None, None, None, None, None, 0, 2, 8, None) == OK
    # fp32 states: 16-byte aligned inputs, 16 (fp32) or 8 (bf16) byte aligned output
    assert lib.attn_merge_states_f32(p, p, p, p, p, 0, None, 4, 2, 6, None) == INVALID   # D % 4
    assert lib.attn_merge_states_f32(p, p, p, p, ctypes.c_void_p(0x10008), 0, None, 4, 2, 8, None) == INVALID
    assert lib.attn_merge_states_f32(ctypes.c_void_p(0x10008), p, p, p, p, 0, None, 4, 2, 8, None) == INVALID
    assert lib.attn_merge_states_f32(None, None, None, None, None, 1, None, 0, 2, 8, None) == OK
    assert lib.attn_merge_states_f32(None, p, p, p, p, 1, None, 4, 2, 8, None) == INVALID


def test_head_slice_argument_checks(lib):
    p = ctypes.c_void_p(0x10000)
    # head range outside the pool's heads, head_dim not a multiple of 8, misaligned pointers
    assert lib.attn_pack_kv_heads(p, 10, 8, 16, 64, p, 4, 6, 4, p, None, None) == INVALID
    assert lib.attn_pack_kv_heads(p, 10, 8, 16, 60, p, 4, 0, 4, p, None, None) == INVALID
    assert lib.attn_unpack_kv_heads(ctypes.c_void_p(0x10008), 10, 8, 16, 64, p, 4, 0, 4, p, None, None) == INVALID
    assert lib.attn_pack_kv_heads(p, 10, 8, 16, 64, p, 0, 0, 4, p, None, None) == OK      # nothing to move


def test_append_requires_bound_workspace(lib):
    st, h, _ = plan(lib, [1], [1], [4])
    dummy = ctypes.c_void_p(0x10000)
    assert lib.attn_append_kv(h, dummy, dummy, dummy, None) == 5     # not bound
    lib.attn_plan_destroy(h)


def test_ragged_plan_covers_every_request(lib):
    qo = np.array([0, 1, 301, 301, 350], dtype=np.int32)        # a 1-row request and an empty one
    kv = np.array([0, 9, 309, 320, 369], dtype=np.int32)        # token CSR
    handle = ctypes.c_void_p()
    ws = ctypes.c_size_t()
    st = lib.attn_plan_ragged(qo.ctypes.data_as(ctypes.c_void_p), kv.ctypes.data_as(ctypes.c_void_p), 4, 8, 2,
                              64, 1, 0.125, 152, ctypes.byref(handle), ctypes.byref(ws))
    assert st == OK
    info, u, it = units_of(lib, handle)
    assert info.num_decode_units == 0 and info.num_prefill_requests == 3
    rows = set()
    for (row0, nrows, kv_off, kv_len, pos0, g, head0, nh, ntiles, key_end, _, _) in it:
        b = int(np.searchsorted(qo, row0, side="right") - 1)
        assert kv_off == kv[b] and kv_len == kv[b + 1] - kv[b]
        assert pos0 == kv_len - (qo[b + 1] - qo[b]) + (row0 - qo[b])
        for r in range(row0, row0 + nrows):
            for h in range(head0, head0 + nh):
                rows.add((r, h))
    assert rows == {(r, h) for r in range(350) for h in range(8)}
    lib.attn_plan_destroy(handle)


def _check_decode_units(u, qo, kv, Hq, Hkv):
    """Units cover every (decode row, query head) over [0, kv_len) in
    contiguous chunks, chunk 0 once (it carries the sink), and the split
    groups own disjoint partial slots."""
    G = Hq // Hkv
    qo_indptr = np.concatenate([[0], np.cumsum(qo)])
    cover = {}
    for (q_row, page_base, g, head0, nh, t0, t1, chunk, nch, group, part0, _) in u:
        assert t0 % 16 == 0 and t0 < t1 and 1 <= nh <= 16
        assert g * G <= head0 and head0 + nh <= (g + 1) * G
        assert (group >= 0) == (nch > 1)
        for hh in range(head0, head0 + nh):
            cover.setdefault((int(q_row), hh), []).append((int(t0), int(t1), int(chunk), int(nch)))
    decode = [b for b in range(len(qo)) if qo[b] == 1 and kv[b] > 0]
    assert set(cover) == {(int(qo_indptr[b]), hh) for b in decode for hh in range(Hq)}
    for b in decode:
        for hh in range(Hq):
            parts = sorted(cover[(int(qo_indptr[b]), hh)])
            assert parts[0][0] == 0 and parts[-1][1] == kv[b]
            assert all(a[1] == c[0] for a, c in zip(parts, parts[1:]))
            assert sorted(p[2] for p in parts) == list(range(parts[0][3]))
    slots = [int(r[10] + r[7]) for r in u if r[8] > 1]
    assert len(slots) == len(set(slots))


def _check_prefill_items(it, qo, kv, Hq, Hkv, causal):
    """Items cover every (prefill row, query head) once, with the causal
    alignment's position and visible-key bound."""
    G = Hq // Hkv
    qo_indptr = np.concatenate([[0], np.cumsum(qo)])
    seen = {}
    for (row0, nrows, page_base, kv_len, pos0, g, head0, nh, ntiles, key_end, _, _) in it:
        b = int(np.searchsorted(qo_indptr, row0, side="right") - 1)
        assert kv_len == kv[b] and 1 <= nrows <= 128 and nh in (1, 2)
        assert pos0 == kv[b] - qo[b] + (row0 - qo_indptr[b])
        end = min(kv[b], pos0 + nrows) if causal else kv[b]
        assert key_end == end and ntiles == -(-end // 128)
        for hh in range(head0, head0 + nh):
            assert hh // G == g
            for r in range(row0, row0 + nrows):
                seen[(int(r), hh)] = seen.get((int(r), hh), 0) + 1
    expected = {(int(r), hh) for b in range(len(qo)) if qo[b] > 1
                for r in range(qo_indptr[b], qo_indptr[b + 1]) for hh in range(Hq)}
    assert set(seen) == expected and all(v == 1 for v in seen.values())


@pytest.mark.parametrize("seed", range(12))
def test_random_mixed_batches_plan_correctly(lib, seed):
    """Random mixed batches (decode, prefill on cached prefixes, empty
    requests) over random head counts, page sizes and SM counts."""
    rng = np.random.default_rng(500 + seed)
    Hkv = int(rng.choice([1, 2, 4, 8]))
    G = int(rng.choice([1, 2, 3, 8, 12, 20]))
    Hq, P = Hkv * G, int(rng.choice([16, 32, 64, 128]))
    B = int(rng.integers(1, 24))
    kv = rng.integers(0, 6000, size=B)
    kinds = rng.integers(0, 3, size=B)               # 0: decode, 1: prefill, 2: no queries
    qo = np.where(kinds == 0, 1, np.where(kinds == 1, rng.integers(2, 400, size=B), 0))
    qo = np.where(kv == 0, 0, np.minimum(qo, kv))      # qo_len <= kv_len; no queries on empty requests
    pages = (kv + P - 1) // P
    last = np.where(pages > 0, kv - (pages - 1) * P, 0)
    causal = int(rng.integers(0, 2))
    sms = int(rng.choice([1, 7, 152]))
    st, h, ws = plan(lib, qo, pages, last, Hq=Hq, Hkv=Hkv, D=64, P=P, causal=causal, sms=sms)
    assert st == OK
    info, u, it = units_of(lib, h)
    assert info.num_decode_requests == int(np.sum(qo == 1))
    assert info.num_prefill_requests == int(np.sum(qo > 1))
    assert info.total_qo_rows == int(qo.sum())
    assert info.decode_kv_tokens == int(kv[qo == 1].sum())
    _check_decode_units(u, qo, kv, Hq, Hkv)
    _check_prefill_items(it, qo, kv, Hq, Hkv, causal)
    lib.attn_plan_destroy(h)
