"""Host-side checks of the C ABI that need no GPU: the library builds and
loads, exports every function the header declares, rejects bad arguments
before touching the device, and its work list covers exactly the visible key
tiles (checked against the oracle's explicit mask)."""
from __future__ import annotations

import ctypes
import heapq

import numpy as np
import pytest

import oracle.bdlm_oracle as orc
import structured_mask_attention_gb300 as m
from structured_mask_attention_gb300.build import build


@pytest.fixture(scope="module")
def lib():
    build()
    return m.load_library()


def test_exports_every_header_function(lib):
    names = m.header_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n
    assert "sm_103a" in m.bdlm_version()


def _fake(n):
    # aligned, never dereferenced: every call below fails host validation
    return [ctypes.c_void_p(0x100000 + 0x1000 * i) for i in range(n)]


def _fwd(lib, L=256, B=32, Hq=2, Hkv=1, d=64, scale=0.125, ptrs=None, ws=None, ws_bytes=256, o_dtype=0):
    p = ptrs if ptrs is not None else _fake(10)
    ws = ctypes.c_void_p(0x900000) if ws is None else ws
    return lib.bdlm_attn_fwd(*p[:6], L, B, Hq, Hkv, d, scale, p[6], p[7], o_dtype, p[8], p[9], ws, ws_bytes, None)


def test_fwd_validation(lib):
    assert _fwd(lib, L=250, B=32) == 2           # L % B
    assert _fwd(lib, Hq=3, Hkv=2) == 2           # Hq % Hkv
    assert _fwd(lib, d=96) == 2                  # head dim
    assert _fwd(lib, scale=0.0) == 1             # scale
    assert _fwd(lib, scale=float("nan")) == 1
    assert _fwd(lib, o_dtype=7) == 1
    p = _fake(10); p[3] = ctypes.c_void_p(0)
    assert _fwd(lib, ptrs=p) == 1                # null
    p = _fake(10); p[2] = ctypes.c_void_p(0x100008)
    assert _fwd(lib, ptrs=p) == 3                # misaligned
    assert _fwd(lib, ws=ctypes.c_void_p(0)) == 4
    assert _fwd(lib, ws_bytes=16) == 4
    assert "workspace" in m.bdlm_last_error()


def test_shard_and_merge_validation(lib):
    p = _fake(10)
    ws = ctypes.c_void_p(0x900000)
    f = lib.bdlm_attn_fwd_shard
    assert f(*p[:6], 256, 32, 2, 1, 64, 0.1, 10, 5, 0, *p[6:10], ws, 256, None) == 2   # begin > end
    assert f(*p[:6], 256, 32, 2, 1, 64, 0.1, 0, 300, 0, *p[6:10], ws, 256, None) == 2  # end > L
    arr = (ctypes.c_void_p * 1)(0x100000)
    assert lib.bdlm_lse_merge(0, arr, arr, 16, 1, 64, p[0], 0, p[1], None) == 1
    assert lib.bdlm_lse_merge(33, arr, arr, 16, 1, 64, p[0], 0, p[1], None) == 1
    assert lib.bdlm_lse_merge(1, arr, arr, 16, 1, 32, p[0], 0, p[1], None) == 2
    assert lib.bdlm_bwd_preprocess(p[0], 0, p[1], 0, 1, 64, p[2], None) == 2


def test_bwd_validation(lib):
    p = _fake(18)
    ws = ctypes.c_void_p(0x900000)
    need = m.bdlm_workspace_size(m.OP_BWD, 256, 32, 2, 1, 64)
    assert need == 256 + 2 * 2 * 256 * 4
    b = lib.bdlm_attn_bwd
    assert b(*p[:12], 256, 32, 2, 1, 64, 0.1, *p[12:18], 0, ws, need - 1, None) == 4
    assert b(*p[:12], 256, 32, 2, 1, 64, 0.1, *p[12:18], 5, ws, need, None) == 1
    assert m.bdlm_workspace_size(m.OP_BWD, 256, 30, 2, 1, 64) == 0


@pytest.mark.skipif(__import__("torch").cuda.is_available(), reason="host-only check of the no-device path")
def test_valid_call_without_device_reports_error(lib):
    # passes validation, then fails at the first CUDA call because this
    # machine has no GPU: an error status, not a crash
    st = _fwd(lib)
    assert st in (5, 6), st


@pytest.mark.parametrize("L,B,Hq,Hkv,tq,tk,kb,ke,loc", [
    (256, 32, 2, 2, 128, 128, 0, 256, 1),
    (200, 40, 3, 1, 128, 128, 0, 200, 1),
    (384, 128, 2, 1, 128, 128, 0, 384, 1),
    (160, 1, 1, 1, 64, 32, 0, 160, 1),
    (256, 32, 1, 1, 128, 128, 96, 160, 0),   # unaligned shard, no local block
    (256, 32, 1, 1, 128, 128, 0, 0, 1),      # local block only
    (512, 256, 1, 1, 64, 32, 128, 384, 1),
])
def test_worklist_covers_exactly_visible_tiles(lib, L, B, Hq, Hkv, tq, tk, kb, ke, loc):
    items = m.bdlm_worklist(L, B, Hq, Hkv, tq, tk, kb, ke, bool(loc))
    nqt = -(-L // tq)
    assert len(items) == nqt * Hq * 2
    M = orc.mask_2L(L, B)
    keymask = np.zeros(2 * L, dtype=bool)
    keymask[kb:ke] = True
    if loc:
        keymask[L:] = True
    seen = set()
    for (s, h, t, c0, c1, n0, n1, n) in items:
        seen.add((s, h, t))
        assert n == (c1 - c0) + (n1 - n0)
        rows = np.arange(t * tq, min((t + 1) * tq, L)) + s * L
        vis = M[rows] & keymask[None]
        want_c = {j // tk for j in np.nonzero(vis[:, :L].any(0))[0]}
        want_n = {j // tk for j in np.nonzero(vis[:, L:].any(0))[0]}
        got_c = set(range(c0, c1))
        got_n = set(range(n0, n1))
        assert want_c <= got_c and want_n <= got_n
        # no tile outside the visible union except where a contiguous range spans
        # a gap; contiguous ranges are exact at both ends
        if want_c:
            assert min(want_c) == c0 and max(want_c) == c1 - 1
        else:
            assert c0 == c1
        if want_n:
            assert min(want_n) == n0 and max(want_n) == n1 - 1
        else:
            assert n0 == n1
    assert len(seen) == len(items)
    # longest first (block by block for long lists): per stream, the visible
    # key-tile count never exceeds the largest seen so far, by more than one
    # tile for the corrupted stream (whose own-block range can straddle one
    # more tile)
    for s in (0, 1):
        costs = [it[7] for it in items if it[0] == s]
        slack = 0 if s == 0 else 1
        for i in range(1, len(costs)):
            assert costs[i] <= max(costs[:i]) + slack


def test_claiming_in_list_order_balances_clean_costs(lib):
    """The persistent CTAs claim the longest-first list's items in order, each
    item going to the CTA that is free first: per-CTA totals stay within one
    item of each other and within 1 % of the mean."""
    L, B, Hq, Hkv = 131072, 512, 16, 8
    items = m.bdlm_worklist(L, B, Hq, Hkv)
    costs = [it[7] for it in items]
    G = 148
    free_at = [(0, c) for c in range(G)]
    tot = np.zeros(G)
    for cost in costs:
        t, c = heapq.heappop(free_at)
        tot[c] = t + cost
        heapq.heappush(free_at, (tot[c], c))
    assert tot.sum() == sum(costs)
    assert tot.max() - tot.min() <= max(costs)
    assert tot.max() / tot.mean() < 1.01


def test_naive_schedule_lists_items_in_natural_order(lib, monkeypatch):
    """BDLM_SCHED=naive (the load-balancing ablation): query tiles from the
    first to the last, the two streams of one head adjacent, then the heads."""
    L, B, Hq, Hkv = 4096, 256, 4, 2
    monkeypatch.setenv("BDLM_SCHED", "naive")
    items = m.bdlm_worklist(L, B, Hq, Hkv)
    monkeypatch.delenv("BDLM_SCHED")
    lpt = m.bdlm_worklist(L, B, Hq, Hkv)
    assert sorted(items) == sorted(lpt)
    keys = [(t, h, s) for (s, h, t, *_rest) in items]
    assert keys == sorted(keys)
    assert [it[2] for it in lpt][0] == max(it[2] for it in lpt)


def test_varlen_workspace_and_validation_on_host(lib):
    """Packed-batch sizing and argument checks need no GPU: bad offsets give a
    zero workspace size; the entry points reject them before any launch."""
    ws_f = m.bdlm_workspace_size_varlen(m.OP_FWD, (256, 512, 128), 4, 2, 128)
    ws_b = m.bdlm_workspace_size_varlen(m.OP_BWD, (256, 512, 128), 4, 2, 128)
    assert ws_f > 256 and ws_b > ws_f
    # the backward holds D of both streams: 2 * Hq * T fp32
    assert ws_b - ws_f >= 2 * 4 * 896 * 4
    assert m.bdlm_workspace_size_varlen(m.OP_FWD, (256, 0), 4, 2, 128) == 0       # empty sequence
    assert m.bdlm_workspace_size_varlen(m.OP_FWD_SHARD, (256,), 4, 2, 128) == 0   # no packed shard op
    assert m.bdlm_workspace_size_varlen(m.OP_FWD, (256,), 4, 3, 128) == 0         # Hq % Hkv
    lib_ = m.load_library()
    import ctypes
    off = (ctypes.c_int64 * 3)(0, 256, 448)
    st = lib_.bdlm_attn_fwd_varlen(*([None] * 6), ctypes.cast(off, ctypes.c_void_p), 2, 128, 4, 2, 128, 0.1,
                                   None, None, 0, None, None, None, 0, None)
    assert st == 2  # 192-row sequence is not a multiple of B = 128 (checked before the pointers)
    st = lib_.bdlm_attn_fwd_varlen(*([None] * 6), ctypes.cast(off, ctypes.c_void_p), 2, 64, 4, 2, 128, 0.1,
                                   None, None, 0, None, None, None, 0, None)
    assert st == 1  # null pointers


def test_packed_lengths_mix():
    """The packed workloads' length mix: sums to T, every length a positive
    multiple of B within [B, hi], deterministic in the seed."""
    from structured_mask_attention_gb300.inputs import WORKLOADS, packed_lengths, workload_lengths
    for name in ("packed-128k", "batch-64x2k"):
        w = WORKLOADS[name]
        lens = workload_lengths(name)
        assert sum(lens) == w["T"]
        assert all(n % w["B"] == 0 and w["B"] <= n <= w["hi"] for n in lens)
        assert all(n >= w["lo"] for n in lens[:-1])
        assert lens == workload_lengths(name)
    assert workload_lengths("batch-64x2k") == [2048] * 64
    assert packed_lengths(4096, 128, 256, 1024, seed=1) != packed_lengths(4096, 128, 256, 1024, seed=2)


def test_noalloc_size_limit_edge_on_host(lib):
    """The allocation-free backward's array holds 256 + 8 * Hq * L bytes for
    Hq * L up to 4194272: at exactly the limit the size check passes and the
    null pointers are what is rejected (BDLM_ERR_INVALID_ARG); one block more
    is rejected by the size check (BDLM_ERR_WORKSPACE).  Both are decided on
    the host before any device call."""
    f = lib.bdlm_attn_bwd_noalloc
    st = f(*([None] * 12), 4194272, 32, 1, 1, 128, 0.088, *([None] * 6), 0, None)
    assert st == 1, (st, m.bdlm_last_error())
    assert "null pointer" in m.bdlm_last_error()
    st = f(*([None] * 12), 4194304, 32, 1, 1, 128, 0.088, *([None] * 6), 0, None)
    assert st == 4, (st, m.bdlm_last_error())
    assert "4194272" in m.bdlm_last_error()


def test_binding_signatures_match_header():
    """Every function the Python binding declares to ctypes exists in the C
    header with the same number of parameters, and every header function
    has a binding signature."""
    import re
    hdr = open(m.HEADER_PATH).read()
    hdr = re.sub(r"/\*.*?\*/", "", hdr, flags=re.S)
    for name, (_res, args) in m._SIGS.items():
        mm = re.search(r"\b" + name + r"\s*\((.*?)\);", hdr, flags=re.S)
        assert mm, name
        params = [p.strip() for p in mm.group(1).split(",") if p.strip() and p.strip() != "void"]
        assert len(params) == len(args), (name, len(params), len(args))
    assert set(m.header_functions()) == set(m._SIGS)
