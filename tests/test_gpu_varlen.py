"""Packed variable-length batches (batch > 1) through the C ABI, each
sequence's slice checked against the fp64 oracle run on that sequence alone
(sequences do not attend to each other)."""
from __future__ import annotations

import math

import numpy as np
import pytest

import oracle.bdlm_oracle as orc
from structured_mask_attention_gb300.inputs import make_numpy
from tests.parity_util import check_lse, check_rel, to_dev, to_np

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

NAMES = ("Qc", "Kc", "Vc", "Qn", "Kn", "Vn", "dOc", "dOn")


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import structured_mask_attention_gb300 as m
    m.load_library()
    return m


def _batch(lens, Hq, Hkv, d, seed):
    """Per-sequence seeded inputs, packed along the token dimension."""
    per = [make_numpy(L, Hq, Hkv, d, seed=seed + i) for i, L in enumerate(lens)]
    packed = {k: np.concatenate([p[k] for p in per], axis=0) for k in NAMES}
    return per, packed


@pytest.mark.parametrize("lens,B,Hq,Hkv,d", [
    ((256, 512, 128, 384), 64, 4, 2, 128),   # mixed lengths, blocks smaller than a tile
    ((1024, 1024, 1024), 128, 2, 1, 128),     # equal lengths: a plain batch of 3
    ((320, 96, 640), 32, 3, 3, 64),           # ragged tails in every sequence, d = 64
    ((128,), 128, 2, 2, 128),                 # one sequence through the batch path
    (tuple(64 * ((7 * i) % 5 + 1) for i in range(40)), 64, 2, 1, 64),  # 40 sequences, 64..320 rows
])
@pytest.mark.parametrize("order", ["seq", "lpt"])
def test_varlen_against_oracle_per_sequence(lib, lens, B, Hq, Hkv, d, order, monkeypatch):
    """order: the default work list (sequence-major, expanded on the device)
    and the longest-first ablation (built on the host)."""
    m = lib
    monkeypatch.setenv("BDLM_VARLEN_ORDER", order)
    per, packed = _batch(lens, Hq, Hkv, d, seed=sum(lens) + B)
    dev = {k: to_dev(v, torch) for k, v in packed.items()}
    sc = 1.0 / math.sqrt(d)
    ins = [dev[k] for k in NAMES[:6]]
    Oc, On, LSEc, LSEn = m.bdlm_attn_fwd_varlen(*ins, lens, B, sc)
    grads = m.bdlm_attn_bwd_varlen(*ins, Oc, On, dev["dOc"], dev["dOn"], LSEc, LSEn, lens, B, sc,
                                   g_dtype=torch.float32)
    torch.cuda.synchronize()
    off = np.concatenate([[0], np.cumsum(lens)])
    for s, X in enumerate(per):
        a, b = int(off[s]), int(off[s + 1])
        X64 = {k: v.astype(np.float64) for k, v in X.items()}
        ref = orc.fwd_blockwise(*[X64[k] for k in NAMES[:6]], B, sc)
        gref = orc.bwd_blockwise(*[X64[k] for k in NAMES], B, sc)
        check_rel(f"Oc[{s}]", to_np(Oc)[a:b], ref[0])
        check_rel(f"On[{s}]", to_np(On)[a:b], ref[1])
        check_lse(f"LSEc[{s}]", to_np(LSEc)[:, a:b], ref[2])
        check_lse(f"LSEn[{s}]", to_np(LSEn)[:, a:b], ref[3])
        for name, g, r in zip(("dQc", "dKc", "dVc", "dQn", "dKn", "dVn"), grads, gref):
            check_rel(f"{name}[{s}]", to_np(g)[a:b], r)


def test_varlen_rejects_bad_offsets(lib):
    m = lib
    per, packed = _batch((256, 192), 2, 1, 64, seed=3)
    dev = {k: to_dev(v, torch) for k, v in packed.items()}
    ins = [dev[k] for k in NAMES[:6]]
    with pytest.raises(m.BdlmError) as e:
        m.bdlm_attn_fwd_varlen(*ins, (256, 192), 128)   # 192 is not a multiple of B = 128
    assert e.value.status == 2


def test_varlen_refuses_graph_capture(lib):
    """The packed calls copy host data and return BDLM_ERR_UNSUPPORTED (6)
    inside a stream capture, before enqueuing anything."""
    m = lib
    lens = (256, 128)
    per, packed = _batch(lens, 2, 1, 64, seed=5)
    dev = {k: to_dev(v, torch) for k, v in packed.items()}
    ins = [dev[k] for k in NAMES[:6]]
    T = sum(lens)
    out = (torch.empty((T, 2, 64), dtype=torch.bfloat16, device="cuda"),
           torch.empty((T, 2, 64), dtype=torch.bfloat16, device="cuda"),
           torch.empty((2, T), dtype=torch.float32, device="cuda"),
           torch.empty((2, T), dtype=torch.float32, device="cuda"))
    ws = torch.empty(m.bdlm_workspace_size_varlen(m.OP_FWD, lens, 2, 1, 64), dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    status = None
    with torch.cuda.stream(side):
        graph.capture_begin()
        try:
            m.bdlm_attn_fwd_varlen(*ins, lens, 64, out=out, workspace=ws)
        except m.BdlmError as e:
            status = e.status
        finally:
            graph.capture_end()
    assert status == 6
    # the library still works on the same buffers afterwards
    m.bdlm_attn_fwd_varlen(*ins, lens, 64, out=out, workspace=ws)
    torch.cuda.synchronize()
    assert torch.isfinite(out[0].float()).all()


def test_varlen_many_sequences(lib):
    """1536 sequences (the work-list directory and its device expansion at
    scale): sampled sequences against the oracle, each computed alone."""
    from structured_mask_attention_gb300.inputs import make_torch
    m = lib
    B, Hq, Hkv, d = 64, 2, 1, 64
    lens = [64 * (1 + (7 * i) % 3) for i in range(1536)]  # 64, 128 or 192 tokens
    T = sum(lens)
    X = make_torch(T, Hq, Hkv, d, seed=11, device="cuda")
    ins = [X[k] for k in NAMES[:6]]
    sc = 1.0 / math.sqrt(d)
    Oc, On, LSEc, LSEn = m.bdlm_attn_fwd_varlen(*ins, lens, B, sc)
    grads = m.bdlm_attn_bwd_varlen(*ins, Oc, On, X["dOc"], X["dOn"], LSEc, LSEn, lens, B, sc,
                                   g_dtype=torch.float32)
    torch.cuda.synchronize()
    off = np.concatenate([[0], np.cumsum(lens)])
    for s in (0, 1, 2, 777, 1535):
        a, b = int(off[s]), int(off[s + 1])
        X64 = {k: to_np(X[k][a:b]) for k in NAMES}
        ref = orc.fwd_blockwise(*[X64[k] for k in NAMES[:6]], B, sc)
        gref = orc.bwd_blockwise(*[X64[k] for k in NAMES], B, sc)
        check_rel(f"Oc[{s}]", to_np(Oc[a:b]), ref[0])
        check_rel(f"On[{s}]", to_np(On[a:b]), ref[1])
        check_lse(f"LSEc[{s}]", to_np(LSEc[:, a:b]), ref[2])
        check_lse(f"LSEn[{s}]", to_np(LSEn[:, a:b]), ref[3])
        for name, g, r in zip(("dQc", "dKc", "dVc", "dQn", "dKn", "dVn"), grads, gref):
            check_rel(f"{name}[{s}]", to_np(g[a:b]), r)
