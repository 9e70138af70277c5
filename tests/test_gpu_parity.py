"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on the
same seeded bf16 inputs, at sizes the oracle finishes in seconds, covering
several tiles, ragged tails and the degenerate block sizes."""
from __future__ import annotations

import math

import numpy as np
import pytest

import oracle.bdlm_oracle as orc
from structured_mask_attention_gb300.inputs import WORKLOADS, make_numpy
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


def _run_case(m, L, B, Hq, Hkv, d, seed=0, lognormal=0.0, bwd=True, o_dtype=None, brute=False):
    X = make_numpy(L, Hq, Hkv, d, seed=seed, lognormal_sigma=lognormal)
    dev = {k: to_dev(v, torch) for k, v in X.items()}
    X64 = {k: v.astype(np.float64) for k, v in X.items()}
    sc = 1.0 / math.sqrt(d)
    ins = [dev[k] for k in NAMES[:6]]
    Oc, On, LSEc, LSEn = m.bdlm_attn_fwd(*ins, B, sc, o_dtype=o_dtype)
    fwd_ref = (orc.fwd_brute if brute else orc.fwd_blockwise)(*[X64[k] for k in NAMES[:6]], B, sc)
    check_rel("Oc", to_np(Oc), fwd_ref[0])
    check_rel("On", to_np(On), fwd_ref[1])
    check_lse("LSEc", to_np(LSEc), fwd_ref[2])
    check_lse("LSEn", to_np(LSEn), fwd_ref[3])
    if not bwd:
        return
    # the GPU backward reads its own (bf16) O; the oracle uses its own O
    if Oc.dtype != torch.bfloat16:
        Oc, On = Oc.to(torch.bfloat16), On.to(torch.bfloat16)
    grads = m.bdlm_attn_bwd(*ins, Oc, On, dev["dOc"], dev["dOn"], LSEc, LSEn, B, sc, g_dtype=torch.float32)
    gref = (orc.bwd_brute if brute else orc.bwd_blockwise)(*[X64[k] for k in NAMES], B, sc)
    for name, g, r in zip(("dQc", "dKc", "dVc", "dQn", "dKn", "dVn"), grads, gref):
        check_rel(name, to_np(g), r)


def test_tiny_workload_brute(lib):
    w = WORKLOADS["tiny"]
    _run_case(lib, w["L"], w["B"], w["Hq"], w["Hkv"], w["d"], seed=0, brute=True)


@pytest.mark.parametrize("L,B,Hq,Hkv,d", [
    (200, 40, 3, 1, 128),    # ragged q/k tail, blocks straddle tiles
    (384, 128, 4, 2, 128),   # tile-aligned blocks, GQA 2
    (160, 1, 2, 1, 64),      # token-causal clean stream
    (192, 192, 2, 2, 128),   # one block: full attention per stream
    (512, 256, 2, 1, 128),   # blocks larger than a tile
    (640, 160, 5, 1, 64),    # GQA 5, blocks not a multiple of the tile
    (96, 32, 1, 1, 128),     # shorter than one tile
    (1024, 16, 2, 1, 64),    # many small blocks: every key step partially masked
    (768, 96, 4, 4, 128),    # 256-row forward items spanning three blocks, MHA
])
def test_shapes(lib, L, B, Hq, Hkv, d):
    _run_case(lib, L, B, Hq, Hkv, d, seed=L + B)


def test_fp32_output(lib):
    _run_case(lib, 256, 64, 2, 1, 128, seed=3, o_dtype=torch.float32, bwd=False)


def test_lognormal_rows(lib):
    _run_case(lib, 1024, 128, 4, 1, 128, seed=4, lognormal=0.5)


def test_gqa_8k_workload_full(lib):
    w = WORKLOADS["gqa-8k"]
    _run_case(lib, w["L"], w["B"], w["Hq"], w["Hkv"], w["d"], seed=0)


def _sharded(m, X, L, B, Hq, Hkv, d, P, sc):
    dev = {k: to_dev(v, torch) for k, v in X.items()}
    ins = [dev[k] for k in NAMES[:6]]
    bounds = orc.shard_bounds(L, P)
    parts = [m.bdlm_attn_fwd_shard(*ins, B, lo, hi, False, sc) for (lo, hi) in bounds]
    parts.append(m.bdlm_attn_fwd_shard(*ins, B, 0, 0, True, sc))
    Oc, LSEc = m.bdlm_lse_merge([p[0] for p in parts], [p[2] for p in parts], o_dtype=torch.float32)
    On, LSEn = m.bdlm_lse_merge([p[1] for p in parts], [p[3] for p in parts], o_dtype=torch.float32)
    return dev, ins, parts, (Oc, On, LSEc, LSEn), bounds


@pytest.mark.parametrize("L,B,P", [(256, 32, 8), (4096, 128, 8), (4096, 1024, 8), (4096, 512, 8), (4096, 256, 8)])
def test_shard_and_merge(lib, L, B, P):
    """CSBP on one GPU: per-shard partials (each checked against the oracle's
    partial), their LSE merge, and the sharded backward."""
    m = lib
    Hq, Hkv, d = (8, 4, 128) if L >= 4096 else (2, 1, 64)
    X = make_numpy(L, Hq, Hkv, d, seed=P + B)
    X64 = {k: v.astype(np.float64) for k, v in X.items()}
    sc = 1.0 / math.sqrt(d)
    dev, ins, parts, merged, bounds = _sharded(m, X, L, B, Hq, Hkv, d, P, sc)
    (ref_fwd, ref_parts) = orc.fwd_sharded(*[X64[k] for k in NAMES[:6]], B, sc, P)
    for k, (gp, rp) in enumerate(zip(parts, ref_parts)):
        check_lse(f"LSEp_c[{k}]", to_np(gp[2]), rp[2])
        check_lse(f"LSEp_n[{k}]", to_np(gp[3]), rp[3])
        check_rel(f"Op_c[{k}]", to_np(gp[0]), rp[0])
        check_rel(f"Op_n[{k}]", to_np(gp[1]), rp[1])
    for name, g, r in zip(("Oc", "On"), merged[:2], ref_fwd[:2]):
        check_rel(name, to_np(g), r)
    check_lse("LSEc", to_np(merged[2]), ref_fwd[2])
    check_lse("LSEn", to_np(merged[3]), ref_fwd[3])
    # sharded backward with the merged statistics
    Oc_b, On_b = merged[0].to(torch.bfloat16), merged[1].to(torch.bfloat16)
    Dc = m.bdlm_bwd_preprocess(Oc_b, dev["dOc"])
    Dn = m.bdlm_bwd_preprocess(On_b, dev["dOn"])
    z = lambda H: torch.zeros((L, H, d), dtype=torch.float32, device="cuda")
    dQc, dQn = z(Hq), z(Hq)
    dKc, dVc, dKn, dVn = z(Hkv), z(Hkv), z(Hkv), z(Hkv)
    for (lo, hi) in bounds:
        m.bdlm_attn_bwd_shard(*ins, dev["dOc"], dev["dOn"], merged[2], merged[3], Dc, Dn, B, lo, hi, False,
                              dQc, dQn, dKc, dVc, dKn, dVn, sc)
    m.bdlm_attn_bwd_shard(*ins, dev["dOc"], dev["dOn"], merged[2], merged[3], Dc, Dn, B, 0, 0, True,
                          dQc, dQn, dKc, dVc, dKn, dVn, sc)
    gref = orc.bwd_blockwise(*[X64[k] for k in NAMES], B, sc)
    for name, g, r in zip(("dQc", "dKc", "dVc", "dQn", "dKn", "dVn"), (dQc, dKc, dVc, dQn, dKn, dVn), gref):
        check_rel(name, to_np(g), r)


def test_sharded_vs_unsharded_production_report(lib):
    """Production path: shard-and-merge vs the unsharded kernel, both with
    fp32 outputs, same inputs.  Both paths round P to bf16 (relative 2^-9)
    against their own running maxima, so they differ by that rounding as
    well as by summation order; the difference is reported and held to the
    parity tolerance against the unsharded output (2e-2 * max|O|).  The
    rigorous bound, 2 * 2^-9 * max|V| (each O row is a convex combination of
    V rows), is printed beside it.  The exact comparison (same P in both
    paths, 1e-5) is test_refmax_shard_and_merge_within_1e5."""
    m = lib
    L, B, Hq, Hkv, d, P = 4096, 256, 8, 4, 128, 8
    X = make_numpy(L, Hq, Hkv, d, seed=21)
    sc = 1.0 / math.sqrt(d)
    dev, ins, parts, merged, _ = _sharded(m, X, L, B, Hq, Hkv, d, P, sc)
    Oc, On, LSEc, LSEn = m.bdlm_attn_fwd(*ins, B, sc, o_dtype=torch.float32)
    dO = max((merged[0] - Oc).abs().max().item(), (merged[1] - On).abs().max().item())
    dL = max((merged[2] - LSEc).abs().max().item(), (merged[3] - LSEn).abs().max().item())
    omax = max(Oc.abs().max().item(), On.abs().max().item())
    vmax = max(abs(X["Vc"]).max(), abs(X["Vn"]).max())
    print(f"production sharded vs unsharded: max|dO| = {dO:.3e} (2e-2 max|O| = {2e-2 * omax:.3e}; "
          f"2^-8 max|V| = {2 ** -8 * vmax:.3e}), max|dLSE| = {dL:.3e}")
    assert dL <= 1e-4
    assert dO <= 2e-2 * omax


def _refmax_diff(m, ins, L, B, P, sc, Mc, Mn):
    """Verification mode: the unsharded call and the P + 1 partials, all
    rounding P against the same reference; returns the merged and unsharded
    results and their max differences in O and LSE."""
    full = m.bdlm_attn_fwd_shard_refmax(*ins, B, 0, L, True, Mc, Mn, sc)
    step = L // P
    specs = [(s * step, (s + 1) * step, False) for s in range(P)] + [(0, 0, True)]
    parts = [m.bdlm_attn_fwd_shard_refmax(*ins, B, lo, hi, loc, Mc, Mn, sc) for (lo, hi, loc) in specs]
    Oc, LSEc = m.bdlm_lse_merge([p[0] for p in parts], [p[2] for p in parts], o_dtype=torch.float32)
    On, LSEn = m.bdlm_lse_merge([p[1] for p in parts], [p[3] for p in parts], o_dtype=torch.float32)
    del parts
    dO = max((Oc - full[0]).abs().max().item(), (On - full[1]).abs().max().item())
    dL = max((LSEc - full[2]).abs().max().item(), (LSEn - full[3]).abs().max().item())
    return (Oc, On, LSEc, LSEn), full, dO, dL


@pytest.mark.parametrize("B", [128, 256, 512, 1024])
def test_refmax_shard_and_merge_within_1e5(lib, B):
    """Shard-and-merge equals the unsharded computation up to floating-point
    reduction order (Proposition 1; evolve.pub FAQ "Does CSBP change training
    results?"): with every row's probabilities formed against the same fixed
    reference in both paths (the unsharded forward's LSE), P is rounded to
    bf16 identically, and the merged fp32 O and LSE of P = 8 clean shards
    plus the local corrupted partial stay within 1e-5 of the unsharded fp32
    result.  Both are also checked against the oracle."""
    m = lib
    L, Hq, Hkv, d, P = 4096, 8, 4, 128, 8
    X = make_numpy(L, Hq, Hkv, d, seed=100 + B)
    X64 = {k: v.astype(np.float64) for k, v in X.items()}
    sc = 1.0 / math.sqrt(d)
    dev = {k: to_dev(v, torch) for k, v in X.items()}
    ins = [dev[k] for k in NAMES[:6]]
    _, _, Mc, Mn = m.bdlm_attn_fwd(*ins, B, sc, o_dtype=torch.float32)
    merged, full, dO, dL = _refmax_diff(m, ins, L, B, P, sc, Mc, Mn)
    print(f"B={B}: fixed-reference sharded vs unsharded fp32: max|dO| = {dO:.3e}, max|dLSE| = {dL:.3e}")
    assert dO <= 1e-5 and dL <= 1e-5
    ref = orc.fwd_blockwise(*[X64[k] for k in NAMES[:6]], B, sc)
    for tag, res in (("unsharded", full), ("merged", merged)):
        check_rel(f"Oc ({tag})", to_np(res[0]), ref[0])
        check_rel(f"On ({tag})", to_np(res[1]), ref[1])
        check_lse(f"LSEc ({tag})", to_np(res[2]), ref[2])
        check_lse(f"LSEn ({tag})", to_np(res[3]), ref[3])


def test_refmax_rejects_bad_reference(lib):
    m = lib
    X = make_numpy(256, 2, 1, 64, seed=3)
    ins = [to_dev(X[k], torch) for k in NAMES[:6]]
    bad = torch.zeros((2, 128), dtype=torch.float32, device="cuda")
    with pytest.raises(ValueError):
        m.bdlm_attn_fwd_shard_refmax(*ins, 32, 0, 256, True, bad, bad)


def test_deterministic(lib):
    m = lib
    L, B, Hq, Hkv, d = 1024, 128, 4, 2, 128
    X = make_numpy(L, Hq, Hkv, d, seed=9)
    dev = {k: to_dev(v, torch) for k, v in X.items()}
    ins = [dev[k] for k in NAMES[:6]]
    outs = []
    for _ in range(2):
        f = m.bdlm_attn_fwd(*ins, B)
        g = m.bdlm_attn_bwd(*ins, f[0], f[1], dev["dOc"], dev["dOn"], f[2], f[3], B)
        outs.append([t.clone() for t in (*f, *g)])
    for a, b in zip(*outs):
        assert torch.equal(a, b)


def test_work_claiming_leaves_counters_zero_and_order_free(lib, monkeypatch):
    """The persistent CTAs claim items from counters in the workspace header
    (words 8-13: item counter and finished-CTA count of the forward, dK/dV
    and dQ): after each call the last CTA has zeroed them again, even when a
    call finds them dirty (the call clears them first).  Which CTA runs an
    item does not change its outputs: two runs agree bit for bit.  The
    natural-order ablation (BDLM_SCHED=naive, static round robin) lists the
    items in another order, and a query item's clean-key sweep starts at a
    tile set by its list index, so its sums run in another order: equal to
    rounding."""
    m = lib
    L, B, Hq, Hkv, d = 2048, 256, 4, 2, 128
    X = make_numpy(L, Hq, Hkv, d, seed=13)
    dev = {k: to_dev(v, torch) for k, v in X.items()}
    ins = [dev[k] for k in NAMES[:6]]
    wsf = torch.full((m.bdlm_workspace_size(m.OP_FWD, L, B, Hq, Hkv, d),), 0x5A, dtype=torch.uint8, device="cuda")
    wsb = torch.full((m.bdlm_workspace_size(m.OP_BWD, L, B, Hq, Hkv, d),), 0x5A, dtype=torch.uint8, device="cuda")
    outs = []
    for naive in (False, True, False):
        if naive:
            monkeypatch.setenv("BDLM_SCHED", "naive")
        f = m.bdlm_attn_fwd(*ins, B, workspace=wsf)
        g = m.bdlm_attn_bwd(*ins, f[0], f[1], dev["dOc"], dev["dOn"], f[2], f[3], B, workspace=wsb)
        torch.cuda.synchronize()
        monkeypatch.delenv("BDLM_SCHED", raising=False)
        for ws in (wsf, wsb):
            words = ws[:64].view(torch.int32).cpu()
            assert int(words[0]) == 0  # status word: no wait expired
            assert words[8:14].tolist() == [0] * 6
        outs.append([t.clone() for t in (*f, *g)])
    for a, b, c in zip(*outs):
        assert torch.equal(a, c)
        ref = a.float()
        assert (b.float() - ref).abs().max().item() <= 2e-2 * max(ref.abs().max().item(), 1e-6)


def test_watchdog_reports_timeout(lib):
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    assert lib.bdlm_watchdog_selftest(ws, 20000) == 7
    # the context is still usable afterwards
    _run_case(lib, 128, 32, 1, 1, 64, seed=1, bwd=False)


def test_abi_rejects_bad_arguments_on_gpu(lib):
    m = lib
    X = make_numpy(128, 2, 1, 64, seed=2)
    dev = {k: to_dev(v, torch) for k, v in X.items()}
    ins = [dev[k] for k in NAMES[:6]]
    with pytest.raises(m.BdlmError) as e:
        m.bdlm_attn_fwd(*ins, 48)  # 128 % 48 != 0
    assert e.value.status == 2
    ws = torch.zeros(8, dtype=torch.uint8, device="cuda")
    with pytest.raises(m.BdlmError) as e:
        m.bdlm_attn_bwd(*ins, dev["dOc"], dev["dOn"], dev["dOc"], dev["dOn"],
                        torch.zeros(2, 128, device="cuda"), torch.zeros(2, 128, device="cuda"), 32, workspace=ws)
    assert e.value.status == 4


def test_launch_counter_counts_kernels(lib):
    m = lib
    X = make_numpy(256, 2, 1, 64, seed=2)
    dev = {k: to_dev(v, torch) for k, v in X.items()}
    ins = [dev[k] for k in NAMES[:6]]
    n0 = m.bdlm_kernel_launches()
    f = m.bdlm_attn_fwd(*ins, 32)
    m.bdlm_attn_bwd(*ins, f[0], f[1], dev["dOc"], dev["dOn"], f[2], f[3], 32)
    torch.cuda.synchronize()
    assert m.bdlm_kernel_launches() - n0 == 1 + 4  # fwd; 2 preprocess + dK/dV + dQ
