"""GPU parity at the workloads' full sizes, in the launch configuration the
bench uses: the whole problem runs on the device; the fp64 oracle checks
sampled outputs it can compute one by one (rows' O, LSE and dQ; dK/dV of the
last key blocks, which few rows read) and properties that hold at any size
(per KV head, sum_j dK_j = 0 and sum_j dV_j = sum of the group's dO)."""
from __future__ import annotations

import math

import numpy as np
import pytest

import oracle.bdlm_oracle as orc
from structured_mask_attention_gb300.inputs import SHARDED_BLOCK_SIZES, WORKLOADS, make_torch, workload_lengths
from tests.parity_util import check_lse, check_rel

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


def _host_group(X, kvh, G):
    """fp64 host copies of one KV group's heads (query heads kvh*G..+G-1)."""
    out = {}
    for k in NAMES:
        t = X[k]
        sl = slice(kvh * G, (kvh + 1) * G) if t.shape[1] != X["Kc"].shape[1] else slice(kvh, kvh + 1)
        out[k] = t[:, sl].float().cpu().numpy().astype(np.float64)
    return out


def _sample_rows(L, B, rng, n=12):
    rows = {0, L - 1, B - 1, B, L - B, L // 2}
    rows.update(int(x) for x in rng.integers(0, L, n))
    return sorted(r for r in rows if 0 <= r < L)


def _invariants(X, grads, G):
    """Per KV head: sum over both streams' keys of dK is 0 and of dV equals the
    sum of dO over the group's rows.  Two error terms bound the deviation:
    bf16 rounding of P and dS, random across ~sqrt(n) keys, and the tensor
    cores' fp32 accumulation over ~10^4 MMA steps per gradient element, which
    truncates and shrinks each element by up to ~1e-3 relative (measured
    shrinkage of the dV sums: 2e-4 to 7e-4 at L = 32768)."""
    dQc, dKc, dVc, dQn, dKn, dVn = [g.double() for g in grads]
    Hkv = dKc.shape[1]
    n = 2 * dKc.shape[0]
    acc = 1e-3
    sK = dKc.sum(0) + dKn.sum(0)
    rmsK = torch.sqrt((dKc.square().sum(0) + dKn.square().sum(0)) / n)
    l1K = dKc.abs().sum(0) + dKn.abs().sum(0)
    bound = 2e-2 * math.sqrt(n) * rmsK + acc * l1K + 1e-6
    print(f"  sum dK: max |dev| / bound = {float((sK.abs() / bound).max()):.3f}")
    assert (sK.abs() <= bound).all()
    sV = dVc.sum(0) + dVn.sum(0)
    dO = (X["dOc"].double() + X["dOn"].double()).sum(0).reshape(Hkv, G, -1).sum(1)
    rmsV = torch.sqrt((dVc.square().sum(0) + dVn.square().sum(0)) / n)
    l1V = dVc.abs().sum(0) + dVn.abs().sum(0)
    bound = 2e-2 * math.sqrt(n) * rmsV + acc * l1V + 1e-6
    print(f"  sum dV: max |dev| / bound = {float(((sV - dO).abs() / bound).max()):.3f}")
    assert ((sV - dO).abs() <= bound).all()


def _check_sequence(X, grads, outs, B, sc, G, kvh, rng, n_rows):
    """Sampled oracle parity of one sequence (X, grads, outs: its slices)."""
    Oc, On, LSEc, LSEn = outs
    L = X["Qc"].shape[0]
    N = L // B
    H = _host_group(X, kvh, G)
    hx = [H[k] for k in NAMES]
    rows = _sample_rows(L, B, rng, n_rows)
    for stream, O, LSE, dQ in (("c", Oc, LSEc, grads[0]), ("n", On, LSEn, grads[3])):
        for hh in (0, G - 1):
            h = kvh * G + hh
            o, lse = orc.fwd_rows(*hx[:6], B, sc, stream, hh, rows)
            check_rel(f"O{stream}[h={h}] rows", O[rows, h].float().cpu().numpy(), o)
            check_lse(f"LSE{stream}[h={h}] rows", LSE[h, rows].cpu().numpy(), lse)
            dq = orc.dq_rows(*hx, B, sc, stream, hh, rows)
            check_rel(f"dQ{stream}[h={h}] rows", dQ[rows, h].float().cpu().numpy(), dq)
    tail = sorted({N - 1, max(N - 2, 0)})
    outc, outn = orc.dkv_tail_blocks(*hx, B, sc, 0, tail, sorted({N - 1, 0, N // 2}))
    for (blocks, dK, dV, tag) in ((outc, grads[1], grads[2], "c"), (outn, grads[4], grads[5], "n")):
        for j, (rk, rv) in blocks.items():
            check_rel(f"dK{tag}[kvh={kvh}, block {j}]", dK[j * B:(j + 1) * B, kvh].float().cpu().numpy(), rk)
            check_rel(f"dV{tag}[kvh={kvh}, block {j}]", dV[j * B:(j + 1) * B, kvh].float().cpu().numpy(), rv)


@pytest.mark.parametrize("name", ["packed-128k", "batch-64x2k"])
def test_packed_batch_workload(lib, name):
    """Full-size packed batch through the packed calls: invariants over the
    whole batch, and sampled oracle parity of the first, the longest and the
    last sequence, each computed on that sequence alone."""
    m = lib
    w = WORKLOADS[name]
    T, B, Hq, Hkv, d = w["T"], w["B"], w["Hq"], w["Hkv"], w["d"]
    G = Hq // Hkv
    lens = workload_lengths(name)
    off = np.concatenate([[0], np.cumsum(lens)]).astype(int)
    X = make_torch(T, Hq, Hkv, d, seed=0, device="cuda")
    ins = [X[k] for k in NAMES[:6]]
    sc = 1.0 / math.sqrt(d)
    outs = m.bdlm_attn_fwd_varlen(*ins, lens, B, sc)
    grads = m.bdlm_attn_bwd_varlen(*ins, outs[0], outs[1], X["dOc"], X["dOn"], outs[2], outs[3], lens, B, sc,
                                   g_dtype=torch.float32)
    torch.cuda.synchronize()
    assert all(torch.isfinite(t).all() for t in (*outs, *grads))
    _invariants(X, grads, G)
    rng = np.random.default_rng(T + len(lens))
    for s in sorted({0, int(np.argmax(lens)), len(lens) - 1}):
        a, b = int(off[s]), int(off[s + 1])
        print(f"sequence {s}: rows [{a}, {b})")
        Xs = {k: X[k][a:b] for k in NAMES}
        os_ = (outs[0][a:b], outs[1][a:b], outs[2][:, a:b], outs[3][:, a:b])
        gs = [g[a:b] for g in grads]
        _check_sequence(Xs, gs, os_, B, sc, G, kvh=s % Hkv, rng=rng, n_rows=6)


def _full_size_case(m, name, lognormal=0.0, groups=(0,), n_rows=12):
    w = WORKLOADS[name]
    L, B, Hq, Hkv, d = w["L"], w["B"], w["Hq"], w["Hkv"], w["d"]
    G = Hq // Hkv
    X = make_torch(L, Hq, Hkv, d, seed=0, lognormal_sigma=lognormal, device="cuda")
    ins = [X[k] for k in NAMES[:6]]
    sc = 1.0 / math.sqrt(d)
    Oc, On, LSEc, LSEn = m.bdlm_attn_fwd(*ins, B, sc)
    grads = m.bdlm_attn_bwd(*ins, Oc, On, X["dOc"], X["dOn"], LSEc, LSEn, B, sc, g_dtype=torch.float32)
    torch.cuda.synchronize()
    assert all(torch.isfinite(t).all() for t in (Oc, On, LSEc, LSEn, *grads))
    _invariants(X, grads, G)
    rng = np.random.default_rng(L)
    N = L // B
    for kvh in groups:
        H = _host_group(X, kvh, G)
        hx = [H[k] for k in NAMES]
        rows = _sample_rows(L, B, rng, n_rows)
        for stream, O, LSE, dQ in (("c", Oc, LSEc, grads[0]), ("n", On, LSEn, grads[3])):
            for hh in (0, G - 1):
                h = kvh * G + hh
                o, lse = orc.fwd_rows(*hx[:6], B, sc, stream, hh, rows)
                check_rel(f"O{stream}[h={h}] rows", O[rows, h].float().cpu().numpy(), o)
                check_lse(f"LSE{stream}[h={h}] rows", LSE[h, rows].cpu().numpy(), lse)
                dq = orc.dq_rows(*hx, B, sc, stream, hh, rows)
                check_rel(f"dQ{stream}[h={h}] rows", dQ[rows, h].cpu().numpy(), dq)
        outc, outn = orc.dkv_tail_blocks(*hx, B, sc, 0, [N - 1, N - 2], [N - 1, 0, N // 2])
        for (blocks, dK, dV, tag) in ((outc, grads[1], grads[2], "c"), (outn, grads[4], grads[5], "n")):
            for j, (rk, rv) in blocks.items():
                check_rel(f"dK{tag}[kvh={kvh}, block {j}]", dK[j * B:(j + 1) * B, kvh].cpu().numpy(), rk)
                check_rel(f"dV{tag}[kvh={kvh}, block {j}]", dV[j * B:(j + 1) * B, kvh].cpu().numpy(), rv)


def test_gqa_32k_workload(lib):
    _full_size_case(lib, "gqa-32k", groups=(0, 7))


def test_gqa_32k_lognormal_workload(lib):
    _full_size_case(lib, "gqa-32k", lognormal=0.5, groups=(3,))


def test_long_128k_workload(lib):
    _full_size_case(lib, "long-128k", groups=(0, 5), n_rows=8)


@pytest.mark.parametrize("B", SHARDED_BLOCK_SIZES)
def test_sharded_256k_workload(lib, B):
    """Full size: P = 8 clean shards + the local corrupted partial, merged,
    against the unsharded kernel (fp32 outputs) on the same inputs, and the
    first 4096 rows of both streams against the oracle on the L = 4096 prefix
    problem (rows of the first blocks read only keys of the first blocks)."""
    m = lib
    w = WORKLOADS["sharded-256k"]
    L, Hq, Hkv, d, P = w["L"], w["Hq"], w["Hkv"], w["d"], w["P"]
    X = make_torch(L, Hq, Hkv, d, seed=B, device="cuda")
    ins = [X[k] for k in NAMES[:6]]
    sc = 1.0 / math.sqrt(d)
    bounds = orc.shard_bounds(L, P)
    Oc_u, On_u, LSEc_u, LSEn_u = m.bdlm_attn_fwd(*ins, B, sc, o_dtype=torch.float32)
    parts = []
    for (lo, hi) in bounds:
        parts.append(m.bdlm_attn_fwd_shard(*ins, B, lo, hi, False, sc))
    parts.append(m.bdlm_attn_fwd_shard(*ins, B, 0, 0, True, sc))
    Oc, LSEc = m.bdlm_lse_merge([p[0] for p in parts], [p[2] for p in parts], o_dtype=torch.float32)
    On, LSEn = m.bdlm_lse_merge([p[1] for p in parts], [p[3] for p in parts], o_dtype=torch.float32)
    torch.cuda.synchronize()
    dO = max((Oc - Oc_u).abs().max().item(), (On - On_u).abs().max().item())
    dL = max((LSEc - LSEc_u).abs().max().item(), (LSEn - LSEn_u).abs().max().item())
    # Both paths round P to bf16 (relative 2^-9) against different running
    # maxima; each O row is a convex combination of V rows, so the two paths
    # differ by at most 2 * 2^-9 * max|V|.
    vmax = max(X["Vc"].abs().max().item(), X["Vn"].abs().max().item())
    print(f"B={B}: sharded vs unsharded fp32 max|dO| = {dO:.3e} (bound {2 ** -8 * vmax:.3e}), "
          f"max|dLSE| = {dL:.3e}")
    assert dL <= 1e-4 and dO <= 2 ** -8 * vmax
    # merge kernel vs fp64 merge of the same fp32 partials, on sampled rows
    rng = np.random.default_rng(B)
    rows = np.sort(rng.choice(L, 64, replace=False))
    for (Op_idx, L_idx, got) in ((0, 2, Oc), (1, 3, On)):
        Os = [p[Op_idx][rows].double().cpu().numpy() for p in parts]
        Ls = [p[L_idx][:, rows].double().cpu().numpy() for p in parts]
        ref, _ = orc.lse_merge(Os, Ls)
        err = np.abs(got[rows].double().cpu().numpy() - ref).max()
        assert err <= 1e-5, err
    del parts
    # prefix slice against the oracle (both streams, all heads of KV group 0)
    Ls_ = 4096
    G = Hq // Hkv
    H = {k: X[k][:Ls_, :G if X[k].shape[1] == Hq else 1].float().cpu().numpy().astype(np.float64) for k in NAMES}
    ref = orc.fwd_blockwise(*[H[k] for k in NAMES[:6]], B, sc)
    check_rel("Oc prefix", Oc[:Ls_, :G].cpu().numpy(), ref[0])
    check_rel("On prefix", On[:Ls_, :G].cpu().numpy(), ref[1])
    check_lse("LSEc prefix", LSEc[:G, :Ls_].cpu().numpy(), ref[2])
    check_lse("LSEn prefix", LSEn[:G, :Ls_].cpu().numpy(), ref[3])
