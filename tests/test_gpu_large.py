"""GPU parity at the workloads' full sizes, in the launch configuration the
bench uses: the whole problem runs on the device; the fp64 oracle checks
whole KV-head groups (every row and key of the group: O, LSE, dQ, dK, dV of
both streams at L = 32768; O and LSE of every row, and dK/dV of the clean key
blocks read by the most rows, at L = 131072), sampled outputs it can compute
one by one (rows' O, LSE and dQ; dK/dV of single key blocks), and properties
that hold at any size (per KV head, sum_j dK_j = 0 and sum_j dV_j = sum of
the group's dO).  The oracle runs in worker processes over row blocks
(tests/oracle_pool.py)."""
from __future__ import annotations

import math

import numpy as np
import pytest

import oracle.bdlm_oracle as orc
from structured_mask_attention_gb300.inputs import SHARDED_BLOCK_SIZES, WORKLOADS, make_torch, workload_lengths
from tests import oracle_pool
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
    shrinkage of the dV sums: 2e-4 to 7e-4 at L = 32768).  The longest
    accumulations are also compared with the oracle directly (every key of a
    KV group at L = 32768; clean blocks 0 and N/2, read by the most rows, at
    L = 131072), at the parity tolerance."""
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


def _group_oracle(X, outs, grads, kvh, G, B, sc, full_bwd, dkv_clean_blocks=()):
    """One KV-head group against the oracle: O and LSE of every row of both
    streams; with full_bwd, dQ of every row and dK/dV of every key; dK/dV of
    the listed clean key blocks (computed from the full-row statistics, as the
    gradient of those keys alone)."""
    L = X["Qc"].shape[0]
    H = _host_group(X, kvh, G)
    sl = slice(kvh * G, (kvh + 1) * G)
    fo = oracle_pool.forward(H, B, sc)
    Oc, On, LSEc, LSEn = outs
    tag = f"[kvh={kvh}, all rows]"
    check_rel(f"Oc{tag}", Oc[:, sl].float().cpu().numpy(), fo[0])
    check_rel(f"On{tag}", On[:, sl].float().cpu().numpy(), fo[1])
    check_lse(f"LSEc{tag}", LSEc[sl].cpu().numpy(), fo[2])
    check_lse(f"LSEn{tag}", LSEn[sl].cpu().numpy(), fo[3])
    stats = (fo[2], fo[3], oracle_pool.preprocess(fo[0], H["dOc"]), oracle_pool.preprocess(fo[1], H["dOn"]))
    dQc, dKc, dVc, dQn, dKn, dVn = grads
    kv = slice(kvh, kvh + 1)
    if full_bwd:
        g = oracle_pool.backward(H, stats, B, sc)
        for name, got, ref in (("dQc", dQc[:, sl], g[0]), ("dKc", dKc[:, kv], g[1]), ("dVc", dVc[:, kv], g[2]),
                               ("dQn", dQn[:, sl], g[3]), ("dKn", dKn[:, kv], g[4]), ("dVn", dVn[:, kv], g[5])):
            check_rel(f"{name}{tag}", got.float().cpu().numpy(), ref)
    for j in dkv_clean_blocks:
        g = oracle_pool.backward(H, stats, B, sc, kv_begin=j * B, kv_end=(j + 1) * B, include_local=False)
        r = slice(j * B, (j + 1) * B)
        check_rel(f"dKc[kvh={kvh}, clean block {j} of {L // B}]", dKc[r, kv].float().cpu().numpy(), g[1][r])
        check_rel(f"dVc[kvh={kvh}, clean block {j} of {L // B}]", dVc[r, kv].float().cpu().numpy(), g[2][r])


def _full_size_case(m, name, lognormal=0.0, groups=(0,), n_rows=12, full_group=None, full_bwd=True,
                    dkv_clean_blocks=(), shape=None):
    w = shape if shape is not None else WORKLOADS[name]
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
    if full_group is not None:
        _group_oracle(X, (Oc, On, LSEc, LSEn), grads, full_group, G, B, sc, full_bwd, dkv_clean_blocks)


def test_gqa_32k_workload(lib):
    """L = 32768, B = 256, 40/8 heads: sampled rows of KV groups 0 and 7,
    and all of KV group 2 (5 query heads) against the oracle."""
    _full_size_case(lib, "gqa-32k", groups=(0, 7), full_group=2)


def test_gqa_32k_lognormal_workload(lib):
    """The same with LogNormal(0, 0.5) per-token Q/K factors: all of KV
    group 3 against the oracle."""
    _full_size_case(lib, "gqa-32k", lognormal=0.5, groups=(3,), full_group=3)


def test_long_128k_workload(lib):
    """L = 131072, B = 512, 16/8 heads: sampled rows of groups 0 and 5; O and
    LSE of every row of group 6; dK/dV of group 6's clean key blocks 0 and
    N/2, which accumulate over the most rows (block 0: every row of both
    streams but the corrupted block 0, 2 x 262144 - 512 rows)."""
    N = WORKLOADS["long-128k"]["L"] // WORKLOADS["long-128k"]["B"]
    _full_size_case(lib, "long-128k", groups=(0, 5), n_rows=8, full_group=6, full_bwd=False,
                    dkv_clean_blocks=(0, N // 2))


def test_head_dim_64_long_lists(lib):
    """d = 64 (the kernels' other head size) at L = 65536, B = 512, 8/4 heads:
    256 query tiles per stream, so the forward and dQ lists are blocked per
    KV head, and every CTA claims many items of each list.  Invariants over
    all heads, sampled rows of KV groups 0 and 3, tail and long-accumulation
    dK/dV blocks."""
    shape = {"L": 65536, "B": 512, "Hq": 8, "Hkv": 4, "d": 64}
    _full_size_case(lib, "d64-64k", groups=(0, 3), n_rows=8, shape=shape)


@pytest.mark.parametrize("B", SHARDED_BLOCK_SIZES)
def test_sharded_256k_workload(lib, B):
    """Full size, L = 262144, 8/4 heads: P = 8 clean shards + the local
    corrupted partial, merged, against the unsharded kernel on the same
    inputs, forward and backward:
      * production path: reported, held to 2e-2 * max|unsharded|;
      * fixed-reference mode (same P in both paths): max |dO|, |dLSE| <= 1e-5;
      * the merge kernel against the fp64 merge of the same partials, 1e-5;
      * the 9-partial backward (fp32 dQ accumulated in shard order, dK/dV
        per shard) against the unsharded backward;
      * the first 4096 rows of both streams (O, LSE, dQ) against the oracle
        on the L = 4096 prefix problem (those rows read only keys of the
        first 4096 tokens)."""
    m = lib
    w = WORKLOADS["sharded-256k"]
    L, Hq, Hkv, d, P = w["L"], w["Hq"], w["Hkv"], w["d"], w["P"]
    G = Hq // Hkv
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
    omax = max(Oc_u.abs().max().item(), On_u.abs().max().item())
    vmax = max(X["Vc"].abs().max().item(), X["Vn"].abs().max().item())
    print(f"B={B}: production sharded vs unsharded fp32 max|dO| = {dO:.3e} (2e-2 max|O| = {2e-2 * omax:.3e}; "
          f"2^-8 max|V| = {2 ** -8 * vmax:.3e}), max|dLSE| = {dL:.3e}")
    assert dL <= 1e-4 and dO <= 2e-2 * omax
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
    Hp = {k: X[k][:Ls_, :G if X[k].shape[1] == Hq else 1].float().cpu().numpy().astype(np.float64) for k in NAMES}
    ref = orc.fwd_blockwise(*[Hp[k] for k in NAMES[:6]], B, sc)
    check_rel("Oc prefix", Oc[:Ls_, :G].cpu().numpy(), ref[0])
    check_rel("On prefix", On[:Ls_, :G].cpu().numpy(), ref[1])
    check_lse("LSEc prefix", LSEc[:G, :Ls_].cpu().numpy(), ref[2])
    check_lse("LSEn prefix", LSEn[:G, :Ls_].cpu().numpy(), ref[3])
    # fixed-reference mode: the same P in both paths, fp32 summation order only
    full = m.bdlm_attn_fwd_shard_refmax(*ins, B, 0, L, True, LSEc_u, LSEn_u, sc)
    rparts = [m.bdlm_attn_fwd_shard_refmax(*ins, B, lo, hi, False, LSEc_u, LSEn_u, sc) for (lo, hi) in bounds]
    rparts.append(m.bdlm_attn_fwd_shard_refmax(*ins, B, 0, 0, True, LSEc_u, LSEn_u, sc))
    rOc, rLc = m.bdlm_lse_merge([p[0] for p in rparts], [p[2] for p in rparts], o_dtype=torch.float32)
    rOn, rLn = m.bdlm_lse_merge([p[1] for p in rparts], [p[3] for p in rparts], o_dtype=torch.float32)
    del rparts
    rdO = max((rOc - full[0]).abs().max().item(), (rOn - full[1]).abs().max().item())
    rdL = max((rLc - full[2]).abs().max().item(), (rLn - full[3]).abs().max().item())
    print(f"B={B}: fixed-reference sharded vs unsharded fp32 max|dO| = {rdO:.3e}, max|dLSE| = {rdL:.3e}")
    assert rdO <= 1e-5 and rdL <= 1e-5
    del full, rOc, rOn, rLc, rLn
    # backward: the 9-partial sharded path against the unsharded backward
    gu = m.bdlm_attn_bwd(*ins, Oc_u.to(torch.bfloat16), On_u.to(torch.bfloat16), X["dOc"], X["dOn"], LSEc_u,
                         LSEn_u, B, sc, g_dtype=torch.float32)
    Dc = m.bdlm_bwd_preprocess(Oc.to(torch.bfloat16), X["dOc"])
    Dn = m.bdlm_bwd_preprocess(On.to(torch.bfloat16), X["dOn"])
    z = lambda H: torch.zeros((L, H, d), dtype=torch.float32, device="cuda")
    gs = [z(Hq), z(Hq), z(Hkv), z(Hkv), z(Hkv), z(Hkv)]  # dQc, dQn, dKc, dVc, dKn, dVn
    for (lo, hi, loc) in [(lo, hi, False) for (lo, hi) in bounds] + [(0, 0, True)]:
        m.bdlm_attn_bwd_shard(*ins, X["dOc"], X["dOn"], LSEc, LSEn, Dc, Dn, B, lo, hi, loc, *gs, sc)
    torch.cuda.synchronize()
    sharded = dict(zip(("dQc", "dQn", "dKc", "dVc", "dKn", "dVn"), gs))
    unsharded = dict(zip(("dQc", "dKc", "dVc", "dQn", "dKn", "dVn"), gu))
    for name in ("dQc", "dKc", "dVc", "dQn", "dKn", "dVn"):
        a, b = sharded[name], unsharded[name]
        err, scale_ = (a - b).abs().max().item(), b.abs().max().item()
        print(f"  {name}: sharded vs unsharded max|err| / max|ref| = {err / scale_:.3e}")
        assert torch.isfinite(a).all() and err <= 2e-2 * scale_, name
    gref = orc.bwd_blockwise(*[Hp[k] for k in NAMES], B, sc)
    check_rel("dQc prefix (sharded)", sharded["dQc"][:Ls_, :G].cpu().numpy(), gref[0])
    check_rel("dQn prefix (sharded)", sharded["dQn"][:Ls_, :G].cpu().numpy(), gref[3])
