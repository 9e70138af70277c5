"""Pins for the fp64 oracle, against things other than the oracle itself.

Each pin is chosen so that a plausible mistake in the oracle (a wrong block
comparison, a dropped mask term, a wrong scale or sign, a transposed operand, a
missing GQA reduction) fails at least one of them; ``test_planted_mistakes``
plants such mistakes and checks that.
"""
from __future__ import annotations

import os

import numpy as np
import pytest
import torch

import oracle.bdlm_oracle as orc
from structured_mask_attention_gb300.inputs import bf16_round, make_numpy

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(L, Hq, Hkv, d, seed=1, dv=None):
    rng = np.random.default_rng(seed)
    dv = d if dv is None else dv
    f = lambda *s: rng.standard_normal(s)
    return (f(L, Hq, d), f(L, Hkv, d), f(L, Hkv, dv), f(L, Hq, d), f(L, Hkv, d), f(L, Hkv, dv),
            f(L, Hq, dv), f(L, Hq, dv))


def _load_mask(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as fh:
        for line in fh:
            if line.startswith("#") or not line.strip():
                continue
            rows.append([c == "1" for c in line.strip() if c in "01"])
    return np.array(rows, dtype=bool)


# --------------------------------------------------------------------------- mask
def test_mask_matches_hand_typed_fixture():
    assert (orc.mask_2L(6, 2) == _load_mask("mask_L6_B2.txt")).all()


@pytest.mark.parametrize("L,B", [(8, 1), (8, 2), (16, 4), (64, 8), (64, 64), (96, 32)])
def test_visible_ranges_cover_mask(L, B):
    M = orc.mask_2L(L, B)
    for stream, off in (("c", 0), ("n", L)):
        for i in range(L):
            vis = np.zeros(2 * L, dtype=bool)
            for (s, lo, hi) in orc.visible_ranges(stream, i // B, L, B):
                base = 0 if s == "c" else L
                vis[base + lo:base + hi] = True
            assert (vis == M[off + i]).all()


@pytest.mark.parametrize("L,B", [(8, 1), (16, 4), (64, 8), (256, 32), (512, 512)])
def test_visible_pairs_closed_form(L, B):
    # sum_b B(b+1)B + sum_b B(bB + B) = L(L+B), half of the dense count near B << L
    assert orc.mask_2L(L, B).sum() == orc.visible_pairs(L, B) == L * (L + B)


# --------------------------------------------------------------- brute vs blockwise
@pytest.mark.parametrize("L,B,Hq,Hkv", [(8, 1, 1, 1), (8, 2, 2, 1), (16, 4, 5, 1),
                                        (64, 8, 4, 2), (64, 64, 2, 2), (48, 16, 10, 2)])
def test_blockwise_equals_brute(L, B, Hq, Hkv):
    d = 8
    Qc, Kc, Vc, Qn, Kn, Vn, dOc, dOn = _rand(L, Hq, Hkv, d, seed=L + B)
    sc = 0.3
    a = orc.fwd_brute(Qc, Kc, Vc, Qn, Kn, Vn, B, sc)
    b = orc.fwd_blockwise(Qc, Kc, Vc, Qn, Kn, Vn, B, sc)
    for x, y in zip(a, b):
        np.testing.assert_allclose(x, y, rtol=0, atol=1e-12)
    ga = orc.bwd_brute(Qc, Kc, Vc, Qn, Kn, Vn, dOc, dOn, B, sc)
    gb = orc.bwd_blockwise(Qc, Kc, Vc, Qn, Kn, Vn, dOc, dOn, B, sc)
    for x, y in zip(ga, gb):
        np.testing.assert_allclose(x, y, rtol=0, atol=1e-12)


# ------------------------------------------------------------------ packed batches
def test_packed_mask_matches_hand_typed_fixture():
    assert (orc.mask_packed((4, 2), 2) == _load_mask("mask_packed_4_2_B2.txt")).all()


@pytest.mark.parametrize("lens,B", [((8,), 2), ((16, 8, 24), 4), ((6, 6, 6), 3), ((32, 4), 4)])
def test_packed_mask_pairs_and_single_sequence(lens, B):
    M = orc.mask_packed(lens, B)
    assert M.sum() == sum(n * (n + B) for n in lens)
    if len(lens) == 1:
        assert (M == orc.mask_2L(lens[0], B)).all()


@pytest.mark.parametrize("lens,B,Hq,Hkv", [((16, 8, 24), 4, 4, 2), ((6, 12), 3, 3, 1), ((8, 8, 8, 8), 8, 2, 2)])
def test_packed_brute_equals_per_sequence(lens, B, Hq, Hkv):
    """The packed definition (one mask over the whole batch) equals each
    sequence computed alone: the decomposition the packed GPU tests use."""
    T, d = sum(lens), 8
    Qc, Kc, Vc, Qn, Kn, Vn, dOc, dOn = _rand(T, Hq, Hkv, d, seed=T + B)
    sc = 0.35
    M = orc.mask_packed(lens, B)
    fwd = orc.fwd_brute(Qc, Kc, Vc, Qn, Kn, Vn, B, sc, mask=M)
    bwd = orc.bwd_brute(Qc, Kc, Vc, Qn, Kn, Vn, dOc, dOn, B, sc, mask=M)
    off = np.concatenate([[0], np.cumsum(lens)])
    for s in range(len(lens)):
        a, b = off[s], off[s + 1]
        x = [t[a:b] for t in (Qc, Kc, Vc, Qn, Kn, Vn, dOc, dOn)]
        rf = orc.fwd_blockwise(*x[:6], B, sc)
        rb = orc.bwd_blockwise(*x, B, sc)
        for got, ref in zip((fwd[0][a:b], fwd[1][a:b], fwd[2][:, a:b], fwd[3][:, a:b]), rf):
            np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)
        for got, ref in zip(bwd, rb):
            np.testing.assert_allclose(got[a:b], ref, rtol=0, atol=1e-12)


# ------------------------------------------------------------------ closed forms
def test_zero_keys_uniform_softmax():
    """K = 0 makes every visible score 0: LSE_i = ln(#visible_i) with
    #visible = (blk+1)B in both streams, and O_i is the mean of visible V."""
    L, B, H, d = 24, 4, 2, 6
    Qc, Kc, Vc, Qn, Kn, Vn, _, _ = _rand(L, H, H, d, seed=3)
    Kc[:] = 0; Kn[:] = 0
    Oc, On, LSEc, LSEn = orc.fwd_blockwise(Qc, Kc, Vc, Qn, Kn, Vn, B, 0.7)
    cnt = (np.arange(L) // B + 1) * B
    np.testing.assert_allclose(LSEc, np.log(cnt)[None].repeat(H, 0), atol=1e-13)
    np.testing.assert_allclose(LSEn, np.log(cnt)[None].repeat(H, 0), atol=1e-13)
    for i in range(L):
        b = i // B
        np.testing.assert_allclose(Oc[i], Vc[:(b + 1) * B].mean(0), atol=1e-13)
        np.testing.assert_allclose(On[i], np.concatenate([Vc[:b * B], Vn[b * B:(b + 1) * B]]).mean(0), atol=1e-13)


def test_onehot_values_reveal_hand_typed_mask():
    """K = 0 and V = one-hot of the key's global index: O_i * #visible_i is
    exactly row i of the hand-typed mask."""
    L, B = 6, 2
    M = _load_mask("mask_L6_B2.txt")
    eye = np.eye(2 * L)
    Vc = eye[:L][:, None, :]; Vn = eye[L:][:, None, :]
    Z = np.zeros((L, 1, 4))
    Qc = np.random.default_rng(0).standard_normal((L, 1, 4)); Qn = Qc.copy()
    for fn in (orc.fwd_blockwise, orc.fwd_brute):
        Oc, On, _, _ = fn(Qc, Z, Vc, Qn, Z, Vn, B, 1.0)
        O = np.concatenate([Oc[:, 0], On[:, 0]])
        np.testing.assert_allclose(O * M.sum(1, keepdims=True), M.astype(float), atol=1e-13)


# --------------------------------------------------- textbook special cases (torch)
def _sdpa(Q, K, V, causal=False, mask=None):
    """torch's fp64 CPU scaled-dot-product attention on [L, H, d] arrays, KV
    heads expanded by contiguous grouping."""
    g = Q.shape[1] // K.shape[1]
    q = torch.tensor(Q).permute(1, 0, 2)
    k = torch.tensor(K).repeat_interleave(g, dim=1).permute(1, 0, 2)
    v = torch.tensor(V).repeat_interleave(g, dim=1).permute(1, 0, 2)
    return q, k, v


def _sdpa_out(q, k, v, scale, causal=False, mask=None):
    return torch.nn.functional.scaled_dot_product_attention(
        q, k, v, attn_mask=mask, is_causal=causal, scale=scale)


def test_single_block_is_full_attention_per_stream():
    """B = L: clean rows see all clean keys (no mask), corrupted rows see only
    the corrupted stream (no mask)."""
    L, Hq, Hkv, d = 32, 4, 2, 8
    Qc, Kc, Vc, Qn, Kn, Vn, dOc, dOn = _rand(L, Hq, Hkv, d, seed=5)
    sc = 0.2
    Oc, On, LSEc, LSEn = orc.fwd_blockwise(Qc, Kc, Vc, Qn, Kn, Vn, L, sc)
    g = orc.bwd_blockwise(Qc, Kc, Vc, Qn, Kn, Vn, dOc, dOn, L, sc)
    for (Q, K, V, dO, O, dQ, dK, dV) in ((Qc, Kc, Vc, dOc, Oc, g[0], g[1], g[2]),
                                         (Qn, Kn, Vn, dOn, On, g[3], g[4], g[5])):
        q, k, v = _sdpa(Q, K, V)
        K_ = torch.tensor(K, requires_grad=True); V_ = torch.tensor(V, requires_grad=True)
        Q_ = torch.tensor(Q, requires_grad=True)
        gq = Hq // Hkv
        out = _sdpa_out(Q_.permute(1, 0, 2), K_.repeat_interleave(gq, 1).permute(1, 0, 2),
                        V_.repeat_interleave(gq, 1).permute(1, 0, 2), sc)
        np.testing.assert_allclose(O, out.permute(1, 0, 2).detach().numpy(), atol=1e-12)
        (out * torch.tensor(dO).permute(1, 0, 2)).sum().backward()
        np.testing.assert_allclose(dQ, Q_.grad.numpy(), atol=1e-11)
        np.testing.assert_allclose(dK, K_.grad.numpy(), atol=1e-11)
        np.testing.assert_allclose(dV, V_.grad.numpy(), atol=1e-11)
    # LSE: ln sum exp over all keys of the own stream, by torch.logsumexp
    S = torch.einsum("lhd,mhd->hlm", torch.tensor(Qc), torch.tensor(Kc).repeat_interleave(Hq // Hkv, 1)) * sc
    np.testing.assert_allclose(LSEc, torch.logsumexp(S, -1).numpy(), atol=1e-12)


def test_unit_blocks_are_token_causal():
    """B = 1: the clean stream is token-causal attention (torch is_causal);
    corrupted row i reads clean keys 0..i-1 and its own corrupted key."""
    L, Hq, Hkv, d = 24, 2, 1, 8
    Qc, Kc, Vc, Qn, Kn, Vn, dOc, dOn = _rand(L, Hq, Hkv, d, seed=6)
    sc = 0.4
    Oc, On, LSEc, LSEn = orc.fwd_blockwise(Qc, Kc, Vc, Qn, Kn, Vn, 1, sc)
    grads = orc.bwd_blockwise(Qc, Kc, Vc, Qn, Kn, Vn, dOc, dOn, 1, sc)
    # clean stream: causal SDPA + autograd
    Q_ = torch.tensor(Qc, requires_grad=True); K_ = torch.tensor(Kc, requires_grad=True)
    V_ = torch.tensor(Vc, requires_grad=True)
    out = _sdpa_out(Q_.permute(1, 0, 2), K_.repeat_interleave(Hq, 1).permute(1, 0, 2),
                    V_.repeat_interleave(Hq, 1).permute(1, 0, 2), sc, causal=True)
    np.testing.assert_allclose(Oc, out.permute(1, 0, 2).detach().numpy(), atol=1e-12)
    # corrupted stream: keys [clean 0..L-1, corrupted 0..L-1] with a strictly
    # lower-triangular clean part and a diagonal corrupted part
    Kn_ = torch.tensor(Kn, requires_grad=True); Vn_ = torch.tensor(Vn, requires_grad=True)
    Kall = torch.cat([torch.tensor(Kc), Kn_]).repeat_interleave(Hq, 1).permute(1, 0, 2)
    Vall = torch.cat([torch.tensor(Vc), Vn_]).repeat_interleave(Hq, 1).permute(1, 0, 2)
    vis = torch.cat([torch.ones(L, L, dtype=torch.bool).tril(-1), torch.eye(L, dtype=torch.bool)], dim=1)
    Qn_ = torch.tensor(Qn, requires_grad=True)
    outn = _sdpa_out(Qn_.permute(1, 0, 2), Kall, Vall, sc, mask=vis)
    np.testing.assert_allclose(On, outn.permute(1, 0, 2).detach().numpy(), atol=1e-12)
    # dQ of both streams from autograd (dK/dV of the clean keys mix both
    # streams' rows: covered by the B = L case and finite differences)
    (out * torch.tensor(dOc).permute(1, 0, 2)).sum().backward()
    (outn * torch.tensor(dOn).permute(1, 0, 2)).sum().backward()
    np.testing.assert_allclose(grads[0], Q_.grad.numpy(), atol=1e-11)
    np.testing.assert_allclose(grads[3], Qn_.grad.numpy(), atol=1e-11)
    # corrupted keys are read only by corrupted rows, so autograd of the
    # corrupted-stream output alone gives dKn and dVn
    np.testing.assert_allclose(grads[4], Kn_.grad.numpy(), atol=1e-11)
    np.testing.assert_allclose(grads[5], Vn_.grad.numpy(), atol=1e-11)


# --------------------------------------------------------- finite differences
def test_finite_differences():
    """Central differences of f = sum(dO * O) in fp64 at random coordinates of
    all six inputs agree with the analytic gradients."""
    L, B, Hq, Hkv, d = 16, 4, 4, 2, 4
    X = list(_rand(L, Hq, Hkv, d, seed=7))
    dOc, dOn = X[6], X[7]
    sc = 0.5
    grads = orc.bwd_blockwise(*X[:6], dOc, dOn, B, sc)
    # map gradient order (dQc, dKc, dVc, dQn, dKn, dVn) to input index
    gmap = {0: 0, 1: 1, 2: 2, 3: 3, 4: 4, 5: 5}

    def f(inp):
        Oc, On, _, _ = orc.fwd_blockwise(*inp, B, sc)
        return (Oc * dOc).sum() + (On * dOn).sum()

    rng = np.random.default_rng(11)
    eps = 1e-6
    for k in range(6):
        for _ in range(6):
            idx = tuple(rng.integers(0, s) for s in X[k].shape)
            inp = [x.copy() for x in X[:6]]
            inp[k][idx] += eps
            fp = f(inp)
            inp[k][idx] -= 2 * eps
            fm = f(inp)
            fd = (fp - fm) / (2 * eps)
            an = grads[gmap[k]][idx]
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (k, idx, fd, an)


# --------------------------------------------------------- gradient invariants
@pytest.mark.parametrize("L,B,Hq,Hkv", [(32, 4, 4, 2), (40, 8, 6, 3)])
def test_gradient_invariants(L, B, Hq, Hkv):
    """Per key/value head, over all keys of both streams: sum_j dK_j = 0
    (every row of dS sums to 0) and sum_j dV_j = sum over the group's rows of
    dO (every row of P sums to 1)."""
    X = _rand(L, Hq, Hkv, 8, seed=L)
    g = orc.bwd_blockwise(*X, B, 0.35)
    sK = g[1].sum(0) + g[4].sum(0)
    sV = g[2].sum(0) + g[5].sum(0)
    np.testing.assert_allclose(sK, 0.0, atol=1e-12)
    G = Hq // Hkv
    dO = X[6] + X[7]
    want = np.stack([dO[:, h * G:(h + 1) * G].sum((0, 1)) for h in range(Hkv)])
    np.testing.assert_allclose(sV, want, atol=1e-11)


# ------------------------------------------------------------ Proposition 1
@pytest.mark.parametrize("L,B,P", [(32, 4, 4), (32, 8, 8), (48, 16, 3), (64, 32, 8), (32, 32, 2), (24, 2, 6)])
def test_sharded_equals_unsharded(L, B, P):
    """CSBP identity: P clean-shard partials plus the local corrupted partial,
    LSE-merged, give the unsharded outputs and gradients (shards need not
    align to blocks)."""
    X = _rand(L, 4, 2, 8, seed=P)
    sc = 0.3
    ref = orc.fwd_blockwise(*X[:6], B, sc)
    got, parts = orc.fwd_sharded(*X[:6], B, sc, P)
    for x, y in zip(ref, got):
        np.testing.assert_allclose(x, y, atol=1e-12)
    gref = orc.bwd_blockwise(*X, B, sc)
    ggot = orc.bwd_sharded(*X, B, sc, P)
    for x, y in zip(gref, ggot):
        np.testing.assert_allclose(x, y, atol=1e-12)


def test_corrupted_block0_local_only():
    """Corrupted block 0 reads no clean key: its clean-shard partials are
    empty (O = 0, LSE = -inf)."""
    L, B = 16, 4
    X = _rand(L, 2, 2, 4, seed=2)
    Oc, On, LSEc, LSEn = orc.fwd_partial(*X[:6], B, 0.5, 0, L, False)
    assert np.isneginf(LSEn[:, :B]).all() and (On[:B] == 0).all()
    assert np.isfinite(LSEn[:, B:]).all()


# ----------------------------------------------------------------- merge
def _direct_softmax(S, V):
    m = S.max(-1, keepdims=True)
    w = np.exp(S - m)
    return (w @ V) / w.sum(-1, keepdims=True), (m[..., 0] + np.log(w.sum(-1)))


def test_merge_random_splits_equal_direct_softmax():
    rng = np.random.default_rng(4)
    rows, H, n, d = 7, 3, 40, 5
    S = rng.standard_normal((H, rows, n)) * 3
    V = rng.standard_normal((n, d))
    Od = np.stack([_direct_softmax(S[h], V)[0] for h in range(H)], 1)
    Ld = np.stack([_direct_softmax(S[h], V)[1] for h in range(H)])
    cuts = np.sort(rng.choice(np.arange(1, n), 4, replace=False))
    edges = [0, *cuts, n]
    Os, Ls = [], []
    for a, b in zip(edges[:-1], edges[1:]):
        o = np.stack([_direct_softmax(S[h][:, a:b], V[a:b])[0] for h in range(H)], 1)
        l = np.stack([_direct_softmax(S[h][:, a:b], V[a:b])[1] for h in range(H)])
        Os.append(o); Ls.append(l)
    O, L_ = orc.lse_merge(Os, Ls)
    np.testing.assert_allclose(O, Od, atol=1e-13)
    np.testing.assert_allclose(L_, Ld, atol=1e-13)


def test_merge_identity_neutral_and_associative():
    rng = np.random.default_rng(9)
    mk = lambda: (rng.standard_normal((5, 2, 3)), rng.standard_normal((2, 5)))
    a, b, c = mk(), mk(), mk()
    O, L_ = orc.lse_merge([a[0]], [a[1]])
    np.testing.assert_allclose(O, a[0], atol=1e-15); np.testing.assert_allclose(L_, a[1], atol=1e-15)
    empty = (np.zeros_like(a[0]), np.full_like(a[1], -np.inf))
    O, L_ = orc.lse_merge([a[0], empty[0]], [a[1], empty[1]])
    np.testing.assert_allclose(O, a[0], atol=1e-15); np.testing.assert_allclose(L_, a[1], atol=1e-15)
    ab = orc.lse_merge([a[0], b[0]], [a[1], b[1]])
    bc = orc.lse_merge([b[0], c[0]], [b[1], c[1]])
    l = orc.lse_merge([ab[0], c[0]], [ab[1], c[1]])
    r = orc.lse_merge([a[0], bc[0]], [a[1], bc[1]])
    np.testing.assert_allclose(l[0], r[0], atol=1e-13); np.testing.assert_allclose(l[1], r[1], atol=1e-13)
    O, L_ = orc.lse_merge([empty[0], empty[0]], [empty[1], empty[1]])
    assert (O == 0).all() and np.isneginf(L_).all()


# ------------------------------------------------------------ sampled forms
def test_sampled_forms_match_blockwise():
    L, B, Hq, Hkv, d = 64, 8, 4, 2, 8
    X = _rand(L, Hq, Hkv, d, seed=12)
    sc = 0.3
    Oc, On, LSEc, LSEn = orc.fwd_blockwise(*X[:6], B, sc)
    g = orc.bwd_blockwise(*X, B, sc)
    rows = [0, 5, 8, 33, 63]
    for stream, O, LSE, dQ in (("c", Oc, LSEc, g[0]), ("n", On, LSEn, g[3])):
        for h in (0, 3):
            o, l = orc.fwd_rows(*X[:6], B, sc, stream, h, rows)
            np.testing.assert_allclose(o, O[rows, h], atol=1e-12)
            np.testing.assert_allclose(l, LSE[h, rows], atol=1e-12)
            np.testing.assert_allclose(orc.dq_rows(*X, B, sc, stream, h, rows), dQ[rows, h], atol=1e-12)
    outc, outn = orc.dkv_tail_blocks(*X, B, sc, 1, [7, 6, 2], [0, 5])
    for j, (dk, dv) in outc.items():
        np.testing.assert_allclose(dk, g[1][j * B:(j + 1) * B, 1], atol=1e-12)
        np.testing.assert_allclose(dv, g[2][j * B:(j + 1) * B, 1], atol=1e-12)
    for j, (dk, dv) in outn.items():
        np.testing.assert_allclose(dk, g[4][j * B:(j + 1) * B, 1], atol=1e-12)
        np.testing.assert_allclose(dv, g[5][j * B:(j + 1) * B, 1], atol=1e-12)


# ------------------------------------------------------------ input rounding
def test_bf16_round_matches_torch():
    x = np.random.default_rng(0).standard_normal(100000).astype(np.float32) * 10
    x[:4] = [1.00390625, 1.01171875, -2.0078125, 3.0]  # exact ties (even / odd)
    want = torch.tensor(x).to(torch.bfloat16).float().numpy()
    np.testing.assert_array_equal(bf16_round(x), want)


def test_inputs_are_seeded_and_bf16():
    a = make_numpy(32, 2, 1, 8, seed=0, lognormal_sigma=0.5)
    b = make_numpy(32, 2, 1, 8, seed=0, lognormal_sigma=0.5)
    for k in a:
        np.testing.assert_array_equal(a[k], b[k])
        np.testing.assert_array_equal(bf16_round(a[k]), a[k])


# ------------------------------------------------------------ planted mistakes
def test_planted_mistakes_are_caught(monkeypatch):
    """Plant plausible mistakes in the oracle (CPU only) and check that the
    pins above reject each one."""
    good = orc.visible_ranges

    def inclusive_prefix(stream, b, L, B, kv_begin=0, kv_end=None, include_local=True):
        # corrupted rows wrongly read their own clean block
        r = good(stream, b, L, B, kv_begin, kv_end, include_local)
        if stream == "n" and b * B < L:
            r = [(s, lo, hi + B if s == "c" else hi) for (s, lo, hi) in r] or [("c", b * B, (b + 1) * B)] + r
        return r

    def causal_within_block(stream, b, L, B, kv_begin=0, kv_end=None, include_local=True):
        # corrupted rows lose their own block
        return [x for x in good(stream, b, L, B, kv_begin, kv_end, include_local) if x[0] == "c"] or \
            good(stream, b, L, B, kv_begin, kv_end, include_local)

    for bad in (inclusive_prefix, causal_within_block):
        monkeypatch.setattr(orc, "visible_ranges", bad)
        with pytest.raises(AssertionError):
            test_onehot_values_reveal_hand_typed_mask()
        monkeypatch.setattr(orc, "visible_ranges", good)

    # a transposed V gradient (P dO instead of P^T dO) and a dropped scale on dK
    real_partial = orc.bwd_partial

    def no_scale_dk(*a, **k):
        r = list(real_partial(*a, **k))
        sc = a[13]
        r[1] = r[1] / sc; r[4] = r[4] / sc
        return tuple(r)

    monkeypatch.setattr(orc, "bwd_partial", no_scale_dk)
    with pytest.raises(AssertionError):
        test_finite_differences()
    monkeypatch.setattr(orc, "bwd_partial", real_partial)


def _planted(fn, old, new):
    """``fn`` recompiled from its source with one edit (a planted mistake), in
    the oracle module's namespace."""
    import inspect
    import textwrap
    src = textwrap.dedent(inspect.getsource(fn))
    assert old in src, (fn.__name__, old)
    ns = dict(vars(orc))
    exec(compile(src.replace(old, new), f"<planted {fn.__name__}>", "exec"), ns)
    return ns[fn.__name__]


@pytest.mark.parametrize("fn_name,old,new,pin", [
    # gradient arithmetic: a sign error in dS, P in place of dS for dQ, and a
    # dropped GQA reduction for dK (only the group's first head counted)
    ("bwd_partial", "(dP - D[h, r][:, None])", "(dP + D[h, r][:, None])", "test_single_block_is_full_attention_per_stream"),
    ("bwd_partial", "scale * (dS @ K)", "scale * (Pm @ K)", "test_single_block_is_full_attention_per_stream"),
    ("bwd_partial", "+= gK[off:off + n]", "+= gK[off:off + n] * (h % g == 0)", "test_single_block_is_full_attention_per_stream"),
    # masks: corrupted rows reading their own clean block; a packed batch whose
    # rows see the other sequences
    ("mask_2L", "noisy_clean = col < row", "noisy_clean = col <= row", "test_mask_matches_hand_typed_fixture"),
    ("mask_packed", "same = seq[:, None] == seq[None, :]", "same = seq[:, None] >= 0", "test_packed_mask_matches_hand_typed_fixture"),
])
def test_planted_source_mistakes_are_caught(monkeypatch, fn_name, old, new, pin):
    """Plant a mistake in the oracle's source (CPU only) and check that the
    named pin rejects it."""
    monkeypatch.setattr(orc, fn_name, _planted(getattr(orc, fn_name), old, new))
    with pytest.raises(AssertionError):
        globals()[pin]()
