"""fp64 CPU oracle for block-diffusion (BDLM) two-stream attention.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
module.  The CUDA library never imports, links or calls it, and this module
imports nothing from the CUDA package: the two sides share no code.

Source pages (all describe one preprint, "Block Parallelism For Efficient
Distributed Long-Context Diffusion Language Model Training", arXiv 2609.19242):

* arxiv.science abstract page, "Abstract": a BDLM pairs autoregressive
  dependencies across blocks with parallel denoising inside a block; the model
  sees a combined clean-plus-corrupted sequence of length 2L.
* evolve.pub review, "Scope & Claims" (Eq. 3, Eq. 6): the objective separates
  over target blocks, so each corrupted block's computation is a unit of work.
* evolve.pub review, FAQ "What is context-sharded block parallelism (CSBP)?":
  corrupted K/V stay with their block, the shared clean context is sharded, and
  only clean K/V and their gradients cross shards.
* evolve.pub review, "Key claims" / FAQ "Does CSBP change training results?"
  (Proposition 1, App. A, Table 3): the sharded computation equals the full
  length-2L computation up to floating-point reduction order.

The two-stream block mask (global order: clean rows 0..L-1, then corrupted rows
0..L-1; blk(i) = floor(i / B)):

* clean row i   -> clean key j      iff blk(j) <= blk(i)   (block-causal)
* clean row     -> corrupted key    never
* corrupted row i -> clean key j    iff blk(j) <  blk(i)   (strict clean prefix)
* corrupted row i -> corrupted key j iff blk(j) == blk(i)  (own block, bidirectional)

Attention per query head h (key/value head floor(h / g), g = Hq / Hkv):
s_ij = scale * q_i . k_j on the mask, LSE_i = ln sum_j exp(s_ij),
p_ij = exp(s_ij - LSE_i), O_i = sum_j p_ij v_j.  Backward with upstream dO and
no gradient through LSE: D_i = dO_i . O_i, dP_ij = dO_i . v_j,
dS_ij = p_ij (dP_ij - D_i), dQ_i = scale sum_j dS_ij k_j,
dK_j = scale sum_{h in group} sum_i dS_ij q_i, dV_j = sum_{h in group} sum_i p_ij dO_i.

Layouts: Q, K, V, O and gradients are token-major ``[L, H, d]`` float64 arrays;
LSE and D are ``[H, L]``.  Inputs are expected to already hold the values the
GPU sees (bf16-representable numbers), upcast to float64.

Every function here is pinned by ``tests/test_oracle.py`` against things other
than itself: hand-typed mask fixtures (one sequence, and a packed batch of
two), closed forms, torch's fp64 scaled-dot-product attention (and its
autograd) in the cases where the mask reduces to textbook attention, central
finite differences, exact gradient invariants and the Proposition-1 sharding
identity.
"""
from __future__ import annotations

import numpy as np

NEG_INF = -np.inf


# --------------------------------------------------------------------------
# the mask
# --------------------------------------------------------------------------
def block_index(i, B):
    """Block of token position i: blocks of B consecutive tokens (abstract page:
    the sequence is split into blocks; denoising runs in parallel inside one)."""
    return np.asarray(i) // B


def mask_2L(L: int, B: int) -> np.ndarray:
    """Explicit 2L x 2L boolean visibility matrix, clean rows/keys first.

    Follows the two-stream BDLM mask described in the module docstring
    (arxiv.science abstract: autoregressive across blocks, parallel within a
    block; CSBP FAQ on the evolve.pub review: corrupted blocks attend to the
    shared clean context plus their own block)."""
    if L % B:
        raise ValueError("L must be a multiple of B")
    bi = block_index(np.arange(L), B)
    row = bi[:, None]
    col = bi[None, :]
    clean_clean = col <= row
    clean_noisy = np.zeros((L, L), dtype=bool)
    noisy_clean = col < row
    noisy_noisy = col == row
    return np.block([[clean_clean, clean_noisy], [noisy_clean, noisy_noisy]])


def visible_ranges(stream: str, b: int, L: int, B: int, kv_begin: int = 0,
                   kv_end: int | None = None, include_local: bool = True):
    """Key ranges seen by the rows of block b of one stream.

    Returns a list of (key_stream, start, end) half-open ranges.  Clean rows
    of block b see clean keys [0, (b+1)B); corrupted rows of block b see clean
    keys [0, bB) and corrupted keys [bB, (b+1)B) (the mask in the module
    docstring).  ``kv_begin``/``kv_end`` restrict the clean keys to one
    contiguous clean shard and ``include_local`` keeps or drops the corrupted
    own-block keys: this is the per-shard view of CSBP (evolve.pub FAQ on CSBP:
    the clean context is sharded, corrupted K/V stay local)."""
    if kv_end is None:
        kv_end = L
    out = []
    clean_hi = (b + 1) * B if stream == "c" else b * B
    lo, hi = max(0, kv_begin), min(clean_hi, kv_end)
    if hi > lo:
        out.append(("c", lo, hi))
    if stream == "n" and include_local:
        out.append(("n", b * B, (b + 1) * B))
    return out


# --------------------------------------------------------------------------
# (i) brute force: explicit mask, dense 2L x 2L
# --------------------------------------------------------------------------
def _group(Hq, Hkv):
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    return Hq // Hkv


def mask_packed(seq_lens, B: int) -> np.ndarray:
    """Explicit 2T x 2T visibility matrix of a packed batch: sequences of the
    given lengths stored back to back (T = sum of the lengths), clean rows/keys
    of all sequences first.  A row sees a key only inside its own sequence,
    and there the two-stream mask of ``mask_2L`` holds with block indices
    counted from the sequence's first token.  (Reading: the pages fix no batch
    layout; sequences of a batch are independent problems.)"""
    lens = [int(n) for n in seq_lens]
    if any(n <= 0 or n % B for n in lens):
        raise ValueError("every sequence length must be a positive multiple of B")
    seq = np.concatenate([np.full(n, s) for s, n in enumerate(lens)])
    pos = np.concatenate([np.arange(n) for n in lens])
    bi = block_index(pos, B)
    same = seq[:, None] == seq[None, :]
    row, col = bi[:, None], bi[None, :]
    T = len(pos)
    return np.block([[same & (col <= row), np.zeros((T, T), dtype=bool)],
                     [same & (col < row), same & (col == row)]])


def fwd_brute(Qc, Kc, Vc, Qn, Kn, Vn, B, scale, mask=None):
    """Dense masked softmax attention over the combined 2L sequence with the
    explicit mask of ``mask_2L`` (abstract page: the model attends over the
    combined clean-plus-corrupted sequence), or with ``mask`` when given (a
    packed batch: ``mask_packed``).  Tiny shapes only."""
    L, Hq, d = Qc.shape
    Hkv = Kc.shape[1]
    g = _group(Hq, Hkv)
    M = mask_2L(L, B) if mask is None else mask
    O = np.zeros((2 * L, Hq, Vc.shape[2]))
    LSE = np.zeros((Hq, 2 * L))
    for h in range(Hq):
        kh = h // g
        Q = np.concatenate([Qc[:, h], Qn[:, h]])
        K = np.concatenate([Kc[:, kh], Kn[:, kh]])
        V = np.concatenate([Vc[:, kh], Vn[:, kh]])
        S = scale * (Q @ K.T)
        S = np.where(M, S, NEG_INF)
        m = S.max(axis=1, keepdims=True)
        lse = m[:, 0] + np.log(np.exp(S - m).sum(axis=1))
        P = np.exp(S - lse[:, None])
        O[:, h] = P @ V
        LSE[h] = lse
    return O[:L], O[L:], LSE[:, :L], LSE[:, L:]


def bwd_brute(Qc, Kc, Vc, Qn, Kn, Vn, dOc, dOn, B, scale, mask=None):
    """Backward of ``fwd_brute`` with the explicit mask (``mask`` when given):
    the softmax-attention gradient formulas of the module docstring, dense.
    Returns (dQc, dKc, dVc, dQn, dKn, dVn)."""
    L, Hq, d = Qc.shape
    Hkv = Kc.shape[1]
    g = _group(Hq, Hkv)
    M = mask_2L(L, B) if mask is None else mask
    dQ = np.zeros((2 * L, Hq, d))
    dK = np.zeros((2 * L, Hkv, d))
    dV = np.zeros((2 * L, Hkv, Vc.shape[2]))
    for h in range(Hq):
        kh = h // g
        Q = np.concatenate([Qc[:, h], Qn[:, h]])
        K = np.concatenate([Kc[:, kh], Kn[:, kh]])
        V = np.concatenate([Vc[:, kh], Vn[:, kh]])
        dO = np.concatenate([dOc[:, h], dOn[:, h]])
        S = np.where(M, scale * (Q @ K.T), NEG_INF)
        m = S.max(axis=1, keepdims=True)
        lse = m[:, 0] + np.log(np.exp(S - m).sum(axis=1))
        P = np.exp(S - lse[:, None])
        O = P @ V
        D = (dO * O).sum(axis=1)
        dP = dO @ V.T
        dS = P * (dP - D[:, None])
        dQ[:, h] = scale * (dS @ K)
        dK[:, kh] += scale * (dS.T @ Q)
        dV[:, kh] += P.T @ dO
    return dQ[:L], dK[:L], dV[:L], dQ[L:], dK[L:], dV[L:]


# --------------------------------------------------------------------------
# (ii) blockwise: per (stream, block, head), visible keys gathered as ranges
# --------------------------------------------------------------------------
def _gather(ranges, Kc_h, Kn_h):
    parts = [(Kc_h if s == "c" else Kn_h)[lo:hi] for (s, lo, hi) in ranges]
    if not parts:
        return np.zeros((0, Kc_h.shape[1]))
    return np.concatenate(parts)


def _softmax_rows(S):
    """Row-wise natural-log LSE and probabilities; a row with no key gets
    LSE = -inf and probabilities of zero (empty partial convention)."""
    if S.shape[1] == 0:
        return np.full(S.shape[0], NEG_INF), S
    m = S.max(axis=1, keepdims=True)
    lse = m[:, 0] + np.log(np.exp(S - m).sum(axis=1))
    return lse, np.exp(S - lse[:, None])


def fwd_partial(Qc, Kc, Vc, Qn, Kn, Vn, B, scale, kv_begin=0, kv_end=None,
                include_local=True, heads=None, blocks=None):
    """Attention of both streams restricted to clean keys [kv_begin, kv_end)
    and (optionally) the corrupted own block.  Each (stream, block, head) is
    computed independently, the per-target-block separation of the evolve.pub
    review, "Scope & Claims" (Eq. 3, Eq. 6).  With the defaults this is the
    full two-stream forward.

    Rows with no visible key get O = 0 and LSE = -inf.  ``heads`` and
    ``blocks`` restrict the work to a subset (rows outside stay zero / -inf).
    Returns (Oc, On, LSEc, LSEn)."""
    L, Hq, d = Qc.shape
    Hkv = Kc.shape[1]
    g = _group(Hq, Hkv)
    N = L // B
    if L % B:
        raise ValueError("L must be a multiple of B")
    heads = range(Hq) if heads is None else heads
    blocks = range(N) if blocks is None else blocks
    dv = Vc.shape[2]
    Oc = np.zeros((L, Hq, dv)); On = np.zeros((L, Hq, dv))
    LSEc = np.full((Hq, L), NEG_INF); LSEn = np.full((Hq, L), NEG_INF)
    for h in heads:
        kh = h // g
        for stream, Q, O, LSE in (("c", Qc, Oc, LSEc), ("n", Qn, On, LSEn)):
            for b in blocks:
                r = slice(b * B, (b + 1) * B)
                rg = visible_ranges(stream, b, L, B, kv_begin, kv_end, include_local)
                K = _gather(rg, Kc[:, kh], Kn[:, kh])
                V = _gather(rg, Vc[:, kh], Vn[:, kh])
                S = scale * (Q[r, h] @ K.T)
                lse, P = _softmax_rows(S)
                O[r, h] = P @ V if K.shape[0] else 0.0
                LSE[h, r] = lse
    return Oc, On, LSEc, LSEn


def fwd_blockwise(Qc, Kc, Vc, Qn, Kn, Vn, B, scale, heads=None, blocks=None):
    """Full two-stream forward computed block by block (see ``fwd_partial``)."""
    return fwd_partial(Qc, Kc, Vc, Qn, Kn, Vn, B, scale, heads=heads, blocks=blocks)


def lse_merge(O_parts, LSE_parts):
    """Exact combination of softmax attention over disjoint key sets.

    With M = max_p LSE_p: LSE = M + ln sum_p exp(LSE_p - M) and
    O = sum_p exp(LSE_p - LSE) O_p; parts with LSE_p = -inf contribute
    nothing, and a row whose parts are all -inf gets O = 0, LSE = -inf.
    This is how CSBP's per-shard partials reproduce the full computation
    (evolve.pub FAQ "Does CSBP change training results": equal up to
    floating-point reduction order; Proposition 1).

    O_parts: list of arrays [rows, H, d]; LSE_parts: list of arrays [H, rows].
    Returns (O, LSE)."""
    Ls = np.stack(LSE_parts)                      # [P, H, rows]
    M = Ls.max(axis=0)                            # [H, rows]
    finite = np.isfinite(M)
    Msafe = np.where(finite, M, 0.0)
    w = np.where(np.isfinite(Ls), np.exp(Ls - Msafe[None]), 0.0)
    tot = w.sum(axis=0)
    LSE = np.where(finite, Msafe + np.log(np.where(finite, tot, 1.0)), NEG_INF)
    O = np.zeros_like(O_parts[0], dtype=np.float64)
    for p, Op in enumerate(O_parts):
        coef = np.where(finite & np.isfinite(Ls[p]), np.exp(Ls[p] - np.where(finite, LSE, 0.0)), 0.0)
        O += coef.T[:, :, None] * Op
    return O, LSE


def shard_bounds(L: int, P: int):
    """P contiguous, equal clean shards [sL/P, (s+1)L/P) (the clean context is
    split across ranks as in conventional context parallelism: evolve.pub
    review "Scope & Claims", Sec. 4 / Fig. 3)."""
    if L % P:
        raise ValueError("L must be a multiple of P")
    return [(s * L // P, (s + 1) * L // P) for s in range(P)]


def fwd_sharded(Qc, Kc, Vc, Qn, Kn, Vn, B, scale, P):
    """CSBP on one machine: P partials against the clean shards, one local
    partial for the corrupted own block, combined by ``lse_merge``.
    Returns (Oc, On, LSEc, LSEn) and the list of partials."""
    L = Qc.shape[0]
    parts = [fwd_partial(Qc, Kc, Vc, Qn, Kn, Vn, B, scale, lo, hi, False)
             for (lo, hi) in shard_bounds(L, P)]
    parts.append(fwd_partial(Qc, Kc, Vc, Qn, Kn, Vn, B, scale, 0, 0, True))
    Oc, LSEc = lse_merge([p[0] for p in parts], [p[2] for p in parts])
    On, LSEn = lse_merge([p[1] for p in parts], [p[3] for p in parts])
    return (Oc, On, LSEc, LSEn), parts


def bwd_partial(Qc, Kc, Vc, Qn, Kn, Vn, dOc, dOn, LSEc, LSEn, Dc, Dn, B, scale,
                kv_begin=0, kv_end=None, include_local=True, heads=None, blocks=None):
    """Gradient contributions of the keys in one partial (clean keys
    [kv_begin, kv_end) plus, optionally, the corrupted own block), given the
    full-row LSE and D = rowsum(dO * O).  With the full-row statistics the
    contributions of disjoint key sets are independent and add up to the
    unsharded gradient (evolve.pub FAQ on CSBP: only clean K/V gradients cross
    shards; Proposition 1).  Returns (dQc, dKc, dVc, dQn, dKn, dVn)."""
    L, Hq, d = Qc.shape
    Hkv = Kc.shape[1]
    g = _group(Hq, Hkv)
    N = L // B
    heads = range(Hq) if heads is None else heads
    blocks = range(N) if blocks is None else blocks
    dQc = np.zeros_like(Qc, dtype=np.float64); dQn = np.zeros_like(Qn, dtype=np.float64)
    dKc = np.zeros_like(Kc, dtype=np.float64); dKn = np.zeros_like(Kn, dtype=np.float64)
    dVc = np.zeros_like(Vc, dtype=np.float64); dVn = np.zeros_like(Vn, dtype=np.float64)
    dK = {"c": dKc, "n": dKn}
    dV = {"c": dVc, "n": dVn}
    for h in heads:
        kh = h // g
        for stream, Q, dO, LSE, D, dQ in (("c", Qc, dOc, LSEc, Dc, dQc),
                                          ("n", Qn, dOn, LSEn, Dn, dQn)):
            for b in blocks:
                r = slice(b * B, (b + 1) * B)
                rg = visible_ranges(stream, b, L, B, kv_begin, kv_end, include_local)
                if not rg:
                    continue
                K = _gather(rg, Kc[:, kh], Kn[:, kh])
                V = _gather(rg, Vc[:, kh], Vn[:, kh])
                S = scale * (Q[r, h] @ K.T)
                Pm = np.exp(S - LSE[h, r][:, None])
                dP = dO[r, h] @ V.T
                dS = Pm * (dP - D[h, r][:, None])
                dQ[r, h] += scale * (dS @ K)
                gK = scale * (dS.T @ Q[r, h])
                gV = Pm.T @ dO[r, h]
                off = 0
                for (s, lo, hi) in rg:
                    n = hi - lo
                    dK[s][lo:hi, kh] += gK[off:off + n]
                    dV[s][lo:hi, kh] += gV[off:off + n]
                    off += n
    return dQc, dKc, dVc, dQn, dKn, dVn


def bwd_preprocess(O, dO):
    """D_i = sum over the head dimension of dO_i * O_i, laid out [H, rows]
    (the softmax-attention backward's row statistic; the gradients the
    evolve.pub review's Proposition 1 covers need it)."""
    return np.einsum("lhd,lhd->hl", dO, O)


def bwd_blockwise(Qc, Kc, Vc, Qn, Kn, Vn, dOc, dOn, B, scale):
    """Full two-stream backward, block by block: forward for LSE and O, the
    row statistic D, then ``bwd_partial`` over all keys."""
    Oc, On, LSEc, LSEn = fwd_blockwise(Qc, Kc, Vc, Qn, Kn, Vn, B, scale)
    Dc, Dn = bwd_preprocess(Oc, dOc), bwd_preprocess(On, dOn)
    return bwd_partial(Qc, Kc, Vc, Qn, Kn, Vn, dOc, dOn, LSEc, LSEn, Dc, Dn, B, scale)


def bwd_sharded(Qc, Kc, Vc, Qn, Kn, Vn, dOc, dOn, B, scale, P):
    """CSBP backward on one machine: merged forward statistics, then one
    gradient contribution per clean shard and one for the local corrupted
    block; dK/dV of disjoint key sets are written, dQ is summed over the
    partials in fixed order (shards 0..P-1, then the local partial)."""
    (Oc, On, LSEc, LSEn), _ = fwd_sharded(Qc, Kc, Vc, Qn, Kn, Vn, B, scale, P)
    Dc, Dn = bwd_preprocess(Oc, dOc), bwd_preprocess(On, dOn)
    L = Qc.shape[0]
    acc = None
    specs = [(lo, hi, False) for (lo, hi) in shard_bounds(L, P)] + [(0, 0, True)]
    for (lo, hi, loc) in specs:
        g = bwd_partial(Qc, Kc, Vc, Qn, Kn, Vn, dOc, dOn, LSEc, LSEn, Dc, Dn, B,
                        scale, lo, hi, loc)
        acc = list(g) if acc is None else [a + x for a, x in zip(acc, g)]
    return tuple(acc)


# --------------------------------------------------------------------------
# row- and key-sampled forms for sizes where the blockwise oracle is too slow
# --------------------------------------------------------------------------
def fwd_rows(Qc, Kc, Vc, Qn, Kn, Vn, B, scale, stream, h, rows):
    """O and LSE of selected rows of one stream and head, each computed from
    its own visible key set (same definition as ``fwd_partial``)."""
    L, Hq, d = Qc.shape
    g = _group(Hq, Kc.shape[1])
    kh = h // g
    Q = Qc if stream == "c" else Qn
    O = np.zeros((len(rows), Vc.shape[2]))
    LSE = np.zeros(len(rows))
    for k, i in enumerate(rows):
        rg = visible_ranges(stream, int(i) // B, L, B)
        K = _gather(rg, Kc[:, kh], Kn[:, kh])
        V = _gather(rg, Vc[:, kh], Vn[:, kh])
        s = scale * (K @ Q[i, h])
        m = s.max()
        lse = m + np.log(np.exp(s - m).sum())
        O[k] = np.exp(s - lse) @ V
        LSE[k] = lse
    return O, LSE


def dq_rows(Qc, Kc, Vc, Qn, Kn, Vn, dOc, dOn, B, scale, stream, h, rows):
    """dQ of selected rows of one stream and head.  A row's dQ needs only its
    own forward statistics: D_i from its O_i, then dS over its visible keys."""
    L, Hq, d = Qc.shape
    g = _group(Hq, Kc.shape[1])
    kh = h // g
    Q = Qc if stream == "c" else Qn
    dO = dOc if stream == "c" else dOn
    O, LSE = fwd_rows(Qc, Kc, Vc, Qn, Kn, Vn, B, scale, stream, h, rows)
    out = np.zeros((len(rows), d))
    for k, i in enumerate(rows):
        rg = visible_ranges(stream, int(i) // B, L, B)
        K = _gather(rg, Kc[:, kh], Kn[:, kh])
        V = _gather(rg, Vc[:, kh], Vn[:, kh])
        p = np.exp(scale * (K @ Q[i, h]) - LSE[k])
        Di = dO[i, h] @ O[k]
        dS = p * (V @ dO[i, h] - Di)
        out[k] = scale * (dS @ K)
    return out


def dkv_tail_blocks(Qc, Kc, Vc, Qn, Kn, Vn, dOc, dOn, B, scale, kv_head, blocks_c, blocks_n):
    """dK and dV of one key/value head, restricted to the clean key blocks
    ``blocks_c`` and corrupted key blocks ``blocks_n``.

    A clean key of block j is read by clean rows of blocks >= j and corrupted
    rows of blocks > j; a corrupted key of block j only by the corrupted rows
    of block j (the mask in the module docstring).  Keys near the end of the
    sequence are read by few rows, so their exact gradients stay cheap at any
    L.  Returns dicts {block: (dK [B, d], dV [B, d])} for each stream."""
    L, Hq, d = Qc.shape
    Hkv = Kc.shape[1]
    g = _group(Hq, Hkv)
    N = L // B
    heads = range(kv_head * g, (kv_head + 1) * g)
    need_c = set()
    need_n = set()
    for j in blocks_c:
        need_c.update(range(j, N)); need_n.update(range(j + 1, N))
    for j in blocks_n:
        need_n.add(j)
    outc = {j: (np.zeros((B, d)), np.zeros((B, Vc.shape[2]))) for j in blocks_c}
    outn = {j: (np.zeros((B, d)), np.zeros((B, Vc.shape[2]))) for j in blocks_n}
    for h in heads:
        for stream, need, Q, dO in (("c", need_c, Qc, dOc), ("n", need_n, Qn, dOn)):
            for b in sorted(need):
                r = slice(b * B, (b + 1) * B)
                rg = visible_ranges(stream, b, L, B)
                K = _gather(rg, Kc[:, kv_head], Kn[:, kv_head])
                V = _gather(rg, Vc[:, kv_head], Vn[:, kv_head])
                S = scale * (Q[r, h] @ K.T)
                lse, Pm = _softmax_rows(S)
                O = Pm @ V
                D = (dO[r, h] * O).sum(axis=1)
                dS = Pm * (dO[r, h] @ V.T - D[:, None])
                gK = scale * (dS.T @ Q[r, h])
                gV = Pm.T @ dO[r, h]
                off = 0
                for (s, lo, hi) in rg:
                    for j in range(lo // B, hi // B):
                        tgt = (outc if s == "c" else outn).get(j)
                        if tgt is not None:
                            a = off + (j * B - lo)
                            tgt[0][:] += gK[a:a + B]
                            tgt[1][:] += gV[a:a + B]
                    off += hi - lo
    return outc, outn


# --------------------------------------------------------------------------
# work accounting used by the measurements
# --------------------------------------------------------------------------
def visible_pairs(L: int, B: int) -> int:
    """Visible (query, key) pairs per query head over both streams:
    sum_b B (b+1) B + sum_b B (bB + B) = L (L + B)."""
    return L * (L + B)
