"""Context-sharded block parallelism (CSBP) across ranks: the partition, the
exchange plan and the per-rank driver.

The scheme ("Block Parallelism For Efficient Distributed Long-Context
Diffusion Language Model Training": evolve.pub review, FAQ "What is
context-sharded block parallelism (CSBP)?", Sec. 4 / Fig. 3; load balancing,
App. I / Table 5 per the review's Strengths):

* R ranks.  The clean sequence is split into R contiguous shards of whole
  blocks; rank r owns clean shard r: its clean query rows and its clean keys
  and values.
* Every corrupted block is owned whole by one rank (block parallelism): its
  queries, keys, values and their gradients never leave that rank.  The
  work of a block of either stream grows with its index (block j has B rows
  that each read (j + 1) B keys), so rank r, whose clean shard is the r-th
  slice of blocks, takes the mirror slice of corrupted blocks, the
  (R - 1 - r)-th: every rank then carries the same work,
  B^2 ((R - 1) n^2 + n (n + 1)) for n = L / (B R) blocks per slice (the
  load balancing of App. I), and both of its row sets are contiguous.
* Forward on rank r: for every clean shard s in order 0..R-1 a partial
  (O_s, LSE_s) of the rank's rows against shard s's keys, then the local
  partial (corrupted rows against their own block), merged exactly by
  log-sum-exp in that fixed order.  Only clean K/V cross ranks: here they are
  all-gathered once; a ring that holds two shards at a time is the same
  plan with less memory.
* Backward on rank r, with the merged LSE and D = rowsum(dO * O) of its own
  rows: per clean shard s, dQ of its rows (summed over s in order) and the
  contribution of its rows to shard s's clean dK / dV; the clean
  contributions are summed over ranks onto the shard's owner
  (reduce-scatter; an all-reduce where the backend has none); the local
  partial gives dQ and the corrupted dK / dV of the rank's own blocks, which
  stay local.

This module holds the plan, the exchange and the order of the steps.  The
arithmetic comes from a ``compute`` object and the transport from a ``comm``
object passed in by the caller:

* ``compute.fwd(rows, kv, kv_data, local)``: partial forward of the rank's
  rows ``rows`` (a ``Rows``) against the clean keys ``kv`` = (begin, end),
  whose K and V are ``kv_data``, and, if ``local``, the rows' own corrupted
  blocks; returns (Oc, On, LSEc, LSEn) of those rows, rows with no key
  giving O = 0, LSE = -inf.
* ``compute.merge(parts)``: exact LSE merge of such partials, in order.
* ``compute.preprocess(O, dO)``: D of the rows.
* ``compute.bwd(rows, kv, kv_data, local, stats)``: gradient contributions
  of those keys from the rows, given the merged statistics; returns
  (dQc, dQn, dK_clean, dV_clean, dK_noisy, dV_noisy), the clean key
  gradients over ``kv`` and the corrupted ones over the rows' own blocks.
* ``comm``: ``rank``, ``world``, ``all_gather(x) -> list`` and
  ``sum_to_owner(x, owner) -> x or None`` (the sum over ranks, on the owner).

On GB300s the compute object is the library's tensor-core kernels
restricted to a rank's rows (`bdlm_attn_fwd_shard_rows`,
`bdlm_attn_bwd_shard_rows`: row ranges per stream, gradients accumulated
over calls) and the transport is NCCL over NVLink (no TMA multicast, and no
kernel reads a peer's memory: shards are copied into local HBM first).  The
row-restricted kernels are checked on one GPU with every rank's calls made
in turn (tests/test_gpu_csbp_rows.py); the plan and this driver are checked
with gloo ranks on the CPU and the fp64 oracle as the compute object
(tests/test_csbp_ranks.py).  The kernels index full-length tensors, so a
rank would hold its rows in full-length buffers; the multi-GPU path is
unmeasured on hardware.
"""
from __future__ import annotations

from dataclasses import dataclass, field


@dataclass(frozen=True)
class Rows:
    """The query rows a rank owns: clean rows of blocks [c0, c1) and
    corrupted rows of blocks [n0, n1)."""
    c0: int
    c1: int
    n0: int
    n1: int

    @property
    def noisy_blocks(self):
        return tuple(range(self.n0, self.n1))


@dataclass
class CSBPPlan:
    """Ownership of a length-L, block-size-B problem on R ranks."""
    L: int
    B: int
    R: int
    clean_shards: list = field(default_factory=list)  # per rank: (first block, end block)
    noisy_owner: list = field(default_factory=list)   # per corrupted block: its rank
    load: list = field(default_factory=list)          # per rank: rows x keys of its work, both streams

    @staticmethod
    def build(L: int, B: int, R: int) -> "CSBPPlan":
        if L <= 0 or B <= 0 or R <= 0 or L % B:
            raise ValueError("need L, B, R > 0 and L a multiple of B")
        N = L // B
        if N % R:
            raise ValueError("the clean shards hold whole blocks: (L / B) must be a multiple of R")
        per = N // R
        plan = CSBPPlan(L, B, R)
        plan.clean_shards = [(r * per, (r + 1) * per) for r in range(R)]
        # corrupted blocks: the mirror slice of the rank's clean shard
        plan.noisy_owner = [R - 1 - j // per for j in range(N)]
        # work of block j of either stream: B rows reading (j + 1) B keys
        cost = [B * (j + 1) * B for j in range(N)]
        plan.load = [sum(cost[j] for j in range(a, b)) for (a, b) in plan.clean_shards]
        for j, r in enumerate(plan.noisy_owner):
            plan.load[r] += cost[j]
        return plan

    def rows(self, r: int) -> Rows:
        c0, c1 = self.clean_shards[r]
        n0, n1 = self.clean_shards[self.R - 1 - r]
        return Rows(c0, c1, n0, n1)

    def shard_keys(self, s: int):
        """Clean key range (token indices) of shard s."""
        a, b = self.clean_shards[s]
        return a * self.B, b * self.B

    def imbalance(self) -> float:
        """Largest rank load over the mean."""
        return max(self.load) / (sum(self.load) / self.R)


def gather_clean_kv(comm, Kc_local, Vc_local):
    """Every rank's clean K / V shard, in rank order: the one exchange of the
    forward (an all-gather; a ring would hold two shards at a time)."""
    return list(zip(comm.all_gather(Kc_local), comm.all_gather(Vc_local)))


def forward(plan: CSBPPlan, comm, compute, shards):
    """Forward of the rank's rows: partials against every clean shard in
    order (``shards`` from ``gather_clean_kv``), then the local partial,
    merged.  Returns the rank's (Oc, On, LSEc, LSEn) rows."""
    rows = plan.rows(comm.rank)
    parts = [compute.fwd(rows, plan.shard_keys(s), shards[s], False) for s in range(plan.R)]
    parts.append(compute.fwd(rows, (0, 0), None, True))
    return compute.merge(parts)


def backward(plan: CSBPPlan, comm, compute, shards, out, dO):
    """Backward of the rank's rows given its merged forward outputs
    ``out`` = (Oc, On, LSEc, LSEn) and upstream ``dO`` = (dOc, dOn) of its
    rows.  Returns (dQc, dQn) of its rows, the clean (dK, dV) of its own
    shard (summed over every rank's rows) and the corrupted (dK, dV) of its
    own blocks."""
    rows = plan.rows(comm.rank)
    Oc, On, LSEc, LSEn = out
    stats = (LSEc, LSEn, compute.preprocess(Oc, dO[0]), compute.preprocess(On, dO[1]))
    dQc = dQn = None
    mine = None
    for s in range(plan.R):
        gq_c, gq_n, gk, gv, _, _ = compute.bwd(rows, plan.shard_keys(s), shards[s], False, stats)
        dQc = gq_c if dQc is None else dQc + gq_c
        dQn = gq_n if dQn is None else dQn + gq_n
        k = comm.sum_to_owner(gk, s)
        v = comm.sum_to_owner(gv, s)
        if s == comm.rank:
            mine = (k, v)
    gq_c, gq_n, _, _, gkn, gvn = compute.bwd(rows, (0, 0), None, True, stats)
    return (dQc + gq_c, dQn + gq_n), mine, (gkn, gvn)
