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
  (``policy="contiguous"``, rank r taking the r-th slice as a split by token
  position would, is kept as the unbalanced ablation.)
* Forward on rank r: for every clean shard s in order 0..R-1 a partial
  (O_s, LSE_s) of the rank's rows against shard s's keys, then the local
  partial (corrupted rows against their own block), merged exactly by
  log-sum-exp in that fixed order, each partial folded into a running merge
  as it is computed.  Only clean K/V cross ranks: here they are
  all-gathered once; a ring that holds two shards at a time is the same
  plan with less memory.  Once all shards are gathered the rank may instead
  make one call over the whole clean sequence (``gathered=True``): the same
  result without partials or a merge.
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

On GB300s the compute object is ``KernelCompute``: the library's
tensor-core kernels restricted to a rank's rows, on rank-local tensors
(`bdlm_attn_fwd_rank`, `bdlm_attn_bwd_rank`: row ranges per stream,
gradients accumulated over calls), and the transport is ``TorchComm``, NCCL over NVLink through
torch.distributed (no TMA multicast, and no kernel reads a peer's memory:
shards are copied into local HBM first).  Checked: the plan and this driver
with gloo ranks on the CPU and the fp64 oracle as the compute object
(tests/test_csbp_ranks.py); the driver with ``KernelCompute`` for every rank
on one GPU, the ranks as host threads exchanging through host-side
collectives, and over NCCL through ``TorchComm`` as a one-rank group
(tests/test_gpu_csbp_rows.py).  A rank holds only its own rows
and the clean K / V it receives.  No run on several GPUs exists.
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


POLICIES = ("mirror", "contiguous")


@dataclass
class CSBPPlan:
    """Ownership of a length-L, block-size-B problem on R ranks."""
    L: int
    B: int
    R: int
    policy: str = "mirror"
    clean_shards: list = field(default_factory=list)  # per rank: (first block, end block)
    noisy_owner: list = field(default_factory=list)   # per corrupted block: its rank
    load: list = field(default_factory=list)          # per rank: rows x keys of its work, both streams

    @staticmethod
    def build(L: int, B: int, R: int, policy: str = "mirror") -> "CSBPPlan":
        """``policy``: "mirror" (rank r takes the (R - 1 - r)-th slice of
        corrupted blocks: every rank carries the same work) or "contiguous"
        (rank r takes the r-th slice, the split by token position of plain
        context parallelism; an ablation without load balancing)."""
        if L <= 0 or B <= 0 or R <= 0 or L % B:
            raise ValueError("need L, B, R > 0 and L a multiple of B")
        if policy not in POLICIES:
            raise ValueError(f"policy must be one of {POLICIES}")
        N = L // B
        if N % R:
            raise ValueError("the clean shards hold whole blocks: (L / B) must be a multiple of R")
        per = N // R
        plan = CSBPPlan(L, B, R, policy)
        plan.clean_shards = [(r * per, (r + 1) * per) for r in range(R)]
        plan.noisy_owner = [(R - 1 - j // per) if policy == "mirror" else j // per for j in range(N)]
        # work of block j of either stream: B rows reading (j + 1) B keys
        cost = [B * (j + 1) * B for j in range(N)]
        plan.load = [sum(cost[j] for j in range(a, b)) for (a, b) in plan.clean_shards]
        for j, r in enumerate(plan.noisy_owner):
            plan.load[r] += cost[j]
        return plan

    def rows(self, r: int) -> Rows:
        c0, c1 = self.clean_shards[r]
        n0, n1 = self.clean_shards[self.R - 1 - r if self.policy == "mirror" else r]
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


def _gathered(shards):
    """The whole clean K and V from the all-gathered shards."""
    import torch
    return torch.cat([k for (k, _) in shards]), torch.cat([v for (_, v) in shards])


def forward(plan: CSBPPlan, comm, compute, shards, gathered: bool = False):
    """Forward of the rank's rows given ``shards`` from ``gather_clean_kv``.
    Per-shard schedule (default): partials against every clean shard in
    order, then the local partial, merged (the order a ring that overlaps
    the exchange with compute would follow).  ``gathered``: one call over the
    whole clean sequence and the local blocks (the rank holds every clean
    shard after the all-gather; no partials, no merge).  Returns the rank's
    (Oc, On, LSEc, LSEn) rows."""
    rows = plan.rows(comm.rank)
    if gathered:
        return compute.merge([compute.fwd(rows, (0, plan.L), _gathered(shards), True)])
    # a running merge: each partial is folded in as it is computed, so that
    # no more than two are held (the LSE merge is associative)
    acc = None
    for s in range(plan.R):
        part = compute.fwd(rows, plan.shard_keys(s), shards[s], False)
        acc = part if acc is None else compute.merge([acc, part])
    return compute.merge([acc, compute.fwd(rows, (0, 0), None, True)])


def backward(plan: CSBPPlan, comm, compute, shards, out, dO, gathered: bool = False):
    """Backward of the rank's rows given its merged forward outputs
    ``out`` = (Oc, On, LSEc, LSEn) and upstream ``dO`` = (dOc, dOn) of its
    rows.  Returns (dQc, dQn) of its rows, the clean (dK, dV) of its own
    shard (summed over every rank's rows) and the corrupted (dK, dV) of its
    own blocks.  ``gathered``: one call over the whole clean sequence, its
    clean dK / dV then summed shard by shard onto the owners."""
    rows = plan.rows(comm.rank)
    Oc, On, LSEc, LSEn = out
    stats = (LSEc, LSEn, compute.preprocess(Oc, dO[0]), compute.preprocess(On, dO[1]))
    mine = None
    if gathered:
        dQc, dQn, gk, gv, gkn, gvn = compute.bwd(rows, (0, plan.L), _gathered(shards), True, stats)
        for s in range(plan.R):
            a, b = plan.shard_keys(s)
            k = comm.sum_to_owner(gk[a:b], s)
            v = comm.sum_to_owner(gv[a:b], s)
            if s == comm.rank:
                mine = (k, v)
        return (dQc, dQn), mine, (gkn, gvn)
    dQc = dQn = None
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


class TorchComm:
    """The transport over torch.distributed: gloo for CPU tensors, NCCL for
    CUDA tensors (no kernel of this library reads a peer's memory: every
    exchanged shard lands in the rank's own memory first).  Uses the default
    process group."""

    def __init__(self):
        import torch.distributed as dist
        self._dist = dist
        self.rank = dist.get_rank()
        self.world = dist.get_world_size()

    def all_gather(self, x):
        """Every rank's ``x`` (same shape on every rank), in rank order."""
        import torch
        x = x.contiguous()
        out = [torch.empty_like(x) for _ in range(self.world)]
        self._dist.all_gather(out, x)
        return out

    def sum_to_owner(self, x, owner):
        """The sum over ranks of ``x`` on rank ``owner`` (None elsewhere)."""
        t = x.clone().contiguous()
        self._dist.reduce(t, dst=owner, op=self._dist.ReduceOp.SUM)
        return t if self.rank == owner else None


class KernelCompute:
    """One rank's compute on its GPU through the library's rank-local calls
    (``bdlm_attn_fwd_rank``, ``bdlm_lse_merge``, ``bdlm_bwd_preprocess``,
    ``bdlm_attn_bwd_rank``).

    ``local`` holds the rank's own tensors on the device: "Qc", "Kc", "Vc",
    "dOc" are the rows of its clean shard, "Qn", "Kn", "Vn", "dOn" the rows of
    its corrupted blocks ([rows, H, d], bf16).  Nothing of length L is held:
    the calls take the rank's rows as they are, each clean shard (or the whole
    gathered clean sequence) as received, and return results for the rank's
    rows and the call's keys only."""

    def __init__(self, lib, plan: CSBPPlan, rank: int, local: dict, scale: float):
        import torch
        self.lib, self.plan, self.scale = lib, plan, scale
        B = plan.B
        rw = plan.rows(rank)
        self.rc, self.rn = (rw.c0 * B, rw.c1 * B), (rw.n0 * B, rw.n1 * B)
        self.loc = {k: v.contiguous() for k, v in local.items()}
        kn = self.loc["Kn"]
        self.no_keys = torch.empty((0,) + tuple(kn.shape[1:]), dtype=kn.dtype, device=kn.device)

    def _kv(self, kv_data):
        if kv_data is None:
            return self.no_keys, self.no_keys
        return kv_data[0].contiguous(), kv_data[1].contiguous()

    def fwd(self, rows, kv, kv_data, local):
        Kc, Vc = self._kv(kv_data)
        x = self.loc
        return self.lib.bdlm_attn_fwd_rank(x["Qc"], Kc, Vc, x["Qn"], x["Kn"], x["Vn"], self.plan.L, self.plan.B,
                                           kv[0], kv[1], local, self.rc, self.rn, self.scale)

    def merge(self, parts):
        import torch
        oc, lc = self.lib.bdlm_lse_merge([p[0] for p in parts], [p[2] for p in parts], o_dtype=torch.float32)
        on, ln = self.lib.bdlm_lse_merge([p[1] for p in parts], [p[3] for p in parts], o_dtype=torch.float32)
        return oc, on, lc, ln

    def preprocess(self, O, dO):
        return self.lib.bdlm_bwd_preprocess(O.contiguous(), dO.contiguous())

    def bwd(self, rows, kv, kv_data, local, stats):
        import torch
        Kc, Vc = self._kv(kv_data)
        x = self.loc
        f32 = dict(dtype=torch.float32, device=x["Qc"].device)
        z = lambda t: torch.zeros(t.shape, **f32)
        acc = (z(x["Qc"]), z(x["Qn"]), z(Kc), z(Vc), z(x["Kn"]), z(x["Vn"]))
        LSEc, LSEn, Dc, Dn = (t.contiguous() for t in stats)
        self.lib.bdlm_attn_bwd_rank(x["Qc"], Kc, Vc, x["Qn"], x["Kn"], x["Vn"], x["dOc"], x["dOn"], LSEc, LSEn, Dc,
                                    Dn, self.plan.L, self.plan.B, kv[0], kv[1], local, self.rc, self.rn, *acc,
                                    self.scale)
        return acc
