"""Multi-rank CSBP (context-sharded block parallelism) on the CPU: the
partition and exchange plan of structured_mask_attention_gb300/csbp.py run as
two and four gloo ranks, with the fp64 oracle as the compute object.  Each
rank starts with only its own data (its clean shard's rows, keys and values;
its corrupted blocks), receives the other clean shards through the exchange,
and its outputs and gradients must equal the unsharded oracle's
(Proposition 1, evolve.pub FAQ "Does CSBP change training results?")."""
from __future__ import annotations

import math
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

from structured_mask_attention_gb300 import csbp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


class _GlooComm:
    def __init__(self):
        self.rank = dist.get_rank()
        self.world = dist.get_world_size()

    def all_gather(self, x):
        t = torch.from_numpy(np.ascontiguousarray(x))
        out = [torch.empty_like(t) for _ in range(self.world)]
        dist.all_gather(out, t)
        return [o.numpy() for o in out]

    def sum_to_owner(self, x, owner):
        t = torch.from_numpy(np.ascontiguousarray(x)).clone()
        dist.reduce(t, dst=owner, op=dist.ReduceOp.SUM)
        return t.numpy() if self.rank == owner else None


class _OracleCompute:
    """The oracle on one rank's rows: its local arrays are placed into
    full-length zero arrays (rows it does not own get zero queries, upstream
    gradients and statistics, so they contribute nothing) and the oracle's
    partial functions compute the requested key range."""

    def __init__(self, orc, local, rows, L, B, sc):
        self.orc, self.loc, self.rows, self.L, self.B, self.sc = orc, local, rows, L, B, sc
        self.crow = slice(rows.c0 * B, rows.c1 * B)
        self.nrows = np.concatenate([np.arange(j * B, (j + 1) * B) for j in rows.noisy_blocks]) \
            if rows.noisy_blocks else np.zeros(0, dtype=np.int64)
        self.blocks = sorted(set(range(rows.c0, rows.c1)) | set(rows.noisy_blocks))

    def _put(self, name, shape_from):
        full = np.zeros((self.L,) + self.loc[shape_from].shape[1:])
        if name.endswith("c"):
            full[self.crow] = self.loc[name]
        else:
            full[self.nrows] = self.loc[name]
        return full

    def _inputs(self, kv, kv_data, local):
        Qc, Qn = self._put("Qc", "Qc"), self._put("Qn", "Qn")
        Kc = np.zeros((self.L,) + self.loc["Kc"].shape[1:])
        Vc = np.zeros_like(Kc)
        if kv_data is not None:
            Kc[kv[0]:kv[1]], Vc[kv[0]:kv[1]] = kv_data
        Kn, Vn = (self._put("Kn", "Kn"), self._put("Vn", "Vn")) if local else (np.zeros_like(Kc), np.zeros_like(Kc))
        return Qc, Kc, Vc, Qn, Kn, Vn

    def fwd(self, rows, kv, kv_data, local):
        Oc, On, LSEc, LSEn = self.orc.fwd_partial(*self._inputs(kv, kv_data, local), self.B, self.sc, kv[0], kv[1],
                                                  local, blocks=self.blocks)
        return Oc[self.crow], On[self.nrows], LSEc[:, self.crow], LSEn[:, self.nrows]

    def merge(self, parts):
        Oc, LSEc = self.orc.lse_merge([p[0] for p in parts], [p[2] for p in parts])
        On, LSEn = self.orc.lse_merge([p[1] for p in parts], [p[3] for p in parts])
        return Oc, On, LSEc, LSEn

    def preprocess(self, O, dO):
        return self.orc.bwd_preprocess(O, dO)

    def bwd(self, rows, kv, kv_data, local, stats):
        LSEc_r, LSEn_r, Dc_r, Dn_r = stats
        H = LSEc_r.shape[0]
        stat = lambda v, sel: (lambda a: (a.__setitem__((slice(None), sel), v), a)[1])(np.zeros((H, self.L)))
        g = self.orc.bwd_partial(*self._inputs(kv, kv_data, local), self._put("dOc", "dOc"),
                                 self._put("dOn", "dOn"), stat(LSEc_r, self.crow), stat(LSEn_r, self.nrows),
                                 stat(Dc_r, self.crow), stat(Dn_r, self.nrows), self.B, self.sc, kv[0], kv[1], local,
                                 blocks=self.blocks)
        dQc, dKc, dVc, dQn, dKn, dVn = g
        return (dQc[self.crow], dQn[self.nrows], dKc[kv[0]:kv[1]], dVc[kv[0]:kv[1]], dKn[self.nrows],
                dVn[self.nrows])


def _rank_main(rank, world, port, L, B, Hq, Hkv, d, out):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import oracle.bdlm_oracle as orc
    from structured_mask_attention_gb300.inputs import make_numpy
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        X = {k: v.astype(np.float64) for k, v in make_numpy(L, Hq, Hkv, d, seed=11).items()}
        sc = 1.0 / math.sqrt(d)
        plan = csbp.CSBPPlan.build(L, B, world)
        rows = plan.rows(rank)
        crow = slice(rows.c0 * B, rows.c1 * B)
        nrows = np.concatenate([np.arange(j * B, (j + 1) * B) for j in rows.noisy_blocks])
        # this rank's own data only
        local = {"Qc": X["Qc"][crow], "Kc": X["Kc"][crow], "Vc": X["Vc"][crow], "dOc": X["dOc"][crow],
                 "Qn": X["Qn"][nrows], "Kn": X["Kn"][nrows], "Vn": X["Vn"][nrows], "dOn": X["dOn"][nrows]}
        comm = _GlooComm()
        comp = _OracleCompute(orc, local, rows, L, B, sc)
        shards = csbp.gather_clean_kv(comm, local["Kc"], local["Vc"])
        o = csbp.forward(plan, comm, comp, shards)
        (dqc, dqn), (dkc, dvc), (dkn, dvn) = csbp.backward(plan, comm, comp, shards, o,
                                                          (local["dOc"], local["dOn"]))
        names = ("Qc", "Kc", "Vc", "Qn", "Kn", "Vn")
        rf = orc.fwd_blockwise(*[X[k] for k in names], B, sc)
        rg = orc.bwd_blockwise(*[X[k] for k in names], X["dOc"], X["dOn"], B, sc)
        err = 0.0
        for got, ref in ((o[0], rf[0][crow]), (o[1], rf[1][nrows]), (o[2], rf[2][:, crow]), (o[3], rf[3][:, nrows]),
                         (dqc, rg[0][crow]), (dqn, rg[3][nrows]), (dkc, rg[1][crow]), (dvc, rg[2][crow]),
                         (dkn, rg[4][nrows]), (dvn, rg[5][nrows])):
            err = max(err, float(np.abs(got - ref).max() / max(1.0, np.abs(ref).max())))
        out.put((rank, err, len(rows.noisy_blocks)))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world,L,B", [(2, 256, 16), (4, 256, 16)])
def test_csbp_ranks_match_unsharded_oracle(world, L, B):
    Hq, Hkv, d = 2, 1, 16
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, L, B, Hq, Hkv, d, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=300) for _ in range(world))
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert sum(n for (_, _, n) in got) == L // B        # every corrupted block owned once
    for rank, err, _ in got:
        assert err <= 1e-12, (rank, err)


def test_csbp_plan_covers_and_balances():
    for (L, B, R) in ((262144, 1024, 8), (131072, 512, 8), (4096, 128, 4), (256, 16, 2)):
        plan = csbp.CSBPPlan.build(L, B, R)
        N = L // B
        assert [a for (a, _) in plan.clean_shards] == [r * N // R for r in range(R)]
        assert plan.clean_shards[-1][1] == N
        assert sorted(j for r in range(R) for j in plan.rows(r).noisy_blocks) == list(range(N))
        assert plan.imbalance() == 1.0, (L, B, R, plan.imbalance())
        for r in range(R):
            rw = plan.rows(r)
            assert (rw.n0, rw.n1) == plan.clean_shards[R - 1 - r]   # the mirror slice, contiguous
    with pytest.raises(ValueError):
        csbp.CSBPPlan.build(256, 16, 3)   # 16 blocks do not split into 3 whole-block shards
