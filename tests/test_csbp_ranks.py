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


def _np(x):
    return x.numpy() if isinstance(x, torch.Tensor) else np.asarray(x)


def _t(*xs):
    return tuple(torch.from_numpy(np.ascontiguousarray(x)) for x in xs)


class _OracleCompute:
    """The oracle on one rank's rows: its local arrays are placed into
    full-length zero arrays (rows it does not own get zero queries, upstream
    gradients and statistics, so they contribute nothing) and the oracle's
    partial functions compute the requested key range.  Takes and returns
    CPU tensors, the currency of the transport."""

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
            Kc[kv[0]:kv[1]], Vc[kv[0]:kv[1]] = _np(kv_data[0]), _np(kv_data[1])
        Kn, Vn = (self._put("Kn", "Kn"), self._put("Vn", "Vn")) if local else (np.zeros_like(Kc), np.zeros_like(Kc))
        return Qc, Kc, Vc, Qn, Kn, Vn

    def fwd(self, rows, kv, kv_data, local):
        Oc, On, LSEc, LSEn = self.orc.fwd_partial(*self._inputs(kv, kv_data, local), self.B, self.sc, kv[0], kv[1],
                                                  local, blocks=self.blocks)
        return _t(Oc[self.crow], On[self.nrows], LSEc[:, self.crow], LSEn[:, self.nrows])

    def merge(self, parts):
        Oc, LSEc = self.orc.lse_merge([_np(p[0]) for p in parts], [_np(p[2]) for p in parts])
        On, LSEn = self.orc.lse_merge([_np(p[1]) for p in parts], [_np(p[3]) for p in parts])
        return _t(Oc, On, LSEc, LSEn)

    def preprocess(self, O, dO):
        return _t(self.orc.bwd_preprocess(_np(O), _np(dO)))[0]

    def bwd(self, rows, kv, kv_data, local, stats):
        LSEc_r, LSEn_r, Dc_r, Dn_r = (_np(x) for x in stats)
        H = LSEc_r.shape[0]
        stat = lambda v, sel: (lambda a: (a.__setitem__((slice(None), sel), v), a)[1])(np.zeros((H, self.L)))
        g = self.orc.bwd_partial(*self._inputs(kv, kv_data, local), self._put("dOc", "dOc"),
                                 self._put("dOn", "dOn"), stat(LSEc_r, self.crow), stat(LSEn_r, self.nrows),
                                 stat(Dc_r, self.crow), stat(Dn_r, self.nrows), self.B, self.sc, kv[0], kv[1], local,
                                 blocks=self.blocks)
        dQc, dKc, dVc, dQn, dKn, dVn = g
        return _t(dQc[self.crow], dQn[self.nrows], dKc[kv[0]:kv[1]], dVc[kv[0]:kv[1]], dKn[self.nrows],
                  dVn[self.nrows])


def _rank_main(rank, world, port, L, B, Hq, Hkv, d, out, policy="mirror", gathered=False):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import oracle.bdlm_oracle as orc
    from structured_mask_attention_gb300.inputs import make_numpy
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        X = {k: v.astype(np.float64) for k, v in make_numpy(L, Hq, Hkv, d, seed=11).items()}
        sc = 1.0 / math.sqrt(d)
        plan = csbp.CSBPPlan.build(L, B, world, policy)
        rows = plan.rows(rank)
        crow = slice(rows.c0 * B, rows.c1 * B)
        nrows = np.concatenate([np.arange(j * B, (j + 1) * B) for j in rows.noisy_blocks])
        # this rank's own data only
        local = {"Qc": X["Qc"][crow], "Kc": X["Kc"][crow], "Vc": X["Vc"][crow], "dOc": X["dOc"][crow],
                 "Qn": X["Qn"][nrows], "Kn": X["Kn"][nrows], "Vn": X["Vn"][nrows], "dOn": X["dOn"][nrows]}
        comm = csbp.TorchComm()
        comp = _OracleCompute(orc, local, rows, L, B, sc)
        shards = csbp.gather_clean_kv(comm, *_t(local["Kc"], local["Vc"]))
        o = [_np(x) for x in csbp.forward(plan, comm, comp, shards, gathered)]
        (dqc, dqn), (dkc, dvc), (dkn, dvn) = csbp.backward(plan, comm, comp, shards, _t(*o),
                                                          _t(local["dOc"], local["dOn"]), gathered)
        dqc, dqn, dkc, dvc, dkn, dvn = (_np(x) for x in (dqc, dqn, dkc, dvc, dkn, dvn))
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


@pytest.mark.parametrize("world,L,B,policy,gathered", [(2, 256, 16, "mirror", False), (4, 256, 16, "mirror", False),
                                                        (4, 256, 16, "contiguous", False),
                                                        (4, 256, 16, "mirror", True)])
def test_csbp_ranks_match_unsharded_oracle(world, L, B, policy, gathered):
    Hq, Hkv, d = 2, 1, 16
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, L, B, Hq, Hkv, d, q, policy, gathered))
             for r in range(world)]
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
    with pytest.raises(ValueError):
        csbp.CSBPPlan.build(256, 16, 2, "lpt")


def test_csbp_contiguous_ablation_is_unbalanced():
    """The split by token position (rank r owns clean and corrupted slice r)
    puts the most work on the last rank: slice r of n blocks holds
    n^2 (r + 1/2) + n/2 block-units of work per stream, so the largest load
    over the mean is (2 R n - n + 1) / (R n + 1) -> 2 - 1/R."""
    for (L, B, R) in ((262144, 1024, 8), (131072, 512, 4), (4096, 128, 2)):
        plan = csbp.CSBPPlan.build(L, B, R, "contiguous")
        n = L // B // R
        assert [plan.rows(r).n0 for r in range(R)] == [r * n for r in range(R)]
        assert abs(plan.imbalance() - (2 * R * n - n + 1) / (R * n + 1)) < 1e-12
        assert plan.load == sorted(plan.load)
