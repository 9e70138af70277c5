"""Multi-rank CSBP's per-rank compute on one GPU: every rank of the plan
(structured_mask_attention_gb300/csbp.py: clean shard r, the mirror slice of
corrupted blocks) makes its calls in turn with the row-restricted kernels
(bdlm_attn_fwd_shard_rows, bdlm_attn_bwd_shard_rows).  Each rank merges the
partials of its own rows; the backward adds every rank's contributions into
shared fp32 accumulators (the sum a reduce-scatter makes across ranks).
The reassembled outputs and gradients must match the fp64 oracle, and a
call must leave the rows outside its ranges untouched."""
from __future__ import annotations

import math

import numpy as np
import pytest

import oracle.bdlm_oracle as orc
from structured_mask_attention_gb300 import csbp
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


@pytest.mark.parametrize("L,B,R,Hq,Hkv,d", [
    (4096, 256, 4, 8, 4, 128),   # rank slices of 1024 rows
    (4096, 128, 8, 4, 2, 128),   # 8 ranks, slices of 512 rows
    (512, 32, 4, 2, 1, 64),      # slices of 128 rows: forward items (256 rows) straddle two ranks
    (768, 32, 4, 3, 1, 128),     # slices of 192 rows: no tile boundary matches a rank boundary
])
def test_rank_rows_reassemble_unsharded(lib, L, B, R, Hq, Hkv, d):
    m = lib
    X = make_numpy(L, Hq, Hkv, d, seed=L + R)
    X64 = {k: v.astype(np.float64) for k, v in X.items()}
    dev = {k: to_dev(v, torch) for k, v in X.items()}
    ins = [dev[k] for k in NAMES[:6]]
    sc = 1.0 / math.sqrt(d)
    plan = csbp.CSBPPlan.build(L, B, R)
    f32 = dict(dtype=torch.float32, device="cuda")
    Oc, On = torch.zeros((L, Hq, d), **f32), torch.zeros((L, Hq, d), **f32)
    LSEc, LSEn = torch.full((Hq, L), float("nan"), **f32), torch.full((Hq, L), float("nan"), **f32)
    specs = [(*plan.shard_keys(s), False) for s in range(R)] + [(0, 0, True)]
    for r in range(R):
        rw = plan.rows(r)
        rc, rn = (rw.c0 * B, rw.c1 * B), (rw.n0 * B, rw.n1 * B)
        parts = [m.bdlm_attn_fwd_shard_rows(*ins, B, lo, hi, loc, rc, rn, sc) for (lo, hi, loc) in specs]
        # rows outside the rank's ranges keep the outputs' initial values
        for p in parts:
            for (a, b), O, LSE in ((rc, p[0], p[2]), (rn, p[1], p[3])):
                assert not O[:a].any() and not O[b:].any()
                assert torch.isneginf(LSE[:, :a]).all() and torch.isneginf(LSE[:, b:]).all()
        oc, lc = m.bdlm_lse_merge([p[0] for p in parts], [p[2] for p in parts], o_dtype=torch.float32)
        on, ln = m.bdlm_lse_merge([p[1] for p in parts], [p[3] for p in parts], o_dtype=torch.float32)
        Oc[rc[0]:rc[1]], LSEc[:, rc[0]:rc[1]] = oc[rc[0]:rc[1]], lc[:, rc[0]:rc[1]]
        On[rn[0]:rn[1]], LSEn[:, rn[0]:rn[1]] = on[rn[0]:rn[1]], ln[:, rn[0]:rn[1]]
    assert not torch.isnan(LSEc).any() and not torch.isnan(LSEn).any()   # every row owned by some rank
    ref = orc.fwd_blockwise(*[X64[k] for k in NAMES[:6]], B, sc)
    check_rel("Oc (ranks)", to_np(Oc), ref[0])
    check_rel("On (ranks)", to_np(On), ref[1])
    check_lse("LSEc (ranks)", to_np(LSEc), ref[2])
    check_lse("LSEn (ranks)", to_np(LSEn), ref[3])
    # backward: merged statistics, every rank's contributions added up
    Dc = m.bdlm_bwd_preprocess(Oc.to(torch.bfloat16), dev["dOc"])
    Dn = m.bdlm_bwd_preprocess(On.to(torch.bfloat16), dev["dOn"])
    z = lambda H: torch.zeros((L, H, d), **f32)
    dQc, dQn, dKc, dVc, dKn, dVn = z(Hq), z(Hq), z(Hkv), z(Hkv), z(Hkv), z(Hkv)
    for r in range(R):
        rw = plan.rows(r)
        rc, rn = (rw.c0 * B, rw.c1 * B), (rw.n0 * B, rw.n1 * B)
        for (lo, hi, loc) in specs:
            m.bdlm_attn_bwd_shard_rows(*ins, dev["dOc"], dev["dOn"], LSEc, LSEn, Dc, Dn, B, lo, hi, loc, rc, rn,
                                       dQc, dQn, dKc, dVc, dKn, dVn, sc)
    gref = orc.bwd_blockwise(*[X64[k] for k in NAMES], B, sc)
    for name, g, r_ in zip(("dQc", "dKc", "dVc", "dQn", "dKn", "dVn"), (dQc, dKc, dVc, dQn, dKn, dVn), gref):
        check_rel(f"{name} (ranks)", to_np(g), r_)


def test_rank_rows_validation(lib):
    m = lib
    X = make_numpy(256, 2, 1, 64, seed=3)
    ins = [to_dev(X[k], torch) for k in NAMES[:6]]
    with pytest.raises(m.BdlmError) as e:
        m.bdlm_attn_fwd_shard_rows(*ins, 32, 0, 256, True, (0, 300), (0, 256))
    assert e.value.status == 2
    with pytest.raises(m.BdlmError) as e:
        m.bdlm_attn_fwd_shard_rows(*ins, 32, 0, 256, True, (128, 64), (0, 256))
    assert e.value.status == 2


class _ThreadComm:
    """R ranks as host threads of one process, exchanging through shared
    slots and a barrier.  Only the host waits: every rank's kernels go to the
    device's default stream in the order the threads issue them, and no
    kernel waits on another."""

    class Shared:
        def __init__(self, world):
            import threading
            self.world = world
            self.slots = [None] * world
            self.barrier = threading.Barrier(world, timeout=600)

    def __init__(self, shared, rank):
        self.s, self.rank, self.world = shared, rank, shared.world

    def all_gather(self, x):
        self.s.slots[self.rank] = x.clone()
        self.s.barrier.wait()
        out = list(self.s.slots)
        self.s.barrier.wait()
        return out

    def sum_to_owner(self, x, owner):
        self.s.slots[self.rank] = x.clone()
        self.s.barrier.wait()
        res = None
        if self.rank == owner:   # summed in rank order
            res = self.s.slots[0].clone()
            for t in self.s.slots[1:]:
                res += t
        self.s.barrier.wait()
        return res


@pytest.mark.parametrize("L,B,R,Hq,Hkv,d,policy,gathered", [
    (1024, 64, 4, 4, 2, 128, "mirror", False),
    (2048, 64, 8, 2, 1, 128, "mirror", False),
    (1024, 32, 4, 2, 2, 64, "contiguous", False),
    (2048, 64, 8, 2, 1, 128, "mirror", True),
    (768, 32, 4, 3, 1, 64, "contiguous", True),
])
def test_csbp_driver_on_kernels(lib, L, B, R, Hq, Hkv, d, policy, gathered):
    """The per-rank CSBP driver (csbp.forward / csbp.backward) with
    csbp.KernelCompute on every rank: each rank starts from its own rows
    only, clean K/V are all-gathered, clean dK/dV summed onto the shard
    owners; per-shard partials or one call over the gathered sequence.  The
    reassembled outputs and gradients match the fp64 oracle."""
    import threading

    m = lib
    X = make_numpy(L, Hq, Hkv, d, seed=L + R + 7)
    X64 = {k: v.astype(np.float64) for k, v in X.items()}
    dev = {k: to_dev(v, torch) for k, v in X.items()}
    sc = 1.0 / math.sqrt(d)
    plan = csbp.CSBPPlan.build(L, B, R, policy)
    shared = _ThreadComm.Shared(R)
    results, errors = [None] * R, []

    def rank_job(r):
        try:
            rw = plan.rows(r)
            c, n = slice(rw.c0 * B, rw.c1 * B), slice(rw.n0 * B, rw.n1 * B)
            local = {k: dev[k][c].clone() for k in ("Qc", "Kc", "Vc", "dOc")}
            local.update({k: dev[k][n].clone() for k in ("Qn", "Kn", "Vn", "dOn")})
            comm = _ThreadComm(shared, r)
            comp = csbp.KernelCompute(m, plan, r, local, sc)
            shards = csbp.gather_clean_kv(comm, local["Kc"], local["Vc"])
            o = csbp.forward(plan, comm, comp, shards, gathered)
            g = csbp.backward(plan, comm, comp, shards, o, (local["dOc"], local["dOn"]), gathered)
            torch.cuda.synchronize()
            results[r] = (o, g)
        except BaseException as e:  # release the other ranks, then report
            errors.append(e)
            shared.barrier.abort()

    threads = [threading.Thread(target=rank_job, args=(r,)) for r in range(R)]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=900)
    assert not errors, errors[0]
    f32 = dict(dtype=torch.float32, device="cuda")
    Oc, On = torch.zeros((L, Hq, d), **f32), torch.zeros((L, Hq, d), **f32)
    LSEc, LSEn = torch.zeros((Hq, L), **f32), torch.zeros((Hq, L), **f32)
    dQc, dQn = torch.zeros((L, Hq, d), **f32), torch.zeros((L, Hq, d), **f32)
    dKc, dVc, dKn, dVn = (torch.zeros((L, Hkv, d), **f32) for _ in range(4))
    for r in range(R):
        rw = plan.rows(r)
        c, n = slice(rw.c0 * B, rw.c1 * B), slice(rw.n0 * B, rw.n1 * B)
        (oc, on, lc, ln), ((gqc, gqn), (gkc, gvc), (gkn, gvn)) = results[r]
        Oc[c], On[n], LSEc[:, c], LSEn[:, n] = oc, on, lc, ln
        dQc[c], dQn[n], dKc[c], dVc[c], dKn[n], dVn[n] = gqc, gqn, gkc, gvc, gkn, gvn
    ref = orc.fwd_blockwise(*[X64[k] for k in NAMES[:6]], B, sc)
    check_rel("Oc (driver)", to_np(Oc), ref[0])
    check_rel("On (driver)", to_np(On), ref[1])
    check_lse("LSEc (driver)", to_np(LSEc), ref[2])
    check_lse("LSEn (driver)", to_np(LSEn), ref[3])
    gref = orc.bwd_blockwise(*[X64[k] for k in NAMES], B, sc)
    for name, g, r_ in zip(("dQc", "dKc", "dVc", "dQn", "dKn", "dVn"), (dQc, dKc, dVc, dQn, dKn, dVn), gref):
        check_rel(f"{name} (driver)", to_np(g), r_)


def test_rank_rows_empty_and_one_sided(lib):
    """A call with no rows writes nothing and adds nothing; a call with
    rows of one stream only matches the oracle on those rows."""
    m = lib
    L, B, Hq, Hkv, d = 512, 32, 2, 1, 64
    X = make_numpy(L, Hq, Hkv, d, seed=5)
    X64 = {k: v.astype(np.float64) for k, v in X.items()}
    dev = {k: to_dev(v, torch) for k, v in X.items()}
    ins = [dev[k] for k in NAMES[:6]]
    sc = 1.0 / math.sqrt(d)
    o = m.bdlm_attn_fwd_shard_rows(*ins, B, 0, L, True, (0, 0), (0, 0), sc)
    assert not o[0].any() and not o[1].any()
    assert torch.isneginf(o[2]).all() and torch.isneginf(o[3]).all()
    f = m.bdlm_attn_fwd(*ins, B, sc, o_dtype=torch.float32)
    Dc, Dn = m.bdlm_bwd_preprocess(f[0], dev["dOc"]), m.bdlm_bwd_preprocess(f[1], dev["dOn"])
    z = lambda H: torch.zeros((L, H, d), dtype=torch.float32, device="cuda")
    acc = (z(Hq), z(Hq), z(Hkv), z(Hkv), z(Hkv), z(Hkv))
    m.bdlm_attn_bwd_shard_rows(*ins, dev["dOc"], dev["dOn"], f[2], f[3], Dc, Dn, B, 0, L, True, (0, 0), (0, 0),
                               *acc, sc)
    assert not any(a.any() for a in acc)
    ref = orc.fwd_blockwise(*[X64[k] for k in NAMES[:6]], B, sc)
    o = m.bdlm_attn_fwd_shard_rows(*ins, B, 0, L, True, (0, 0), (100, 400), sc)   # corrupted rows only
    check_rel("On rows 100..400", to_np(o[1])[100:400], ref[1][100:400])
    check_lse("LSEn rows 100..400", to_np(o[3])[:, 100:400], ref[3][:, 100:400])
    assert not o[0].any() and not o[1][:100].any() and not o[1][400:].any()
    o = m.bdlm_attn_fwd_shard_rows(*ins, B, 0, L, True, (37, 300), (0, 0), sc)    # clean rows only
    check_rel("Oc rows 37..300", to_np(o[0])[37:300], ref[0][37:300])
    assert not o[1].any() and not o[0][:37].any() and not o[0][300:].any()


@pytest.mark.parametrize("L,B,R,Hq,Hkv,d", [
    (2048, 128, 4, 4, 2, 128),
    (768, 32, 4, 3, 1, 64),      # slices of 192 rows: tiles straddle the held rows
])
def test_rank_local_tensors(lib, L, B, R, Hq, Hkv, d):
    """bdlm_attn_fwd_rank / bdlm_attn_bwd_rank on tensors that hold only a
    rank's rows and one clean shard's keys: every partial equals the
    full-length call's rows bit for bit, and the ranks' merged outputs and
    summed gradients match the fp64 oracle."""
    m = lib
    X = make_numpy(L, Hq, Hkv, d, seed=L + 3 * R)
    X64 = {k: v.astype(np.float64) for k, v in X.items()}
    dev = {k: to_dev(v, torch) for k, v in X.items()}
    ins = [dev[k] for k in NAMES[:6]]
    sc = 1.0 / math.sqrt(d)
    plan = csbp.CSBPPlan.build(L, B, R)
    f32 = dict(dtype=torch.float32, device="cuda")
    Oc, On = torch.zeros((L, Hq, d), **f32), torch.zeros((L, Hq, d), **f32)
    LSEc, LSEn = torch.zeros((Hq, L), **f32), torch.zeros((Hq, L), **f32)
    dQc, dQn = torch.zeros((L, Hq, d), **f32), torch.zeros((L, Hq, d), **f32)
    dKc, dVc, dKn, dVn = (torch.zeros((L, Hkv, d), **f32) for _ in range(4))
    no_keys = torch.empty((0, Hkv, d), dtype=torch.bfloat16, device="cuda")
    specs = [(*plan.shard_keys(s), False) for s in range(R)] + [(0, 0, True)]
    for r in range(R):
        rw = plan.rows(r)
        rc, rn = (rw.c0 * B, rw.c1 * B), (rw.n0 * B, rw.n1 * B)
        c, n = slice(*rc), slice(*rn)
        loc = {k: dev[k][c].contiguous() for k in ("Qc", "dOc")}
        loc.update({k: dev[k][n].contiguous() for k in ("Qn", "Kn", "Vn", "dOn")})
        kv = lambda lo, hi: ((dev["Kc"][lo:hi].contiguous(), dev["Vc"][lo:hi].contiguous()) if hi > lo
                             else (no_keys, no_keys))
        parts = []
        for (lo, hi, local) in specs:
            Kc_, Vc_ = kv(lo, hi)
            pl = m.bdlm_attn_fwd_rank(loc["Qc"], Kc_, Vc_, loc["Qn"], loc["Kn"], loc["Vn"], L, B, lo, hi, local,
                                      rc, rn, sc)
            pf = m.bdlm_attn_fwd_shard_rows(*ins, B, lo, hi, local, rc, rn, sc)
            for got, full in ((pl[0], pf[0][c]), (pl[1], pf[1][n]), (pl[2], pf[2][:, c]), (pl[3], pf[3][:, n])):
                assert torch.equal(got, full)
            parts.append(pl)
        oc, lc = m.bdlm_lse_merge([p[0] for p in parts], [p[2] for p in parts], o_dtype=torch.float32)
        on, ln = m.bdlm_lse_merge([p[1] for p in parts], [p[3] for p in parts], o_dtype=torch.float32)
        Oc[c], On[n], LSEc[:, c], LSEn[:, n] = oc, on, lc, ln
        Dc, Dn = m.bdlm_bwd_preprocess(oc, loc["dOc"]), m.bdlm_bwd_preprocess(on, loc["dOn"])
        z = lambda t: torch.zeros(t.shape, **f32)
        aq = (z(loc["Qc"]), z(loc["Qn"]))
        akn = (z(loc["Kn"]), z(loc["Vn"]))
        for (lo, hi, local) in specs:
            Kc_, Vc_ = kv(lo, hi)
            akc = (z(Kc_), z(Vc_))
            m.bdlm_attn_bwd_rank(loc["Qc"], Kc_, Vc_, loc["Qn"], loc["Kn"], loc["Vn"], loc["dOc"], loc["dOn"],
                                 lc.contiguous(), ln.contiguous(), Dc, Dn, L, B, lo, hi, local, rc, rn, *aq, *akc,
                                 *akn, sc)
            dKc[lo:hi] += akc[0]
            dVc[lo:hi] += akc[1]
        dQc[c], dQn[n], dKn[n], dVn[n] = aq[0], aq[1], akn[0], akn[1]
    ref = orc.fwd_blockwise(*[X64[k] for k in NAMES[:6]], B, sc)
    check_rel("Oc (rank-local)", to_np(Oc), ref[0])
    check_rel("On (rank-local)", to_np(On), ref[1])
    check_lse("LSEc (rank-local)", to_np(LSEc), ref[2])
    check_lse("LSEn (rank-local)", to_np(LSEn), ref[3])
    gref = orc.bwd_blockwise(*[X64[k] for k in NAMES], B, sc)
    for name, g, r_ in zip(("dQc", "dKc", "dVc", "dQn", "dKn", "dVn"), (dQc, dKc, dVc, dQn, dKn, dVn), gref):
        check_rel(f"{name} (rank-local)", to_np(g), r_)


def test_rank_local_validation(lib):
    m = lib
    L, B, Hq, Hkv, d = 512, 64, 2, 1, 64
    X = make_numpy(L, Hq, Hkv, d, seed=9)
    dev = {k: to_dev(v, torch) for k, v in X.items()}
    no_keys = torch.empty((0, Hkv, d), dtype=torch.bfloat16, device="cuda")
    # the local partial needs whole corrupted blocks (their keys are read)
    with pytest.raises(m.BdlmError) as e:
        m.bdlm_attn_fwd_rank(dev["Qc"][:128], no_keys, no_keys, dev["Qn"][32:160], dev["Kn"][32:160],
                             dev["Vn"][32:160], L, B, 0, 0, True, (0, 128), (32, 160))
    assert e.value.status == 2
    # tensors must hold exactly the call's rows
    with pytest.raises(ValueError):
        m.bdlm_attn_fwd_rank(dev["Qc"][:100], no_keys, no_keys, dev["Qn"][:128], dev["Kn"][:128], dev["Vn"][:128],
                             L, B, 0, 0, True, (0, 128), (0, 128))


def _nccl_single_rank(port, L, B, Hq, Hkv, d, gathered, out):
    """Child process: one NCCL rank runs the CSBP driver with TorchComm and
    KernelCompute and reports its largest relative error against the fp64
    oracle."""
    import os
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    os.environ.setdefault("NCCL_NVLS_ENABLE", "0")
    import numpy as np_
    import torch as t_
    import torch.distributed as dist
    import oracle.bdlm_oracle as orc_
    import structured_mask_attention_gb300 as m
    from structured_mask_attention_gb300 import csbp as csbp_
    from structured_mask_attention_gb300.inputs import make_numpy as mk
    m.load_library()
    t_.cuda.set_device(0)
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{port}", rank=0, world_size=1)
    try:
        X = mk(L, Hq, Hkv, d, seed=21)
        dev = {k: t_.from_numpy(v).to("cuda").to(t_.bfloat16).contiguous() for k, v in X.items()}
        X64 = {k: dev[k].float().cpu().numpy().astype(np_.float64) for k in dev}
        sc = 1.0 / np_.sqrt(d)
        plan = csbp_.CSBPPlan.build(L, B, 1)
        comm = csbp_.TorchComm()
        comp = csbp_.KernelCompute(m, plan, 0, dict(dev), sc)
        shards = csbp_.gather_clean_kv(comm, dev["Kc"], dev["Vc"])
        o = csbp_.forward(plan, comm, comp, shards, gathered)
        (dqc, dqn), (dkc, dvc), (dkn, dvn) = csbp_.backward(plan, comm, comp, shards, o, (dev["dOc"], dev["dOn"]),
                                                           gathered)
        t_.cuda.synchronize()
        names = ("Qc", "Kc", "Vc", "Qn", "Kn", "Vn")
        rf = orc_.fwd_blockwise(*[X64[k] for k in names], B, sc)
        rg = orc_.bwd_blockwise(*[X64[k] for k in names], X64["dOc"], X64["dOn"], B, sc)
        err = 0.0
        for got, ref in ((o[0], rf[0]), (o[1], rf[1]), (dqc, rg[0]), (dkc, rg[1]), (dvc, rg[2]), (dqn, rg[3]),
                         (dkn, rg[4]), (dvn, rg[5])):
            g = got.float().cpu().numpy()
            err = max(err, float(np_.abs(g - ref).max() / np_.abs(ref).max()))
        lerr = max(float(np_.abs(o[2].cpu().numpy() - rf[2]).max()), float(np_.abs(o[3].cpu().numpy() - rf[3]).max()))
        out.put(("ok", err, lerr))
    except BaseException as e:  # reported to the parent
        out.put(("error", repr(e), 0.0))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("gathered", [False, True])
def test_csbp_driver_nccl_single_rank(gathered):
    """The transport on NCCL with CUDA tensors: a one-rank NCCL group runs the
    CSBP driver end to end (all-gather and reduce through torch.distributed)
    on the kernels; outputs and gradients match the fp64 oracle."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import socket
    import torch.multiprocessing as mp
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    p = ctx.Process(target=_nccl_single_rank, args=(port, 512, 64, 2, 1, 64, gathered, q))
    p.start()
    status, err, lerr = q.get(timeout=600)
    p.join(timeout=120)
    assert status == "ok", err
    assert p.exitcode == 0
    assert err <= 2e-2, err
    assert lerr <= 1e-3, lerr


def test_bench_csbp_mode_one_rank(lib):
    """bench.py --csbp at one rank (no process group): the multi-rank CSBP
    step runs end to end through the driver and reports a sane line."""
    import argparse
    import bench
    args = argparse.Namespace(workload="profile-16k", steps=1, warmup=3)
    line = bench.run_csbp(args, 0, 1, 0)
    assert line["config"]["parallelism"] == "csbp1" and line["scaling"] == "strong"
    assert line["ms_per_step"] > 0 and line["value"] > 0 and line["peak_gib_per_rank"] > 0
