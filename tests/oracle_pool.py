"""The fp64 oracle over many row blocks at once, in worker processes.

Test infrastructure: full-size parity checks compare whole KV-head groups
against ``oracle.bdlm_oracle``, whose blockwise functions take the row blocks
to compute (``blocks=``).  Row blocks are independent for the forward (each
row's O and LSE) and for dQ; dK and dV are sums over row blocks.  This module
splits the blocks over worker processes started with ``spawn`` (safe after
CUDA was initialised in the parent), calls the oracle unchanged in each, and
puts the rows back together (dK / dV: summed over the workers in fp64).
Inputs reach the workers as ``.npy`` files they map read-only.  Nothing here
does attention arithmetic of its own.
"""
from __future__ import annotations

import multiprocessing as mp
import os
import shutil
import tempfile
from contextlib import contextmanager

import numpy as np

FWD_IN = ("Qc", "Kc", "Vc", "Qn", "Kn", "Vn")

_X = None  # worker-side inputs (memory-mapped)


def _init(path, names):
    global _X
    _X = {k: np.load(os.path.join(path, k + ".npy"), mmap_mode="r") for k in names}


def _fwd_task(args):
    import oracle.bdlm_oracle as orc
    B, sc, blocks = args
    Oc, On, LSEc, LSEn = orc.fwd_partial(*[_X[k] for k in FWD_IN], B, sc, blocks=blocks)
    out = {}
    for b in blocks:
        r = slice(b * B, (b + 1) * B)
        out[b] = (Oc[r].copy(), On[r].copy(), LSEc[:, r].copy(), LSEn[:, r].copy())
    return out


def _bwd_task(args):
    import oracle.bdlm_oracle as orc
    B, sc, kv_begin, kv_end, include_local, blocks = args
    g = orc.bwd_partial(*[_X[k] for k in FWD_IN], _X["dOc"], _X["dOn"], _X["LSEc"], _X["LSEn"], _X["Dc"],
                        _X["Dn"], B, sc, kv_begin, kv_end, include_local, blocks=blocks)
    dQc, dKc, dVc, dQn, dKn, dVn = g
    rows = {b: (dQc[b * B:(b + 1) * B].copy(), dQn[b * B:(b + 1) * B].copy()) for b in blocks}
    # key rows this call can touch: the clean range, and every corrupted row
    # when the local block is included
    kc = (dKc[kv_begin:kv_end].copy(), dVc[kv_begin:kv_end].copy())
    kn = (dKn.copy(), dVn.copy()) if include_local else None
    return rows, kc, kn


def _workers(per_worker_bytes, nproc=None):
    """Worker count: the host's cores, fewer if their working sets would not
    fit in 60 % of the memory available now."""
    n = nproc or max(1, os.cpu_count() or 1)
    try:
        avail = os.sysconf("SC_AVPHYS_PAGES") * os.sysconf("SC_PAGE_SIZE")
        n = max(1, min(n, int(0.6 * avail // max(per_worker_bytes, 1))))
    except (ValueError, OSError, AttributeError):
        pass
    return n


@contextmanager
def _pool(arrays, nproc=None):
    """A spawn pool of `nproc` workers that map `arrays` (name -> ndarray)
    read-only; BLAS inside each worker is single-threaded."""
    need = sum(int(np.asarray(v).size) * 8 for v in arrays.values()) + (64 << 20)
    base = None  # the default temporary directory, unless shared memory has room
    if os.path.isdir("/dev/shm") and os.access("/dev/shm", os.W_OK) and shutil.disk_usage("/dev/shm").free > 2 * need:
        base = "/dev/shm"
    tmp = tempfile.mkdtemp(prefix="bdlm_oracle_", dir=base)
    saved = {}
    try:
        for k, v in arrays.items():
            np.save(os.path.join(tmp, k + ".npy"), np.ascontiguousarray(v, dtype=np.float64))
        for v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
            saved[v] = os.environ.get(v)
            os.environ[v] = "1"
        n = nproc or max(1, os.cpu_count() or 1)
        ctx = mp.get_context("spawn")
        with ctx.Pool(n, initializer=_init, initargs=(tmp, tuple(arrays))) as pool:
            for v, old in saved.items():
                if old is None:
                    os.environ.pop(v, None)
                else:
                    os.environ[v] = old
            saved = {}
            yield pool, n
    finally:
        for v, old in saved.items():
            if old is None:
                os.environ.pop(v, None)
            else:
                os.environ[v] = old
        shutil.rmtree(tmp, ignore_errors=True)


def _chunks(N, parts):
    """Row blocks dealt round-robin from the last one (the longest rows)
    into `parts` lists, so the lists carry similar work."""
    order = list(range(N - 1, -1, -1))
    return [order[i::parts] for i in range(parts) if order[i::parts]]


def forward(X, B, sc, nproc=None):
    """``oracle.fwd_blockwise`` of the inputs in X (fp64, one KV-head group or
    any heads), computed block by block in worker processes.
    Returns (Oc, On, LSEc, LSEn)."""
    L, Hq, _ = X["Qc"].shape
    dv = X["Vc"].shape[2]
    N = L // B
    Oc = np.zeros((L, Hq, dv)); On = np.zeros((L, Hq, dv))
    LSEc = np.zeros((Hq, L)); LSEn = np.zeros((Hq, L))
    # per worker: its own full-length O of both streams, and a few
    # B x (L + B) score-sized temporaries
    nproc = _workers(2 * L * Hq * dv * 8 + 4 * B * (L + B) * 8, nproc)
    with _pool({k: X[k] for k in FWD_IN}, nproc) as (pool, n):
        for res in pool.imap_unordered(_fwd_task, [(B, sc, ch) for ch in _chunks(N, 4 * n)]):
            for b, (oc, on, lc, ln) in res.items():
                r = slice(b * B, (b + 1) * B)
                Oc[r], On[r], LSEc[:, r], LSEn[:, r] = oc, on, lc, ln
    return Oc, On, LSEc, LSEn


def backward(X, stats, B, sc, kv_begin=0, kv_end=None, include_local=True, nproc=None):
    """``oracle.bwd_partial`` (gradient contributions of the keys in clean
    [kv_begin, kv_end) plus, optionally, the corrupted own blocks, given the
    full-row statistics ``stats`` = (LSEc, LSEn, Dc, Dn)), row blocks in worker
    processes.  With the defaults and the full forward's statistics this is
    the whole backward.  Returns (dQc, dKc, dVc, dQn, dKn, dVn)."""
    L, Hq, d = X["Qc"].shape
    Hkv = X["Kc"].shape[1]
    dv = X["Vc"].shape[2]
    kv_end = L if kv_end is None else kv_end
    N = L // B
    LSEc, LSEn, Dc, Dn = stats
    arrays = {k: X[k] for k in FWD_IN + ("dOc", "dOn")}
    arrays.update(LSEc=LSEc, LSEn=LSEn, Dc=Dc, Dn=Dn)
    dQc = np.zeros((L, Hq, d)); dQn = np.zeros((L, Hq, d))
    dKc = np.zeros((L, Hkv, d)); dVc = np.zeros((L, Hkv, dv))
    dKn = np.zeros((L, Hkv, d)); dVn = np.zeros((L, Hkv, dv))
    # per worker: its own full-length gradients, and a few score-sized temporaries
    span = (kv_end - kv_begin) + (B if include_local else 0)
    nproc = _workers((2 * L * Hq * d + 4 * L * Hkv * d) * 8 + 6 * B * span * 8, nproc)
    with _pool(arrays, nproc) as (pool, n):
        tasks = [(B, sc, kv_begin, kv_end, include_local, ch) for ch in _chunks(N, 2 * n)]
        for rows, kc, kn in pool.imap_unordered(_bwd_task, tasks):
            for b, (qc, qn) in rows.items():
                dQc[b * B:(b + 1) * B] = qc
                dQn[b * B:(b + 1) * B] = qn
            dKc[kv_begin:kv_end] += kc[0]
            dVc[kv_begin:kv_end] += kc[1]
            if kn is not None:
                dKn += kn[0]
                dVn += kn[1]
    return dQc, dKc, dVc, dQn, dKn, dVn


def preprocess(O, dO):
    """D = rowsum(dO * O) through the oracle's own function."""
    import oracle.bdlm_oracle as orc
    return orc.bwd_preprocess(O, dO)
