"""The worker-process form of the oracle (tests/oracle_pool.py) gives the
same numbers as calling the oracle directly: the forward, the whole
backward, and a backward restricted to one clean key block."""
from __future__ import annotations

import math

import numpy as np

import oracle.bdlm_oracle as orc
from structured_mask_attention_gb300.inputs import make_numpy
from tests import oracle_pool


def test_pool_matches_direct_oracle():
    L, B, Hq, Hkv, d = 384, 32, 2, 1, 64
    X = {k: v.astype(np.float64) for k, v in make_numpy(L, Hq, Hkv, d, seed=7).items()}
    sc = 1.0 / math.sqrt(d)
    names = ("Qc", "Kc", "Vc", "Qn", "Kn", "Vn")
    fwd = oracle_pool.forward(X, B, sc, nproc=3)
    ref = orc.fwd_blockwise(*[X[k] for k in names], B, sc)
    for a, b in zip(fwd, ref):
        np.testing.assert_array_equal(a, b)
    D = (oracle_pool.preprocess(fwd[0], X["dOc"]), oracle_pool.preprocess(fwd[1], X["dOn"]))
    stats = (fwd[2], fwd[3], D[0], D[1])
    g = oracle_pool.backward(X, stats, B, sc, nproc=3)
    gref = orc.bwd_blockwise(*[X[k] for k in names], X["dOc"], X["dOn"], B, sc)
    for a, b in zip(g, gref):
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-12 * max(1.0, np.abs(b).max()))
    # keys of clean block 3 only: its dK / dV rows equal the full gradient's
    j = 3
    gj = oracle_pool.backward(X, stats, B, sc, kv_begin=j * B, kv_end=(j + 1) * B, include_local=False, nproc=2)
    for a, b in ((gj[1], gref[1]), (gj[2], gref[2])):
        np.testing.assert_allclose(a[j * B:(j + 1) * B], b[j * B:(j + 1) * B], rtol=0,
                                   atol=1e-12 * max(1.0, np.abs(b).max()))
        assert not a[:j * B].any() and not a[(j + 1) * B:].any()
