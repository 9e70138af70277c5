"""Helpers shared by the GPU parity tests: host inputs -> device tensors, the
oracle on the same values, and the tolerance checks.

Tolerances (written here once, used by every parity test):
  * O, dQ, dK, dV: max |gpu - oracle| <= 2e-2 * max |oracle|, per tensor;
  * LSE: max |gpu - oracle| <= 1e-3 (natural-log units), on rows with a
    visible key; rows with none must be -inf on both sides.
"""
from __future__ import annotations

import numpy as np

REL_TOL = 2e-2
LSE_TOL = 1e-3


def to_dev(x, torch, device="cuda"):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(device=device, dtype=torch.bfloat16)


def to_np(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def check_rel(name, got, ref, tol=REL_TOL):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{name}: non-finite values"
    scale = np.abs(ref).max()
    err = np.abs(got - ref).max() if ref.size else 0.0
    print(f"  {name}: max|err| / max|ref| = {err / max(scale, 1e-30):.3e}")
    assert err <= tol * max(scale, 1e-30), f"{name}: max err {err:.3e} > {tol} * {scale:.3e}"
    return err / max(scale, 1e-30)


def check_lse(name, got, ref, tol=LSE_TOL):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    fin = np.isfinite(ref)
    assert (np.isneginf(got) == ~fin).all(), f"{name}: -inf pattern differs"
    err = np.abs(got[fin] - ref[fin]).max() if fin.any() else 0.0
    print(f"  {name}: max|err| = {err:.3e}")
    assert err <= tol, f"{name}: max err {err:.3e} > {tol}"
    return err
