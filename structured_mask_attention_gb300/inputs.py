"""Seeded synthetic inputs for two-stream BDLM attention.

This module only draws random numbers and rounds them to bf16; it holds no
attention arithmetic.  It is the one piece of code that both the CUDA path's
callers (tests, bench) and the fp64 oracle's callers use, so that both sides
see the same values.

Workloads (all batch 1, clean length L plus a corrupted copy of length L,
block size B, GQA with Hq query heads and Hkv key/value heads, head dim d):

* ``tiny``        L=256,    B=32,  Hq=2,  Hkv=2, d=64   (fp32 N(0,1), numpy PCG64)
* ``gqa-8k``      L=8192,   B=128, Hq=32, Hkv=8, d=128
* ``gqa-32k``     L=32768,  B=256, Hq=40, Hkv=8, d=128  (+ LogNormal(0,0.5) Q/K rows)
* ``long-128k``   L=131072, B=512, Hq=16, Hkv=8, d=128
* ``sharded-256k`` L=262144, B in {128,256,512,1024}, Hq=8, Hkv=4, d=128, P=8
* ``profile-16k`` L=16384, B=512, Hq=16, Hkv=8, d=128 (profiler captures)
* ``packed-128k`` a packed batch of T=131072 tokens per stream, B=512, Hq=16,
  Hkv=8, d=128, sequence lengths from ``packed_lengths`` (log-uniform between
  2048 and 32768, multiples of B)
* ``batch-64x2k`` a plain batch of 64 sequences of 2048 tokens, B=128, Hq=32,
  Hkv=8, d=128

Draw order: Qc, Kc, Vc, Qn, Kn, Vn, dOc, dOn (each N(0,1) in fp32), then, when
requested, one LogNormal(0, sigma) factor per token for each of Qc, Kc, Qn, Kn,
broadcast over heads and head dim.  Values are rounded to bf16 (round to
nearest, ties to even) after scaling.
"""
from __future__ import annotations

import numpy as np

WORKLOADS = {
    "tiny": dict(L=256, B=32, Hq=2, Hkv=2, d=64),
    "gqa-8k": dict(L=8192, B=128, Hq=32, Hkv=8, d=128),
    "gqa-32k": dict(L=32768, B=256, Hq=40, Hkv=8, d=128),
    "long-128k": dict(L=131072, B=512, Hq=16, Hkv=8, d=128),
    "sharded-256k": dict(L=262144, B=1024, Hq=8, Hkv=4, d=128, P=8),
    # same head layout and block size as long-128k at 1/8 of the length, for
    # profiler captures (inputs ~0.4 GB, still larger than L2)
    "profile-16k": dict(L=16384, B=512, Hq=16, Hkv=8, d=128),
    # packed batches (per-sequence lengths; T = total tokens per stream)
    "packed-128k": dict(T=131072, B=512, Hq=16, Hkv=8, d=128, lo=2048, hi=32768, seed=0),
    "batch-64x2k": dict(T=131072, B=128, Hq=32, Hkv=8, d=128, lo=2048, hi=2048, seed=0),
}
SHARDED_BLOCK_SIZES = (128, 256, 512, 1024)

NAMES = ("Qc", "Kc", "Vc", "Qn", "Kn", "Vn", "dOc", "dOn")


def packed_lengths(T, B, lo, hi, seed=0):
    """Sequence lengths of a packed batch of T tokens: drawn log-uniformly in
    [lo, hi] from numpy's PCG64(seed), rounded down to multiples of B (at
    least B), until the total would pass T; the last sequence takes the rest.
    T, lo and hi are multiples of B."""
    assert T % B == 0 and lo % B == 0 and hi % B == 0 and 0 < lo <= hi
    rng = np.random.Generator(np.random.PCG64(seed))
    lens, left = [], T
    while left > 0:
        x = int(np.exp(rng.uniform(np.log(lo), np.log(hi))) // B * B) if hi > lo else lo
        x = min(max(x, B), left)
        lens.append(x)
        left -= x
    return lens


def workload_lengths(name):
    """Sequence lengths of a packed workload of ``WORKLOADS``."""
    w = WORKLOADS[name]
    return packed_lengths(w["T"], w["B"], w["lo"], w["hi"], w["seed"])


def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 value (ties to even), returned
    as float32.  Inputs are finite."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> 16) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) & np.uint32(0xFFFF0000)).view(np.float32)


def _shapes(L, Hq, Hkv, d):
    return {"Qc": (L, Hq, d), "Kc": (L, Hkv, d), "Vc": (L, Hkv, d),
            "Qn": (L, Hq, d), "Kn": (L, Hkv, d), "Vn": (L, Hkv, d),
            "dOc": (L, Hq, d), "dOn": (L, Hq, d)}


def make_numpy(L, Hq, Hkv, d, seed=0, lognormal_sigma=0.0):
    """Host inputs from numpy's PCG64(seed): dict of float32 arrays holding
    bf16-representable values, shapes [L, H, d]."""
    rng = np.random.Generator(np.random.PCG64(seed))
    shp = _shapes(L, Hq, Hkv, d)
    raw = {n: rng.standard_normal(shp[n], dtype=np.float32) for n in NAMES}
    if lognormal_sigma:
        for n in ("Qc", "Kc", "Qn", "Kn"):
            f = rng.lognormal(0.0, lognormal_sigma, size=L).astype(np.float32)
            raw[n] = raw[n] * f[:, None, None]
    return {n: bf16_round(raw[n]) for n in NAMES}


def make_torch(L, Hq, Hkv, d, seed=0, lognormal_sigma=0.0, device="cuda"):
    """Device inputs from torch's generator on ``device`` seeded with ``seed``:
    dict of bf16 tensors [L, H, d].  Used for sizes where a host draw would be
    slow; same draw order and rounding rule as ``make_numpy`` (the streams
    differ from numpy's)."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    shp = _shapes(L, Hq, Hkv, d)
    out = {}
    raw = {n: torch.randn(shp[n], generator=g, device=device, dtype=torch.float32) for n in NAMES}
    if lognormal_sigma:
        for n in ("Qc", "Kc", "Qn", "Kn"):
            f = torch.empty(L, device=device, dtype=torch.float32).log_normal_(0.0, lognormal_sigma, generator=g)
            raw[n] = raw[n] * f[:, None, None]
    for n in NAMES:
        out[n] = raw[n].to(torch.bfloat16)
        del raw[n]
    return out
