#!/usr/bin/env python
"""Benchmark of two-stream BDLM attention (forward + backward) on GB300.

One step = the whole hot path over one batch: the two-stream forward (O, LSE)
and the backward (row statistic D, dK/dV pass, dQ pass) of the long-context
workload L = 131072 clean + 131072 corrupted tokens, B = 512, 16 query heads,
8 KV heads, head dim 128, bf16 inputs ~ N(0, 1), through the library's C ABI.

Metric: useful (mask-visible) fwd+bwd TFLOP/s, 14 d L (L + B) Hq FLOP per
step (the backward counted as 2.5 forwards), plus tokens/s (2L per step) and
the fraction of the bf16 tensor peak.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference]

Under torchrun each rank runs its own replica of the workload on its GPU (no
data-path collective); rank 0 prints one JSON line.  ``--impl reference``
times the fp64 CPU oracle on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "long-128k"
METRIC = "useful fwd+bwd TFLOP/s & tokens/s at 1 GB300; % of bf16 tensor peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def job_time_ms(ms_local, world, device):
    """The job's time for a step: the maximum over ranks of each rank's own
    CUDA-event time (ranks are replicas, so the slowest one ends the step)."""
    if world <= 1:
        return ms_local
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms_local], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank, world, ms):
    """Whole-job rate: the units all ranks processed divided by the job's time."""
    return world * units_per_rank / (ms * 1e-3)


def useful_flops(L, B, Hq, d):
    return 14.0 * d * L * (L + B) * Hq


def strict_flops(L, B, Hq, d):
    return 12.0 * d * L * (L + B) * Hq


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            d = json.load(fh)
        return d, "measured"
    return FALLBACK_PEAKS, "fallback"


def peak_value(peaks, key):
    """Reads a peak from MEASURED_PEAKS.json, tolerating nesting and units."""
    if key in peaks and isinstance(peaks[key], (int, float)):
        return float(peaks[key])
    for v in peaks.values():
        if isinstance(v, dict) and key in v and isinstance(v[key], (int, float)):
            return float(v[key])
    return FALLBACK_PEAKS[key]


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200",
                 "-i", str(gpu_index)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons, power = [], [], set(), []
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
                power.append(float(f[3]))
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "power_w_median": statistics.median(power) if power else None,
                "samples": len(sm)}


# ------------------------------------------------------------------ host memory placement
def gpu_local_cpus(dev):
    """The CPUs of the GPU's own NUMA node, from sysfs (None if unknown).
    Pinned host buffers allocated by a thread on one of these CPUs live in
    the memory next to the GPU; on a node with more than one CPU socket,
    buffers on the other socket's memory are read by the GPU's copy engines
    at a fraction of the link's rate."""
    try:
        import torch
        p = torch.cuda.get_device_properties(dev)
        path = "/sys/bus/pci/devices/%04x:%02x:%02x.0/local_cpulist" % (p.pci_domain_id, p.pci_bus_id,
                                                                        p.pci_device_id)
        with open(path) as fh:
            txt = fh.read().strip()
        cpus = set()
        for part in txt.split(","):
            a, _, b = part.partition("-")
            cpus.update(range(int(a), int(b or a) + 1))
        cpus &= os.sched_getaffinity(0)
        return cpus or None
    except (AttributeError, OSError, ValueError, RuntimeError):
        return None


# ------------------------------------------------------------------ oracle sample
def oracle_sample(L, B, Hq, Hkv, d, budget_s, seed=0):
    """Times the fp64 oracle on the last blocks of one query head of the
    workload (forward, row statistic, backward), until ~budget_s seconds.
    Returns (useful FLOP, seconds, blocks done, threads)."""
    import numpy as np

    import oracle.bdlm_oracle as orc
    from structured_mask_attention_gb300.inputs import make_numpy

    X = make_numpy(L, 1, 1, d, seed=seed)  # one query head, its KV head
    X = {k: v.astype(np.float64) for k, v in X.items()}
    names = ("Qc", "Kc", "Vc", "Qn", "Kn", "Vn")
    sc = 1.0 / math.sqrt(d)
    N = L // B
    flops = 0.0
    t0 = time.perf_counter()
    done = 0
    for b in range(N - 1, -1, -1):
        Oc, On, LSEc, LSEn = orc.fwd_partial(*[X[k] for k in names], B, sc, heads=[0], blocks=[b])
        Dc, Dn = orc.bwd_preprocess(Oc, X["dOc"]), orc.bwd_preprocess(On, X["dOn"])
        orc.bwd_partial(*[X[k] for k in names], X["dOc"], X["dOn"], LSEc, LSEn, Dc, Dn, B, sc, heads=[0],
                        blocks=[b])
        flops += 14.0 * d * 2 * B * (b + 1) * B
        done += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    return flops, dt, done, blas_threads()


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    for v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(v):
            return int(os.environ[v])
    return os.cpu_count()


# ------------------------------------------------------------------ traffic
def sources_digest(paths):
    """First 16 hex digits of the SHA-256 of the concatenated files."""
    h = hashlib.sha256()
    for rel in paths:
        with open(os.path.join(ROOT, rel), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def committed_traffic(kernel, workload):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources and on this workload (else None)."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as fh:
        d = json.load(fh)
    ent = d.get(kernel)
    if not ent:
        return None
    srcs = ent.get("sources", [])
    if not srcs or not all(os.path.exists(os.path.join(ROOT, s)) for s in srcs):
        return None
    if sources_digest(srcs) != ent.get("sources_sha256_16"):
        return None
    if ent.get("workload") != workload:
        return None
    return ent.get("dram_bytes_per_launch_full")


# ------------------------------------------------------------------ native arm
def run_native(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    import structured_mask_attention_gb300 as m
    from structured_mask_attention_gb300.inputs import WORKLOADS, make_torch

    m.load_library()
    w = WORKLOADS[args.workload]
    L, B, Hq, Hkv, d = w["L"], w["B"], w["Hq"], w["Hkv"], w["d"]
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    X = make_torch(L, Hq, Hkv, d, seed=rank, device=dev)
    names = ("Qc", "Kc", "Vc", "Qn", "Kn", "Vn")
    ins = [X[k] for k in names]
    sc = 1.0 / math.sqrt(d)
    e = lambda H, dt=torch.bfloat16: torch.empty((L, H, d), dtype=dt, device=dev)
    fout = (e(Hq), e(Hq), torch.empty((Hq, L), dtype=torch.float32, device=dev),
            torch.empty((Hq, L), dtype=torch.float32, device=dev))
    gout = (e(Hq), e(Hkv), e(Hkv), e(Hq), e(Hkv), e(Hkv))
    ws_f = torch.empty(m.bdlm_workspace_size(m.OP_FWD, L, B, Hq, Hkv, d), dtype=torch.uint8, device=dev)
    ws_b = torch.empty(m.bdlm_workspace_size(m.OP_BWD, L, B, Hq, Hkv, d), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        Oc, On, LSEc, LSEn = m.bdlm_attn_fwd(*ins, B, sc, out=fout, workspace=ws_f)
        m.bdlm_attn_bwd(*ins, Oc, On, X["dOc"], X["dOn"], LSEc, LSEn, B, sc, out=gout, workspace=ws_b)

    def barrier():
        if world > 1:
            dist.barrier()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    m.bdlm_sync_status(ws_f)
    m.bdlm_sync_status(ws_b)

    m.bdlm_timing_report(reset=True)
    m.bdlm_timing_enable(True)
    clocks = ClockSampler(local_rank)
    time.sleep(0.5)
    barrier()
    torch.cuda.synchronize()
    n0 = m.bdlm_kernel_launches()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize()
    barrier()
    launches = m.bdlm_kernel_launches() - n0
    clk = clocks.stop()
    m.bdlm_timing_enable(False)
    ktimes = m.bdlm_timing_report(reset=True)
    ms = job_time_ms(ev0.elapsed_time(ev1), world, dev)
    m.bdlm_sync_status(ws_f)
    m.bdlm_sync_status(ws_b)
    ms_step = ms / args.steps

    # ---- end to end through the public API with host buffers
    # Every step copies its inputs from pinned host memory to the device and
    # reads all of its results (O, LSE, dQ, dK, dV of both streams) back.
    # Steps are pipelined the way a training loop feeds an accelerator, with
    # two device buffer sets and two copy streams: step i+1's Q, K, V go up
    # while step i computes, its dO while its own forward runs; step i's O and
    # LSE come down while its backward runs, its gradients while step i+1
    # computes.  The timed region runs from the first upload to the last
    # download.
    e2e = None
    if not args.no_e2e:
        pin = lambda t: torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
        keys = (*names, "dOc", "dOn")
        # allocate the pinned buffers from a CPU next to the GPU, so that their
        # pages sit in the GPU's NUMA node (the affinity is restored afterwards)
        local_cpus = gpu_local_cpus(dev)
        saved_cpus = os.sched_getaffinity(0)
        if local_cpus:
            os.sched_setaffinity(0, local_cpus)
        try:
            h_in = {k: pin(X[k]) for k in keys}
            h_out = [pin(t) for t in (*fout, *gout)]
        finally:
            os.sched_setaffinity(0, saved_cpus)
        for k in h_in:
            h_in[k].copy_(X[k])
        h2d = sum(t.numel() * t.element_size() for t in h_in.values())
        d2h = sum(t.numel() * t.element_size() for t in h_out)
        sets = []
        for _ in range(2):
            sets.append(({k: torch.empty_like(X[k]) for k in keys},
                         tuple(torch.empty_like(t) for t in fout), tuple(torch.empty_like(t) for t in gout)))
        s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        ev = lambda: torch.cuda.Event()
        # per buffer set: Q/K/V up, dO up, forward done, step done, O/LSE down, gradients down
        qkv_in, do_in, fwd_done, comp_done = [ev(), ev()], [ev(), ev()], [ev(), ev()], [ev(), ev()]
        fo_out, go_out = [ev(), ev()], [ev(), ev()]
        h_fo, h_go = h_out[:len(fout)], h_out[len(fout):]

        def e2e_run(nsteps, spans=None):
            for i in range(nsteps):
                si = i & 1
                dX, fo, go = sets[si]
                if i >= 2:
                    s_in.wait_event(comp_done[si])  # step i-2 no longer reads this set's inputs
                with torch.cuda.stream(s_in):
                    for k in names:
                        dX[k].copy_(h_in[k], non_blocking=True)
                    qkv_in[si].record(s_in)
                    for k in ("dOc", "dOn"):  # needed by the backward only
                        dX[k].copy_(h_in[k], non_blocking=True)
                    do_in[si].record(s_in)
                stream.wait_event(qkv_in[si])
                if i >= 2:
                    stream.wait_event(fo_out[si])  # step i-2's O / LSE are on the host
                if spans is not None:
                    spans.append((torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)))
                    spans[-1][0].record(stream)
                Oc, On, LSEc, LSEn = m.bdlm_attn_fwd(*[dX[k] for k in names], B, sc, out=fo, workspace=ws_f)
                fwd_done[si].record(stream)
                stream.wait_event(do_in[si])
                if i >= 2:
                    stream.wait_event(go_out[si])  # step i-2's gradients are on the host
                m.bdlm_attn_bwd(*[dX[k] for k in names], Oc, On, dX["dOc"], dX["dOn"], LSEc, LSEn, B, sc,
                                out=go, workspace=ws_b)
                if spans is not None:
                    spans[-1][1].record(stream)
                comp_done[si].record(stream)
                # O and LSE go down while the backward runs, the gradients after it
                s_out.wait_event(fwd_done[si])
                with torch.cuda.stream(s_out):
                    for hd, dv in zip(h_fo, fo):
                        hd.copy_(dv, non_blocking=True)
                    fo_out[si].record(s_out)
                s_out.wait_event(comp_done[si])
                with torch.cuda.stream(s_out):
                    for hd, dv in zip(h_go, go):
                        hd.copy_(dv, non_blocking=True)
                    go_out[si].record(s_out)
            stream.wait_stream(s_out)

        # link bandwidth, for the record (one upload, one download, alone)
        t0, t1, t2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        dX0 = sets[0][0]
        t0.record(stream)
        for k in keys:
            dX0[k].copy_(h_in[k], non_blocking=True)
        t1.record(stream)
        for hd, dv in zip(h_out, (*sets[0][1], *sets[0][2])):
            hd.copy_(dv, non_blocking=True)
        t2.record(stream)
        torch.cuda.synchronize()
        h2d_gbs = h2d / (t0.elapsed_time(t1) * 1e-3) / 1e9
        d2h_gbs = d2h / (t1.elapsed_time(t2) * 1e-3) / 1e9

        e2e_run(2)
        torch.cuda.synchronize()
        k2 = max(3, args.steps)
        barrier()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        spans = []
        e2e_clocks = ClockSampler(local_rank)
        a.record(stream)
        s_in.wait_stream(stream)
        e2e_run(k2, spans)
        b.record(stream)
        torch.cuda.synchronize()
        e2e_clk = e2e_clocks.stop()
        compute_ms = statistics.median(x.elapsed_time(y) for x, y in spans)
        barrier()
        ems = job_time_ms(a.elapsed_time(b) / k2, world, dev)
        e2e = {"value": round(job_rate(useful_flops(L, B, Hq, d), world, ems) / 1e12, 3), "unit": "TFLOP/s",
               "ms_per_step": round(ems, 3), "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "tokens_per_s": round(job_rate(2 * L, world, ems), 1), "steps": k2,
               "pipelined": ("two buffer sets; a step's Q/K/V go up during the previous step, its dO during "
                             "its forward, its O/LSE come down during its backward, its gradients during "
                             "the next step"),
               "h2d_gbs_alone": round(h2d_gbs, 1), "d2h_gbs_alone": round(d2h_gbs, 1),
               # the device's own time per step inside this loop (median), and the
               # clocks while it ran: what the copies leave to the computation
               "compute_ms_per_step": round(compute_ms, 3), "clocks": e2e_clk,
               "host_buffers": ("pinned, allocated from the GPU's NUMA-node CPUs (%d CPUs)" % len(local_cpus)
                                if local_cpus else "pinned (the GPU's NUMA node is not known)")}
        del sets, h_in, h_out

    # ---- roofline of the dominant kernel
    peaks, peak_src = load_peaks()
    peak_tf = peak_value(peaks, "bf16_tflops_sustained")
    pairs = L * (L + B) * Hq
    alg = {"bdlm_fwd_tc": 4.0 * d * pairs, "bdlm_bwd_dkv": 8.0 * d * pairs, "bdlm_bwd_dq": 6.0 * d * pairs}
    per_kernel = {}
    for k, (cnt, tot) in ktimes.items():
        ms_k = tot / max(cnt, 1)
        e = {"launches": cnt, "ms_per_launch": round(ms_k, 4),
             "share": round(tot / max(sum(v[1] for v in ktimes.values()), 1e-9), 4)}
        if k in alg and ms_k > 0:
            # executed FLOP per launch (recomputed products included) against the sustained peak
            tf_k = alg[k] / (ms_k * 1e-3) / 1e12
            e.update({"tflops": round(tf_k, 1), "frac": round(tf_k / peak_tf, 4),
                      "traffic": committed_traffic(k, args.workload)})
        elif k == "bdlm_preprocess" and ms_k > 0:
            # one launch per stream: reads O and dO (bf16), writes D (fp32)
            e["gbs"] = round((2 * 2 * L * Hq * d + 4 * L * Hq) / (ms_k * 1e-3) / 1e9, 1)
        per_kernel[k] = e
    dom = max((k for k in ktimes if k in alg), key=lambda k: ktimes[k][1])
    dom_ms = ktimes[dom][1] / ktimes[dom][0]
    achieved = alg[dom] / (dom_ms * 1e-3) / 1e12
    roofline = {"kernel": dom, "bound": "tensor", "achieved": round(achieved, 2), "peak": peak_tf,
                "unit": "TFLOP/s", "frac": round(achieved / peak_tf, 4), "traffic": committed_traffic(dom, args.workload),
                "peak_source": f"{peak_src} bf16_tflops_sustained" + (" (of measured)" if peak_src == "measured"
                                                                      else " (of fallback)"),
                "algorithmic_flop_per_launch": alg[dom]}

    value = job_rate(useful_flops(L, B, Hq, d), world, ms_step) / 1e12
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1), bf16)",
        "config": {"workload": args.workload, "L": L, "B": B, "Hq": Hq, "Hkv": Hkv, "d": d, "batch": 1,
                   "tokens_per_step": 2 * L, "l2": "inputs larger than L2 (129 MB)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "tokens_per_s": round(job_rate(2 * L, world, ms_step), 1),
        "strict_tflops": round(job_rate(strict_flops(L, B, Hq, d), world, ms_step) / 1e12, 3),
        "pct_of_peak": round(100.0 * value / world / peak_tf, 2),
        "clocks": clk, "gpu_launches": int(launches), "kernels": per_kernel, "roofline": roofline,
        "e2e": e2e,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        flops, dt, blocks, thr = oracle_sample(L, B, Hq, Hkv, d, args.cpu_budget)
        line["cpu_baseline"] = {"value": round(flops / dt / 1e12, 6), "unit": "TFLOP/s", "cores": thr,
                                "kind": "oracle",
                                "sample": f"fp64 oracle fwd+bwd of the last {blocks} block(s) of one query head "
                                          f"of {args.workload} (both streams), {dt:.1f} s"}
    return line


class _OneRank:
    """The exchange of a single rank (no process group): its own shard."""
    rank, world = 0, 1

    def all_gather(self, x):
        return [x]

    def sum_to_owner(self, x, owner):
        return x


def run_csbp(args, rank, world, local_rank):
    """Multi-rank CSBP, strong scaling: one sequence of the workload split
    over the ranks by the balanced plan of
    structured_mask_attention_gb300.csbp (rank r: clean slice r, corrupted
    slice R - 1 - r), each rank computing its rows with the rank-local calls
    (gathered schedule), the clean K / V all-gathered and the clean dK / dV
    summed onto their owners through torch.distributed (NCCL).  The step
    time, exchange included, is the maximum over ranks of each rank's
    CUDA-event time; the rate counts the whole sequence's useful FLOP."""
    import torch
    import torch.distributed as dist

    import structured_mask_attention_gb300 as m
    from structured_mask_attention_gb300 import csbp
    from structured_mask_attention_gb300.inputs import WORKLOADS, make_torch

    m.load_library()
    w = WORKLOADS[args.workload]
    L, B, Hq, Hkv, d = w["L"], w["B"], w["Hq"], w["Hkv"], w["d"]
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    plan = csbp.CSBPPlan.build(L, B, world)
    rw = plan.rows(rank)
    # the same seeded sequence on every rank; each keeps only its own rows
    X = make_torch(L, Hq, Hkv, d, seed=0, device=dev)
    c, n = slice(rw.c0 * B, rw.c1 * B), slice(rw.n0 * B, rw.n1 * B)
    local = {k: X[k][c].clone() for k in ("Qc", "Kc", "Vc", "dOc")}
    local.update({k: X[k][n].clone() for k in ("Qn", "Kn", "Vn", "dOn")})
    del X
    torch.cuda.empty_cache()
    comm = csbp.TorchComm() if world > 1 else _OneRank()
    comp = csbp.KernelCompute(m, plan, rank, local, 1.0 / math.sqrt(d))

    def step():
        shards = csbp.gather_clean_kv(comm, local["Kc"], local["Vc"])
        o = csbp.forward(plan, comm, comp, shards, gathered=True)
        return csbp.backward(plan, comm, comp, shards, o, (local["dOc"], local["dOn"]), gathered=True)

    def barrier():
        if world > 1:
            dist.barrier()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    torch.cuda.reset_peak_memory_stats(dev)
    clocks = ClockSampler(local_rank)
    barrier()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize()
    barrier()
    clk = clocks.stop()
    ms = job_time_ms(ev0.elapsed_time(ev1), world, dev)
    peak = torch.tensor([torch.cuda.max_memory_allocated(dev) / 2 ** 30], dtype=torch.float64, device=dev)
    if world > 1:
        dist.all_reduce(peak, op=dist.ReduceOp.MAX)
    ms_step = ms / args.steps
    value = useful_flops(L, B, Hq, d) / (ms_step * 1e-3) / 1e12
    return {"metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_step, 3), "higher_is_better": True,
            "scaling": "strong", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1), bf16)",
            "config": {"workload": args.workload, "L": L, "B": B, "Hq": Hq, "Hkv": Hkv, "d": d,
                       "parallelism": "csbp%d" % world, "assignment": "mirror", "schedule": "gathered",
                       "exchange": "torch.distributed (NCCL)" if world > 1 else "none (one rank)"},
            "tokens_per_s": round(2 * L / (ms_step * 1e-3), 1),
            "peak_gib_per_rank": round(float(peak.item()), 3), "clocks": clk}


def per_rank_memory(L, Hq, Hkv, d, R):
    """Attention tensors one of R ranks holds for a fwd+bwd step (GiB), by
    the shapes alone: bf16 Q, O, dO and fp32 dQ per query head; bf16 K, V and
    fp32 dK, dV per KV head.  Pure BP: every rank processes the whole clean
    sequence (replicated) plus its L / R corrupted tokens.  CSBP: its clean
    shard and its corrupted blocks (2 L / R tokens), plus the clean K / V of
    the other shards while they are exchanged (all-gathered: L tokens of bf16
    K and V; a ring holds two shards)."""
    q_tok = Hq * d * (2 + 2 + 2 + 4)
    kv_tok = Hkv * d * (2 + 2 + 4 + 4)
    bp = (L + L // R) * (q_tok + kv_tok)
    csbp = 2 * (L // R) * (q_tok + kv_tok)
    gathered = L * Hkv * d * 2 * 2
    ring = 2 * (L // R) * Hkv * d * 2 * 2
    g = lambda x: round(x / 2 ** 30, 2)
    return {"pure_bp": g(bp), "csbp_allgather": g(csbp + gathered), "csbp_ring": g(csbp + ring)}


def rank_program_memory(m, plan, rank, Hq, Hkv, d, schedule, dev):
    """Peak device memory (bytes above what was allocated before) of one
    rank's forward + backward through the rank-local calls: its own rows as
    inputs (its clean shard's Q, K, V, dO; its corrupted blocks' Q, K, V, dO),
    the clean K / V it receives (all shards at once when gathered; one shard
    at a time beside its own, as a two-shard ring holds them, per shard), the
    partials, merged outputs, statistics and fp32 gradients.  Input values
    are random: only the sizes matter here."""
    import torch
    L, B = plan.L, plan.B
    rw = plan.rows(rank)
    rc, rn = (rw.c0 * B, rw.c1 * B), (rw.n0 * B, rw.n1 * B)
    nc, nn = rc[1] - rc[0], rn[1] - rn[0]
    sc = 1.0 / math.sqrt(d)
    torch.cuda.synchronize(dev)
    base = torch.cuda.memory_allocated(dev)
    torch.cuda.reset_peak_memory_stats(dev)
    bf = lambda n, H: torch.randn((n, H, d), device=dev, dtype=torch.bfloat16)
    z32 = lambda n, H: torch.zeros((n, H, d), device=dev, dtype=torch.float32)
    Qc, dOc, Kc_own, Vc_own = bf(nc, Hq), bf(nc, Hq), bf(nc, Hkv), bf(nc, Hkv)
    Qn, dOn, Kn, Vn = bf(nn, Hq), bf(nn, Hq), bf(nn, Hkv), bf(nn, Hkv)
    nk = torch.empty((0, Hkv, d), dtype=torch.bfloat16, device=dev)
    if schedule == "gathered":
        Kg, Vg = bf(L, Hkv), bf(L, Hkv)  # after the all-gather
        parts = [m.bdlm_attn_fwd_rank(Qc, Kg, Vg, Qn, Kn, Vn, L, B, 0, L, True, rc, rn, sc)]
    else:  # a running merge, as csbp.forward does: two partials held at most
        parts = []
        for s_ in range(plan.R + 1):
            lo, hi = plan.shard_keys(s_) if s_ < plan.R else (0, 0)
            Ks, Vs = (bf(hi - lo, Hkv), bf(hi - lo, Hkv)) if hi > lo else (nk, nk)  # the shard in flight
            parts.append(m.bdlm_attn_fwd_rank(Qc, Ks, Vs, Qn, Kn, Vn, L, B, lo, hi, s_ == plan.R, rc, rn, sc))
            del Ks, Vs
            if len(parts) == 2:
                mc = m.bdlm_lse_merge([parts[0][0], parts[1][0]], [parts[0][2], parts[1][2]], o_dtype=torch.float32)
                mn = m.bdlm_lse_merge([parts[0][1], parts[1][1]], [parts[0][3], parts[1][3]], o_dtype=torch.float32)
                parts = [(mc[0], mn[0], mc[1], mn[1])]
                del mc, mn
    oc, lc = m.bdlm_lse_merge([p_[0] for p_ in parts], [p_[2] for p_ in parts], o_dtype=torch.float32)
    on, ln = m.bdlm_lse_merge([p_[1] for p_ in parts], [p_[3] for p_ in parts], o_dtype=torch.float32)
    del parts
    Dc, Dn = m.bdlm_bwd_preprocess(oc, dOc), m.bdlm_bwd_preprocess(on, dOn)
    dQc, dQn, dKn, dVn = z32(nc, Hq), z32(nn, Hq), z32(nn, Hkv), z32(nn, Hkv)
    if schedule == "gathered":
        dKg, dVg = z32(L, Hkv), z32(L, Hkv)  # summed shard by shard onto the owners afterwards
        m.bdlm_attn_bwd_rank(Qc, Kg, Vg, Qn, Kn, Vn, dOc, dOn, lc, ln, Dc, Dn, L, B, 0, L, True, rc, rn,
                             dQc, dQn, dKg, dVg, dKn, dVn, sc)
    else:
        for s_ in range(plan.R):
            lo, hi = plan.shard_keys(s_)
            Ks, Vs, dKs, dVs = bf(hi - lo, Hkv), bf(hi - lo, Hkv), z32(hi - lo, Hkv), z32(hi - lo, Hkv)
            m.bdlm_attn_bwd_rank(Qc, Ks, Vs, Qn, Kn, Vn, dOc, dOn, lc, ln, Dc, Dn, L, B, lo, hi, False, rc, rn,
                                 dQc, dQn, dKs, dVs, dKn, dVn, sc)
            del Ks, Vs, dKs, dVs
        e0 = torch.empty((0, Hkv, d), dtype=torch.float32, device=dev)
        m.bdlm_attn_bwd_rank(Qc, nk, nk, Qn, Kn, Vn, dOc, dOn, lc, ln, Dc, Dn, L, B, 0, 0, True, rc, rn,
                             dQc, dQn, e0, e0, dKn, dVn, sc)
    torch.cuda.synchronize(dev)
    return torch.cuda.max_memory_allocated(dev) - base


# ------------------------------------------------------------------ sweep (measurement tables)
def run_sweep(args):
    """Per-config timings, the schedule ablation and the sharded block-size
    sweep; one JSON line each (not the single bench line)."""
    import statistics

    import torch

    import structured_mask_attention_gb300 as m
    from structured_mask_attention_gb300.inputs import SHARDED_BLOCK_SIZES, WORKLOADS, make_torch

    m.load_library()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    peaks, peak_src = load_peaks()
    peak_tf = peak_value(peaks, "bf16_tflops_sustained")
    names = ("Qc", "Kc", "Vc", "Qn", "Kn", "Vn")
    reps, warm = max(10, args.steps), args.warmup

    def timed(fn):
        """Median CUDA-event time (ms) of fn over reps runs after warm runs."""
        for _ in range(warm):
            fn()
        ts = []
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b))
        return statistics.median(ts)

    def emit(d):
        print(json.dumps(d), flush=True)

    want = set(args.sweep_parts.split(","))
    # ---- configs: forward and backward separately
    for name in (("gqa-8k", "gqa-32k", "long-128k") if "config" in want else ()):
        w = WORKLOADS[name]
        L, B, Hq, Hkv, d = w["L"], w["B"], w["Hq"], w["Hkv"], w["d"]
        X = make_torch(L, Hq, Hkv, d, seed=0, device=dev)
        ins = [X[k] for k in names]
        sc = 1.0 / math.sqrt(d)
        f = m.bdlm_attn_fwd(*ins, B, sc)
        g = m.bdlm_attn_bwd(*ins, f[0], f[1], X["dOc"], X["dOn"], f[2], f[3], B, sc)
        fms = timed(lambda: m.bdlm_attn_fwd(*ins, B, sc, out=f))
        bms = timed(lambda: m.bdlm_attn_bwd(*ins, f[0], f[1], X["dOc"], X["dOn"], f[2], f[3], B, sc, out=g))
        tot = fms + bms
        useful = useful_flops(L, B, Hq, d) / (tot * 1e-3) / 1e12
        emit({"sweep": "config", "workload": name, "L": L, "B": B, "Hq": Hq, "Hkv": Hkv, "d": d,
              "fwd_ms": round(fms, 3), "bwd_ms": round(bms, 3), "step_ms": round(tot, 3),
              "useful_tflops": round(useful, 1), "strict_tflops": round(strict_flops(L, B, Hq, d) / (tot * 1e-3) / 1e12, 1),
              "tokens_per_s": round(2 * L / (tot * 1e-3), 1), "pct_of_peak": round(100 * useful / peak_tf, 2),
              "peak": peak_src, "reps": reps})
        if name == "long-128k":
            # schedule ablation: natural order + round robin vs longest first, claimed in list order
            step = lambda: (m.bdlm_attn_fwd(*ins, B, sc, out=f),
                            m.bdlm_attn_bwd(*ins, f[0], f[1], X["dOc"], X["dOn"], f[2], f[3], B, sc, out=g))
            res = {}
            for sched in ("naive", "lpt"):
                os.environ["BDLM_SCHED"] = sched
                res[sched] = timed(step)
            os.environ.pop("BDLM_SCHED", None)
            emit({"sweep": "schedule", "workload": name, "naive_ms": round(res["naive"], 3),
                  "lpt_ms": round(res["lpt"], 3), "speedup": round(res["naive"] / res["lpt"], 3)})
        del X, ins, f, g
        torch.cuda.empty_cache()

    # ---- sharded-256k: block-size sweep, sharded vs unsharded, merge share
    w = WORKLOADS["sharded-256k"]
    L, Hq, Hkv, d, P = w["L"], w["Hq"], w["Hkv"], w["d"], w["P"]
    sc = 1.0 / math.sqrt(d)
    for B in (SHARDED_BLOCK_SIZES if "sharded" in want else ()):
        X = make_torch(L, Hq, Hkv, d, seed=B, device=dev)
        ins = [X[k] for k in names]
        step = L // P
        bounds = [(s * step, (s + 1) * step) for s in range(P)]
        # peak device memory of one fwd+bwd step of each schedule, inputs included
        # (the single-device form of the pure-BP vs CSBP memory ablation)
        torch.cuda.synchronize()
        torch.cuda.reset_peak_memory_stats(dev)
        fu = m.bdlm_attn_fwd(*ins, B, sc)
        gu = m.bdlm_attn_bwd(*ins, fu[0], fu[1], X["dOc"], X["dOn"], fu[2], fu[3], B, sc)
        torch.cuda.synchronize()
        bp_peak = torch.cuda.max_memory_allocated(dev)
        un_f = timed(lambda: m.bdlm_attn_fwd(*ins, B, sc, out=fu))
        un_b = timed(lambda: m.bdlm_attn_bwd(*ins, fu[0], fu[1], X["dOc"], X["dOn"], fu[2], fu[3], B, sc, out=gu))
        del gu
        torch.cuda.synchronize()
        base_mem = torch.cuda.memory_allocated(dev) - sum(t.numel() * t.element_size() for t in fu)
        torch.cuda.reset_peak_memory_stats(dev)
        parts = [m.bdlm_attn_fwd_shard(*ins, B, lo, hi, False, sc) for (lo, hi) in bounds]
        parts.append(m.bdlm_attn_fwd_shard(*ins, B, 0, 0, True, sc))
        spec = [(lo, hi, False) for (lo, hi) in bounds] + [(0, 0, True)]

        def part_fwd():
            for (lo, hi, loc), pt in zip(spec, parts):
                m.bdlm_attn_fwd_shard(*ins, B, lo, hi, loc, sc, out=pt)

        mo = [torch.empty((L, Hq, d), dtype=torch.bfloat16, device=dev) for _ in range(2)]
        ml = [torch.empty((Hq, L), dtype=torch.float32, device=dev) for _ in range(2)]

        def merge():
            m.bdlm_lse_merge([p_[0] for p_ in parts], [p_[2] for p_ in parts], out=mo[0], lse_out=ml[0])
            m.bdlm_lse_merge([p_[1] for p_ in parts], [p_[3] for p_ in parts], out=mo[1], lse_out=ml[1])

        sh_f = timed(part_fwd)
        mg = timed(merge)
        Dc = m.bdlm_bwd_preprocess(mo[0], X["dOc"])
        Dn = m.bdlm_bwd_preprocess(mo[1], X["dOn"])
        pre = timed(lambda: (m.bdlm_bwd_preprocess(mo[0], X["dOc"], out=Dc),
                             m.bdlm_bwd_preprocess(mo[1], X["dOn"], out=Dn)))
        z = lambda H: torch.zeros((L, H, d), dtype=torch.float32, device=dev)
        dQc, dQn, dKc, dVc, dKn, dVn = z(Hq), z(Hq), z(Hkv), z(Hkv), z(Hkv), z(Hkv)

        def part_bwd():
            for (lo, hi, loc) in spec:
                m.bdlm_attn_bwd_shard(*ins, X["dOc"], X["dOn"], ml[0], ml[1], Dc, Dn, B, lo, hi, loc,
                                      dQc, dQn, dKc, dVc, dKn, dVn, sc)

        part_bwd()
        torch.cuda.synchronize()
        # the shard-and-merge step's peak: its partials, merged outputs, D and
        # fp32 gradients on top of the inputs (the unsharded outputs, still
        # allocated for the timing above, are not part of it)
        csbp_peak = torch.cuda.max_memory_allocated(dev) - sum(t.numel() * t.element_size() for t in fu)
        csbp_peak = max(csbp_peak, base_mem)
        sh_b = timed(part_bwd)
        # merge bytes: every non-empty (row, head, partial) O row read, all LSE_p read, O (bf16) and LSE written
        nonempty = sum(int((p_[2] > float("-inf")).sum().item() + (p_[3] > float("-inf")).sum().item())
                       for p_ in parts)
        mbytes = nonempty * d * 4 + len(parts) * 2 * L * Hq * 4 + 2 * L * Hq * (d * 2 + 4)
        pbytes = 2 * (2 * L * Hq * d * 2 + L * Hq * 4)
        sh_tot = sh_f + mg + pre + sh_b
        emit({"sweep": "sharded", "workload": "sharded-256k", "B": B, "P": P,
              "unsharded_fwd_ms": round(un_f, 3), "unsharded_bwd_ms": round(un_b, 3),
              "sharded_fwd_ms": round(sh_f, 3), "merge_ms": round(mg, 3), "preprocess_ms": round(pre, 3),
              "sharded_bwd_ms": round(sh_b, 3), "sharded_total_ms": round(sh_tot, 3),
              "unsharded_useful_tflops": round(useful_flops(L, B, Hq, d) / ((un_f + un_b) * 1e-3) / 1e12, 1),
              "sharded_useful_tflops": round(useful_flops(L, B, Hq, d) / (sh_tot * 1e-3) / 1e12, 1),
              "merge_share": round(mg / sh_tot, 5), "merge_gbs": round(mbytes / (mg * 1e-3) / 1e9, 1),
              "merge_bytes": mbytes, "preprocess_gbs": round(pbytes / (pre * 1e-3) / 1e9, 1),
              "unsharded_peak_gib": round(bp_peak / 2 ** 30, 2), "sharded_peak_gib": round(csbp_peak / 2 ** 30, 2),
              "per_rank_gib_model_R8": per_rank_memory(L, Hq, Hkv, d, 8)})
        del X, ins, fu, parts, mo, ml, Dc, Dn, dQc, dQn, dKc, dVc, dKn, dVn
        torch.cuda.empty_cache()

    # ---- sharded-256k: shard-and-merge vs unsharded fp32 output, production
    # path (P rounded to bf16 against each path's running maximum) and the
    # fixed-reference verification mode (same P in both paths)
    for B in (SHARDED_BLOCK_SIZES if "shardcheck" in want else ()):
        X = make_torch(L, Hq, Hkv, d, seed=B, device=dev)
        ins = [X[k] for k in names]
        step = L // P
        specs = [(s * step, (s + 1) * step, False) for s in range(P)] + [(0, 0, True)]
        u = m.bdlm_attn_fwd(*ins, B, sc, o_dtype=torch.float32)
        res = {}
        for mode in ("production", "fixed_reference"):
            if mode == "production":
                full = u
                parts = [m.bdlm_attn_fwd_shard(*ins, B, lo, hi, loc, sc) for (lo, hi, loc) in specs]
            else:
                full = m.bdlm_attn_fwd_shard_refmax(*ins, B, 0, L, True, u[2], u[3], sc)
                parts = [m.bdlm_attn_fwd_shard_refmax(*ins, B, lo, hi, loc, u[2], u[3], sc) for (lo, hi, loc) in specs]
            oc, lc = m.bdlm_lse_merge([p_[0] for p_ in parts], [p_[2] for p_ in parts], o_dtype=torch.float32)
            on, ln = m.bdlm_lse_merge([p_[1] for p_ in parts], [p_[3] for p_ in parts], o_dtype=torch.float32)
            del parts
            res[mode] = (max((oc - full[0]).abs().max().item(), (on - full[1]).abs().max().item()),
                         max((lc - full[2]).abs().max().item(), (ln - full[3]).abs().max().item()))
            del full, oc, on, lc, ln
        omax = max(u[0].abs().max().item(), u[1].abs().max().item())
        vmax = max(X["Vc"].abs().max().item(), X["Vn"].abs().max().item())
        emit({"sweep": "shardcheck", "workload": "sharded-256k", "B": B, "P": P,
              "production_max_abs_dO": res["production"][0], "production_max_abs_dLSE": res["production"][1],
              "fixed_reference_max_abs_dO": res["fixed_reference"][0],
              "fixed_reference_max_abs_dLSE": res["fixed_reference"][1],
              "max_abs_O": omax, "max_abs_V": vmax})
        del X, ins, u
        torch.cuda.empty_cache()

    # ---- packed batches: one packed call vs one call per sequence
    from structured_mask_attention_gb300.inputs import workload_lengths
    for name in (("packed-128k", "batch-64x2k") if "packed" in want else ()):
        w = WORKLOADS[name]
        T, B, Hq, Hkv, d = w["T"], w["B"], w["Hq"], w["Hkv"], w["d"]
        lens = workload_lengths(name)
        offs = [0]
        for n_ in lens:
            offs.append(offs[-1] + n_)
        X = make_torch(T, Hq, Hkv, d, seed=0, device=dev)
        ins = [X[k] for k in names]
        sc = 1.0 / math.sqrt(d)
        wf = torch.empty(m.bdlm_workspace_size_varlen(m.OP_FWD, lens, Hq, Hkv, d), dtype=torch.uint8, device=dev)
        wb = torch.empty(m.bdlm_workspace_size_varlen(m.OP_BWD, lens, Hq, Hkv, d), dtype=torch.uint8, device=dev)
        f = m.bdlm_attn_fwd_varlen(*ins, lens, B, sc, workspace=wf)
        g = m.bdlm_attn_bwd_varlen(*ins, f[0], f[1], X["dOc"], X["dOn"], f[2], f[3], lens, B, sc, workspace=wb)
        pf = timed(lambda: m.bdlm_attn_fwd_varlen(*ins, lens, B, sc, out=f, workspace=wf))
        pb = timed(lambda: m.bdlm_attn_bwd_varlen(*ins, f[0], f[1], X["dOc"], X["dOn"], f[2], f[3], lens, B, sc,
                                                  out=g, workspace=wb))
        # ablation: longest item first over the whole batch (host-built list)
        os.environ["BDLM_VARLEN_ORDER"] = "lpt"
        af = timed(lambda: m.bdlm_attn_fwd_varlen(*ins, lens, B, sc, out=f, workspace=wf))
        ab = timed(lambda: m.bdlm_attn_bwd_varlen(*ins, f[0], f[1], X["dOc"], X["dOn"], f[2], f[3], lens, B, sc,
                                                  out=g, workspace=wb))
        os.environ.pop("BDLM_VARLEN_ORDER", None)
        # the same sequences one call each (slices of the packed tensors)
        sl = [(a, b_) for a, b_ in zip(offs[:-1], offs[1:])]
        fo = [m.bdlm_attn_fwd(*[t[a:b_] for t in ins], B, sc) for (a, b_) in sl]
        go = [m.bdlm_attn_bwd(*[t[a:b_] for t in ins], fo[i][0], fo[i][1], X["dOc"][a:b_], X["dOn"][a:b_],
                              fo[i][2], fo[i][3], B, sc) for i, (a, b_) in enumerate(sl)]

        def loop_fwd():
            for i, (a, b_) in enumerate(sl):
                m.bdlm_attn_fwd(*[t[a:b_] for t in ins], B, sc, out=fo[i])

        def loop_bwd():
            for i, (a, b_) in enumerate(sl):
                m.bdlm_attn_bwd(*[t[a:b_] for t in ins], fo[i][0], fo[i][1], X["dOc"][a:b_], X["dOn"][a:b_],
                                fo[i][2], fo[i][3], B, sc, out=go[i])

        lf = timed(loop_fwd)
        lb = timed(loop_bwd)
        uf = sum(useful_flops(n_, B, Hq, d) for n_ in lens)
        ptf = uf / ((pf + pb) * 1e-3) / 1e12
        emit({"sweep": "packed", "workload": name, "T": T, "B": B, "Hq": Hq, "Hkv": Hkv, "d": d,
              "n_seqs": len(lens), "lens": lens,
              "packed_fwd_ms": round(pf, 3), "packed_bwd_ms": round(pb, 3), "packed_step_ms": round(pf + pb, 3),
              "lpt_order_step_ms": round(af + ab, 3),
              "per_seq_fwd_ms": round(lf, 3), "per_seq_bwd_ms": round(lb, 3), "per_seq_step_ms": round(lf + lb, 3),
              "packed_useful_tflops": round(ptf, 1),
              "per_seq_useful_tflops": round(uf / ((lf + lb) * 1e-3) / 1e12, 1),
              "packed_tokens_per_s": round(2 * T / ((pf + pb) * 1e-3), 1),
              "pct_of_peak": round(100 * ptf / peak_tf, 2), "speedup": round((lf + lb) / (pf + pb), 3),
              "peak": peak_src, "reps": reps})
        del X, ins, f, g, fo, go, wf, wb
        torch.cuda.empty_cache()

    # ---- multi-rank CSBP: each rank's compute (its row-restricted partial
    # forward and backward calls) timed alone on this GPU, as if it were that
    # rank's device; the exchange is not included.  Mirror assignment of the
    # corrupted slices (balanced) against the split by token position.
    if "ranks" in want:
        from structured_mask_attention_gb300 import csbp
        w = WORKLOADS["long-128k"]
        L, B, Hq, Hkv, d = w["L"], w["B"], w["Hq"], w["Hkv"], w["d"]
        sc = 1.0 / math.sqrt(d)
        X = make_torch(L, Hq, Hkv, d, seed=0, device=dev)
        ins = [X[k] for k in names]
        fu = m.bdlm_attn_fwd(*ins, B, sc)
        gu = m.bdlm_attn_bwd(*ins, fu[0], fu[1], X["dOc"], X["dOn"], fu[2], fu[3], B, sc)
        un = timed(lambda: (m.bdlm_attn_fwd(*ins, B, sc, out=fu),
                            m.bdlm_attn_bwd(*ins, fu[0], fu[1], X["dOc"], X["dOn"], fu[2], fu[3], B, sc, out=gu)))
        del gu
        # merged statistics of the whole problem (the ranks' merged rows equal them up to rounding)
        Dc = m.bdlm_bwd_preprocess(fu[0], X["dOc"])
        Dn = m.bdlm_bwd_preprocess(fu[1], X["dOn"])
        z = lambda H: torch.zeros((L, H, d), dtype=torch.float32, device=dev)
        acc = (z(Hq), z(Hq), z(Hkv), z(Hkv), z(Hkv), z(Hkv))
        for R in (2, 4, 8):
            f32 = dict(dtype=torch.float32, device=dev)
            parts = [(torch.zeros((L, Hq, d), **f32), torch.zeros((L, Hq, d), **f32),
                      torch.full((Hq, L), float("-inf"), **f32), torch.full((Hq, L), float("-inf"), **f32))
                     for _ in range(R + 1)]
            for policy, schedule in [(p_, "per_shard") for p_ in csbp.POLICIES] + [("mirror", "gathered")]:
                plan = csbp.CSBPPlan.build(L, B, R, policy)
                if schedule == "per_shard":  # partials per clean shard + the local one, merged
                    specs = [(*plan.shard_keys(s_), False) for s_ in range(R)] + [(0, 0, True)]
                else:  # one call over the all-gathered clean sequence and the local blocks
                    specs = [(0, L, True)]

                def rank_fwd(r):
                    rw = plan.rows(r)
                    rc, rn = (rw.c0 * B, rw.c1 * B), (rw.n0 * B, rw.n1 * B)
                    for (lo, hi, loc), pt in zip(specs, parts):
                        m.bdlm_attn_fwd_shard_rows(*ins, B, lo, hi, loc, rc, rn, sc, out=pt)

                def rank_bwd(r):
                    rw = plan.rows(r)
                    rc, rn = (rw.c0 * B, rw.c1 * B), (rw.n0 * B, rw.n1 * B)
                    for (lo, hi, loc) in specs:
                        m.bdlm_attn_bwd_shard_rows(*ins, X["dOc"], X["dOn"], fu[2], fu[3], Dc, Dn, B, lo, hi, loc,
                                                   rc, rn, *acc, sc)

                per = [(timed(lambda: rank_fwd(r)), timed(lambda: rank_bwd(r))) for r in range(R)]
                tot = [a + b_ for (a, b_) in per]
                mean = sum(tot) / R
                emit({"sweep": "ranks", "workload": "long-128k", "L": L, "B": B, "Hq": Hq, "Hkv": Hkv, "d": d,
                      "R": R, "policy": policy, "schedule": schedule, "calls_per_rank": 2 * len(specs),
                      "rank_fwd_ms": [round(a, 3) for (a, _) in per], "rank_bwd_ms": [round(b_, 3) for (_, b_) in per],
                      "max_ms": round(max(tot), 3), "mean_ms": round(mean, 3),
                      "imbalance": round(max(tot) / mean, 4), "model_imbalance": round(plan.imbalance(), 4),
                      "sum_over_ranks_ms": round(sum(tot), 3), "unsharded_ms": round(un, 3),
                      "useful_tflops_per_rank_bound": round(useful_flops(L, B, Hq, d) / R / (max(tot) * 1e-3) / 1e12, 1),
                      "reps": reps})
            del parts
        del X, ins, fu, Dc, Dn, acc
        torch.cuda.empty_cache()
        # each rank's device memory through the rank-local calls (rank 0 and
        # the last rank of the balanced plan; nothing else allocated)
        for R in (2, 4, 8):
            plan = csbp.CSBPPlan.build(L, B, R)
            for schedule in ("gathered", "per_shard"):
                peaks = [rank_program_memory(m, plan, r, Hq, Hkv, d, schedule, dev) for r in (0, R - 1)]
                torch.cuda.empty_cache()
                emit({"sweep": "rank_memory", "workload": "long-128k", "R": R, "schedule": schedule,
                      "peak_gib_rank0_last": [round(x / 2 ** 30, 3) for x in peaks],
                      "model_gib": per_rank_memory(L, Hq, Hkv, d, R)})

    # ---- the fp64 oracle on the host cores: a timed sample per config,
    # extrapolated by useful FLOP to the whole config (all heads, both streams)
    for name in (("tiny", "gqa-8k", "gqa-32k", "long-128k", "sharded-256k") if "oracle" in want else ()):
        w = WORKLOADS[name]
        L, B, Hq, Hkv, d = w["L"], w["B"], w["Hq"], w["Hkv"], w["d"]
        if name == "sharded-256k":
            L, B = 4096, 512  # the 4096-token slice the parity tests check against the oracle
        flops, dt, blocks, thr = oracle_sample(L, B, Hq, Hkv, d, budget_s=min(args.cpu_budget, 8.0))
        rate = flops / dt
        full = useful_flops(L, B, Hq, d)
        emit({"sweep": "oracle", "workload": name, "L": L, "B": B, "Hq": Hq, "sample_blocks": blocks,
              "sample_s": round(dt, 2), "oracle_gflops": round(rate / 1e9, 2),
              "full_s": round(full / rate, 3 if full / rate < 10 else 1),
              "extrapolated": blocks < L // B or Hq > 1, "threads": thr})


# ------------------------------------------------------------------ reference arm
def run_reference(args):
    from structured_mask_attention_gb300.inputs import WORKLOADS
    w = WORKLOADS[args.workload]
    L, B, Hq, Hkv, d = w["L"], w["B"], w["Hq"], w["Hkv"], w["d"]
    budget = max(1.0, min(args.cpu_budget, 240.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_sample(L, B, Hq, Hkv, d, budget * 0.25)
    tot_f, tot_t, blocks, thr = 0.0, 0.0, 0, 1
    for _ in range(args.steps):
        f, t, nb, thr = oracle_sample(L, B, Hq, Hkv, d, budget)
        tot_f += f; tot_t += t; blocks += nb
    value = tot_f / tot_t / 1e12
    sample = (f"fp64 oracle fwd+bwd of the last blocks of one query head of {args.workload} (both streams), "
              f"{blocks} blocks over {args.steps} steps")
    return {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * tot_t / args.steps, 1),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded N(0,1), bf16-rounded)",
            "config": {"workload": args.workload, "L": L, "B": B, "Hq": Hq, "Hkv": Hkv, "d": d},
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": thr, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("native", "reference"), default="native")
    ap.add_argument("--workload", choices=(WORKLOAD, "profile-16k"), default=WORKLOAD,
                    help="profile-16k: the same head layout at 1/8 length, for profiler captures")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle work for the CPU baseline")
    ap.add_argument("--sweep", action="store_true",
                    help="measurement tables instead of the bench line: per-config fwd/bwd times, the "
                         "schedule ablation (BDLM_SCHED=naive vs longest first) and the sharded-256k "
                         "block-size sweep with merge and preprocess bandwidth, and packed batches "
                         "(one packed call vs one call per sequence)")
    ap.add_argument("--csbp", action="store_true",
                    help="multi-rank CSBP instead of replicas: one sequence split over the --gpus ranks "
                         "(balanced plan, rank-local calls, clean K/V all-gathered and clean dK/dV reduced "
                         "over NCCL); strong scaling")
    ap.add_argument("--sweep-parts", default="config,sharded,shardcheck,packed,ranks,oracle",
                    help="comma-separated parts of --sweep to run (config includes the schedule ablation; "
                         "shardcheck: sharded vs unsharded fp32 output differences, production path and "
                         "fixed-reference mode; ranks: each rank's compute of multi-rank CSBP at long-128k, "
                         "balanced and by-position assignment)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return
    if args.sweep:
        if rank == 0:
            run_sweep(args)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    line = run_csbp(args, rank, world, local_rank) if args.csbp else run_native(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
