"""Builds libbdlm_attn.so in-tree with nvcc for sm_103a.

Each CUDA source compiles to an object in parallel, then one shared library is
linked next to this file.  No CMake, no torch extension machinery: the
library is plain C ABI (include/bdlm_attn.h).
"""
from __future__ import annotations

import json
import os
import platform
import shutil
import subprocess
import sys
import time
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OBJ = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libbdlm_attn.so")
SOURCES = ["abi.cu", "fwd_tc.cu", "bwd_dq.cu", "bwd_dkv.cu", "small_kernels.cu", "noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for c in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found")


def _flags(ptxas_verbose: bool):
    f = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
                "-I", os.path.join(ROOT, "include"), "-I", CSRC]
    if ptxas_verbose:
        f += ["-Xptxas", "-v"]
    return f


def build(verbose: bool = False, ptxas_verbose: bool = False, force: bool = False) -> str:
    """Compiles every source that changed and links the library; returns its path."""
    os.makedirs(OBJ, exist_ok=True)
    cc = nvcc()
    headers = [os.path.join(CSRC, h) for h in os.listdir(CSRC) if h.endswith((".cuh", ".h"))]
    headers.append(os.path.join(ROOT, "include", "bdlm_attn.h"))
    newest_header = max(os.path.getmtime(h) for h in headers)

    def compile_one(src):
        s = os.path.join(CSRC, src)
        o = os.path.join(OBJ, src + ".o")
        if (not force and not ptxas_verbose and os.path.exists(o)
                and os.path.getmtime(o) >= max(os.path.getmtime(s), newest_header)):
            return o, "", False
        cmd = [cc] + _flags(ptxas_verbose) + ["-c", s, "-o", o]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        return o, r.stderr, True

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose or ptxas_verbose:
        for (o, log, _) in results:
            if log:
                sys.stderr.write(log)
    objs = [o for (o, _, _) in results]
    linked = False
    if force or not os.path.exists(LIB) or os.path.getmtime(LIB) < max(os.path.getmtime(o) for o in objs):
        tmp = LIB + ".tmp"
        cmd = [cc] + ARCH + ["-shared", "-o", tmp] + objs + ["-lcudart_static", "-ldl", "-lpthread", "-lrt"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, LIB)
        linked = True
    # what this call did, for the record: which objects were compiled here
    # and which were reused (up to date with their sources and headers)
    record = {"compiled": [os.path.basename(o) for (o, _, c) in results if c],
              "reused": [os.path.basename(o) for (o, _, c) in results if not c],
              "linked": linked, "nvcc": cc, "arch": ARCH[1], "machine": platform.machine(),
              "time": time.strftime("%Y-%m-%dT%H:%M:%S")}
    with open(os.path.join(OBJ, "build_record.json"), "w") as fh:
        json.dump(record, fh, indent=1)
    print(f"bdlm build: compiled {len(record['compiled'])}, reused {len(record['reused'])} of {len(SOURCES)} "
          f"sources; {'linked' if linked else 'library up to date'} ({record['machine']}, {ARCH[1]})",
          file=sys.stderr)
    return LIB


if __name__ == "__main__":
    print(build(verbose=True, ptxas_verbose="-v" in sys.argv, force="-f" in sys.argv))
