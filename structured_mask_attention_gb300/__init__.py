"""Two-stream block-diffusion (BDLM) attention for GB300 (sm_103a).

Python binding of the C ABI in ``include/bdlm_attn.h``: every function here
has the name of the C entry point it calls and only marshals arguments
(tensor pointers, sizes, the current CUDA stream) and allocates outputs with
torch.  All computation runs in ``libbdlm_attn.so``; if the library is
missing or fails to load, every call raises.  There is no fallback path.

Layouts: Q, K, V, O, dO and gradients are ``[L, H, d]`` contiguous tensors per
stream (clean ``c``, corrupted ``n``); LSE and D are ``[H, L]`` float32.
"""
from __future__ import annotations

import ctypes
import math
import os
import re

__all__ = [
    "BdlmError", "load_library", "bdlm_workspace_size", "bdlm_attn_fwd", "bdlm_attn_fwd_shard",
    "bdlm_attn_fwd_shard_refmax", "bdlm_attn_fwd_shard_rows", "bdlm_attn_bwd_shard_rows",
    "bdlm_attn_fwd_rank", "bdlm_attn_bwd_rank",
    "bdlm_lse_merge", "bdlm_bwd_preprocess", "bdlm_attn_bwd", "bdlm_attn_bwd_noalloc", "bdlm_attn_bwd_shard",
    "bdlm_worklist", "bdlm_workspace_size_varlen", "bdlm_attn_fwd_varlen", "bdlm_attn_bwd_varlen",
    "bdlm_sync_status", "bdlm_watchdog_selftest", "bdlm_sync_status_noalloc", "bdlm_watchdog_selftest_noalloc",
    "bdlm_kernel_launches", "bdlm_last_error",
    "bdlm_version", "bdlm_timing_enable", "bdlm_timing_report", "header_functions", "LIB_PATH",
    "HEADER_PATH",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libbdlm_attn.so")
HEADER_PATH = os.path.join(os.path.dirname(_PKG), "include", "bdlm_attn.h")

STATUS = {0: "BDLM_OK", 1: "BDLM_ERR_INVALID_ARG", 2: "BDLM_ERR_SHAPE", 3: "BDLM_ERR_ALIGN",
          4: "BDLM_ERR_WORKSPACE", 5: "BDLM_ERR_CUDA", 6: "BDLM_ERR_UNSUPPORTED", 7: "BDLM_ERR_TIMEOUT"}
OP_FWD, OP_FWD_SHARD, OP_BWD, OP_BWD_SHARD = 0, 1, 2, 3
BF16, F32 = 0, 1


class BdlmError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


_lib = None

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I = ctypes.c_int
_F = ctypes.c_float
_SZ = ctypes.c_size_t

_SIGS = {
    "bdlm_workspace_size": (_SZ, [_I, _I64, _I64, _I, _I, _I, _I]),
    "bdlm_attn_fwd": (_I, [_P] * 6 + [_I64, _I64, _I, _I, _I, _F, _P, _P, _I, _P, _P, _P, _SZ, _P]),
    "bdlm_attn_fwd_shard": (_I, [_P] * 6 + [_I64, _I64, _I, _I, _I, _F, _I64, _I64, _I, _P, _P, _P, _P, _P,
                                            _SZ, _P]),
    "bdlm_attn_fwd_shard_refmax": (_I, [_P] * 6 + [_I64, _I64, _I, _I, _I, _F, _I64, _I64, _I, _P, _P, _P, _P, _P,
                                                   _P, _P, _SZ, _P]),
    "bdlm_lse_merge": (_I, [_I, _P, _P, _I64, _I, _I, _P, _I, _P, _P]),
    "bdlm_bwd_preprocess": (_I, [_P, _I, _P, _I64, _I, _I, _P, _P]),
    "bdlm_attn_bwd": (_I, [_P] * 12 + [_I64, _I64, _I, _I, _I, _F] + [_P] * 6 + [_I, _P, _SZ, _P]),
    "bdlm_attn_bwd_shard": (_I, [_P] * 12 + [_I64, _I64, _I, _I, _I, _F, _I64, _I64, _I] + [_P] * 6
                            + [_P, _SZ, _P]),
    "bdlm_attn_bwd_noalloc": (_I, [_P] * 12 + [_I64, _I64, _I, _I, _I, _F] + [_P] * 6 + [_I, _P]),
    "bdlm_attn_fwd_shard_rows": (_I, [_P] * 6 + [_I64, _I64, _I, _I, _I, _F, _I64, _I64, _I] + [_I64] * 4
                                 + [_P] * 5 + [_SZ, _P]),
    "bdlm_attn_bwd_shard_rows": (_I, [_P] * 12 + [_I64, _I64, _I, _I, _I, _F, _I64, _I64, _I] + [_I64] * 4
                                 + [_P] * 7 + [_SZ, _P]),
    "bdlm_attn_fwd_rank": (_I, [_P] * 6 + [_I64, _I64, _I, _I, _I, _F, _I64, _I64, _I] + [_I64] * 4
                           + [_P] * 5 + [_SZ, _P]),
    "bdlm_attn_bwd_rank": (_I, [_P] * 12 + [_I64, _I64, _I, _I, _I, _F, _I64, _I64, _I] + [_I64] * 4
                           + [_P] * 7 + [_SZ, _P]),
    "bdlm_worklist": (_I64, [_I64, _I64, _I, _I, _I, _I, _I64, _I64, _I, _P, _I64]),
    "bdlm_workspace_size_varlen": (_SZ, [_I, _P, _I, _I, _I, _I]),
    "bdlm_attn_fwd_varlen": (_I, [_P] * 6 + [_P, _I, _I64, _I, _I, _I, _F, _P, _P, _I, _P, _P, _P, _SZ, _P]),
    "bdlm_attn_bwd_varlen": (_I, [_P] * 12 + [_P, _I, _I64, _I, _I, _I, _F] + [_P] * 6 + [_I, _P, _SZ, _P]),
    "bdlm_sync_status": (_I, [_P, _P]),
    "bdlm_sync_status_noalloc": (_I, [_P]),
    "bdlm_watchdog_selftest_noalloc": (_I, [ctypes.c_uint32, _P]),
    "bdlm_watchdog_selftest": (_I, [_P, _SZ, ctypes.c_uint32, _P]),
    "bdlm_kernel_launches": (ctypes.c_uint64, []),
    "bdlm_timing_enable": (_I, [_I]),
    "bdlm_timing_report": (_I64, [ctypes.c_char_p, _I64, _I]),
    "bdlm_last_error": (ctypes.c_char_p, []),
    "bdlm_version": (ctypes.c_char_p, []),
}


def header_functions(path: str = HEADER_PATH):
    """Names of the functions declared in the C header."""
    with open(path) as fh:
        text = fh.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(bdlm_[a-z_0-9]+)\s*\(", text)))


def load_library(path: str = LIB_PATH):
    """Loads (once) and returns the native library; raises if it is absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"native library {path} is missing; run __graft_entry__.build() "
                           "(structured_mask_attention_gb300.build.build())")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _check(status: int):
    if status != 0:
        raise BdlmError(status, bdlm_last_error())


def bdlm_last_error() -> str:
    return load_library().bdlm_last_error().decode()


def bdlm_version() -> str:
    return load_library().bdlm_version().decode()


def bdlm_kernel_launches() -> int:
    return int(load_library().bdlm_kernel_launches())


def bdlm_timing_enable(on: bool = True) -> None:
    """Turns per-kernel event timing (on the launching stream) on or off."""
    _check(load_library().bdlm_timing_enable(int(bool(on))))


def bdlm_timing_report(reset: bool = True) -> dict:
    """{kernel name: (launches, total_ms)} accumulated since the last reset."""
    lib = load_library()
    buf = ctypes.create_string_buffer(4096)
    n = lib.bdlm_timing_report(buf, len(buf), int(bool(reset)))
    if n < 0:
        raise BdlmError(5, "event timing failed")
    out = {}
    for line in buf.value.decode().splitlines():
        name, cnt, ms = line.split()
        out[name] = (int(cnt), float(ms))
    return out


def bdlm_workspace_size(op: int, L: int, B: int, Hq: int, Hkv: int, d: int, P: int = 1) -> int:
    return int(load_library().bdlm_workspace_size(op, L, B, Hq, Hkv, d, P))


# ----------------------------------------------------------------- torch side
def _torch():
    import torch
    return torch


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _shape(Qc, Kc):
    L, Hq, d = Qc.shape
    Hkv = Kc.shape[1]
    return L, Hq, Hkv, d


def _dt(dtype) -> int:
    torch = _torch()
    return F32 if dtype == torch.float32 else BF16


def _workspace(op, L, B, Hq, Hkv, d, device, ws):
    torch = _torch()
    need = bdlm_workspace_size(op, L, B, Hq, Hkv, d, 1)
    if ws is None:
        ws = torch.empty(max(need, 256), dtype=torch.uint8, device=device)
    return ws


def _check_inputs(*ts):
    torch = _torch()
    for t in ts:
        if not t.is_cuda or not t.is_contiguous() or t.dtype != torch.bfloat16:
            raise ValueError("inputs must be contiguous bf16 CUDA tensors")


def bdlm_attn_fwd(Qc, Kc, Vc, Qn, Kn, Vn, B: int, scale: float | None = None, o_dtype=None,
                  out=None, workspace=None, stream=None):
    """O and LSE of both streams.  Returns (Oc, On, LSEc, LSEn)."""
    torch = _torch()
    _check_inputs(Qc, Kc, Vc, Qn, Kn, Vn)
    L, Hq, Hkv, d = _shape(Qc, Kc)
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    o_dtype = torch.bfloat16 if o_dtype is None else o_dtype
    if out is None:
        out = (torch.empty((L, Hq, d), dtype=o_dtype, device=Qc.device),
               torch.empty((L, Hq, d), dtype=o_dtype, device=Qc.device),
               torch.empty((Hq, L), dtype=torch.float32, device=Qc.device),
               torch.empty((Hq, L), dtype=torch.float32, device=Qc.device))
    Oc, On, LSEc, LSEn = out
    ws = _workspace(OP_FWD, L, B, Hq, Hkv, d, Qc.device, workspace)
    _check(load_library().bdlm_attn_fwd(
        _ptr(Qc), _ptr(Kc), _ptr(Vc), _ptr(Qn), _ptr(Kn), _ptr(Vn), L, B, Hq, Hkv, d, scale,
        _ptr(Oc), _ptr(On), _dt(Oc.dtype), _ptr(LSEc), _ptr(LSEn), _ptr(ws), ws.numel(), _stream(stream)))
    return Oc, On, LSEc, LSEn


def bdlm_attn_fwd_shard(Qc, Kc, Vc, Qn, Kn, Vn, B: int, kv_begin: int, kv_end: int, include_local: bool,
                        scale: float | None = None, out=None, workspace=None, stream=None):
    """fp32 partial (O_p, LSE_p) of both streams against clean keys
    [kv_begin, kv_end) (+ the corrupted own block if include_local).
    Returns (Op_c, Op_n, LSEp_c, LSEp_n)."""
    torch = _torch()
    _check_inputs(Qc, Kc, Vc, Qn, Kn, Vn)
    L, Hq, Hkv, d = _shape(Qc, Kc)
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    if out is None:
        out = (torch.empty((L, Hq, d), dtype=torch.float32, device=Qc.device),
               torch.empty((L, Hq, d), dtype=torch.float32, device=Qc.device),
               torch.empty((Hq, L), dtype=torch.float32, device=Qc.device),
               torch.empty((Hq, L), dtype=torch.float32, device=Qc.device))
    ws = _workspace(OP_FWD_SHARD, L, B, Hq, Hkv, d, Qc.device, workspace)
    _check(load_library().bdlm_attn_fwd_shard(
        _ptr(Qc), _ptr(Kc), _ptr(Vc), _ptr(Qn), _ptr(Kn), _ptr(Vn), L, B, Hq, Hkv, d, scale,
        kv_begin, kv_end, int(bool(include_local)), *[_ptr(t) for t in out], _ptr(ws), ws.numel(),
        _stream(stream)))
    return out


def bdlm_attn_fwd_shard_refmax(Qc, Kc, Vc, Qn, Kn, Vn, B: int, kv_begin: int, kv_end: int, include_local: bool,
                               Mref_c, Mref_n, scale: float | None = None, out=None, workspace=None, stream=None):
    """Verification mode of ``bdlm_attn_fwd_shard``: every row's probabilities
    are formed against the fixed reference ``Mref_c`` / ``Mref_n`` ([Hq, L]
    fp32, natural log, e.g. the unsharded forward's LSE) instead of its
    running maximum.  Returns (Op_c, Op_n, LSEp_c, LSEp_n), fp32."""
    torch = _torch()
    _check_inputs(Qc, Kc, Vc, Qn, Kn, Vn)
    L, Hq, Hkv, d = _shape(Qc, Kc)
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    for t in (Mref_c, Mref_n):
        if not t.is_cuda or not t.is_contiguous() or t.dtype != torch.float32 or tuple(t.shape) != (Hq, L):
            raise ValueError("Mref must be a contiguous float32 CUDA tensor of shape [Hq, L]")
    if out is None:
        out = (torch.empty((L, Hq, d), dtype=torch.float32, device=Qc.device),
               torch.empty((L, Hq, d), dtype=torch.float32, device=Qc.device),
               torch.empty((Hq, L), dtype=torch.float32, device=Qc.device),
               torch.empty((Hq, L), dtype=torch.float32, device=Qc.device))
    ws = _workspace(OP_FWD_SHARD, L, B, Hq, Hkv, d, Qc.device, workspace)
    _check(load_library().bdlm_attn_fwd_shard_refmax(
        _ptr(Qc), _ptr(Kc), _ptr(Vc), _ptr(Qn), _ptr(Kn), _ptr(Vn), L, B, Hq, Hkv, d, scale,
        kv_begin, kv_end, int(bool(include_local)), _ptr(Mref_c), _ptr(Mref_n), *[_ptr(t) for t in out],
        _ptr(ws), ws.numel(), _stream(stream)))
    return out


def bdlm_lse_merge(O_parts, LSE_parts, o_dtype=None, out=None, lse_out=None, write_lse: bool = True,
                   stream=None):
    """Exact LSE merge of fp32 partials [rows, H, d] / [H, rows].
    Returns (O, LSE) (LSE is None when write_lse is False)."""
    torch = _torch()
    n = len(O_parts)
    rows, H, d = O_parts[0].shape
    o_dtype = torch.bfloat16 if o_dtype is None else o_dtype
    O = torch.empty((rows, H, d), dtype=o_dtype, device=O_parts[0].device) if out is None else out
    LSE = None
    if write_lse:
        LSE = torch.empty((H, rows), dtype=torch.float32, device=O_parts[0].device) if lse_out is None else lse_out
    arr_o = (ctypes.c_void_p * n)(*[t.data_ptr() for t in O_parts])
    arr_l = (ctypes.c_void_p * n)(*[t.data_ptr() for t in LSE_parts])
    _check(load_library().bdlm_lse_merge(n, ctypes.cast(arr_o, ctypes.c_void_p), ctypes.cast(arr_l, ctypes.c_void_p),
                                         rows, H, d, _ptr(O), _dt(O.dtype), _ptr(LSE), _stream(stream)))
    return O, LSE


def bdlm_bwd_preprocess(O, dO, out=None, stream=None):
    """D = rowsum(dO * O) as [H, rows] fp32."""
    torch = _torch()
    rows, H, d = O.shape
    D = torch.empty((H, rows), dtype=torch.float32, device=O.device) if out is None else out
    _check(load_library().bdlm_bwd_preprocess(_ptr(O), _dt(O.dtype), _ptr(dO), rows, H, d, _ptr(D), _stream(stream)))
    return D


def bdlm_attn_bwd(Qc, Kc, Vc, Qn, Kn, Vn, Oc, On, dOc, dOn, LSEc, LSEn, B: int, scale: float | None = None,
                  g_dtype=None, out=None, workspace=None, stream=None):
    """Gradients of both streams.  Returns (dQc, dKc, dVc, dQn, dKn, dVn)."""
    torch = _torch()
    _check_inputs(Qc, Kc, Vc, Qn, Kn, Vn, Oc, On, dOc, dOn)
    L, Hq, Hkv, d = _shape(Qc, Kc)
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    g_dtype = torch.bfloat16 if g_dtype is None else g_dtype
    if out is None:
        mk = lambda H: torch.empty((L, H, d), dtype=g_dtype, device=Qc.device)
        out = (mk(Hq), mk(Hkv), mk(Hkv), mk(Hq), mk(Hkv), mk(Hkv))
    dQc, dKc, dVc, dQn, dKn, dVn = out
    ws = _workspace(OP_BWD, L, B, Hq, Hkv, d, Qc.device, workspace)
    _check(load_library().bdlm_attn_bwd(
        _ptr(Qc), _ptr(Kc), _ptr(Vc), _ptr(Qn), _ptr(Kn), _ptr(Vn), _ptr(Oc), _ptr(On), _ptr(dOc), _ptr(dOn),
        _ptr(LSEc), _ptr(LSEn), L, B, Hq, Hkv, d, scale, _ptr(dQc), _ptr(dKc), _ptr(dVc), _ptr(dQn), _ptr(dKn),
        _ptr(dVn), _dt(g_dtype), _ptr(ws), ws.numel(), _stream(stream)))
    return out


def bdlm_attn_bwd_noalloc(Qc, Kc, Vc, Qn, Kn, Vn, Oc, On, dOc, dOn, LSEc, LSEn, B: int,
                          scale: float | None = None, g_dtype=None, out=None, stream=None,
                          check_status: bool = True):
    """bdlm_attn_bwd without a workspace argument, for callers that cannot
    allocate device memory: the library uses its own fixed-size device array
    (Hq * L <= 4194272).  With ``check_status`` (the default) the call waits
    for the stream and raises BdlmError(BDLM_ERR_TIMEOUT) if a kernel gave up
    on a device wait (``bdlm_sync_status_noalloc``); pass False to keep the
    call asynchronous and check later.  Returns (dQc, dKc, dVc, dQn, dKn, dVn)."""
    torch = _torch()
    _check_inputs(Qc, Kc, Vc, Qn, Kn, Vn, Oc, On, dOc, dOn)
    L, Hq, Hkv, d = _shape(Qc, Kc)
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    g_dtype = torch.bfloat16 if g_dtype is None else g_dtype
    if out is None:
        mk = lambda H: torch.empty((L, H, d), dtype=g_dtype, device=Qc.device)
        out = (mk(Hq), mk(Hkv), mk(Hkv), mk(Hq), mk(Hkv), mk(Hkv))
    dQc, dKc, dVc, dQn, dKn, dVn = out
    _check(load_library().bdlm_attn_bwd_noalloc(
        _ptr(Qc), _ptr(Kc), _ptr(Vc), _ptr(Qn), _ptr(Kn), _ptr(Vn), _ptr(Oc), _ptr(On), _ptr(dOc), _ptr(dOn),
        _ptr(LSEc), _ptr(LSEn), L, B, Hq, Hkv, d, scale, _ptr(dQc), _ptr(dKc), _ptr(dVc), _ptr(dQn), _ptr(dKn),
        _ptr(dVn), _dt(g_dtype), _stream(stream)))
    if check_status:
        bdlm_sync_status_noalloc(stream)
    return out


def bdlm_attn_bwd_shard(Qc, Kc, Vc, Qn, Kn, Vn, dOc, dOn, LSEc, LSEn, Dc, Dn, B: int, kv_begin: int,
                        kv_end: int, include_local: bool, dQc_acc, dQn_acc, dKc, dVc, dKn, dVn,
                        scale: float | None = None, workspace=None, stream=None):
    """One shard's gradient contribution (fp32): writes dK/dV rows of the
    shard's keys, accumulates dQ into dQc_acc / dQn_acc."""
    _check_inputs(Qc, Kc, Vc, Qn, Kn, Vn, dOc, dOn)
    L, Hq, Hkv, d = _shape(Qc, Kc)
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    ws = _workspace(OP_BWD_SHARD, L, B, Hq, Hkv, d, Qc.device, workspace)
    _check(load_library().bdlm_attn_bwd_shard(
        _ptr(Qc), _ptr(Kc), _ptr(Vc), _ptr(Qn), _ptr(Kn), _ptr(Vn), _ptr(dOc), _ptr(dOn), _ptr(LSEc), _ptr(LSEn),
        _ptr(Dc), _ptr(Dn), L, B, Hq, Hkv, d, scale, kv_begin, kv_end, int(bool(include_local)),
        _ptr(dQc_acc), _ptr(dQn_acc), _ptr(dKc), _ptr(dVc), _ptr(dKn), _ptr(dVn), _ptr(ws), ws.numel(),
        _stream(stream)))


def bdlm_attn_fwd_shard_rows(Qc, Kc, Vc, Qn, Kn, Vn, B: int, kv_begin: int, kv_end: int, include_local: bool,
                             rows_c, rows_n, scale: float | None = None, out=None, workspace=None, stream=None):
    """One rank's rows of the partial forward: clean rows ``rows_c`` =
    (begin, end) and corrupted rows ``rows_n``, against clean keys
    [kv_begin, kv_end) (+ the rows' own corrupted blocks if include_local).
    Only those rows of the fp32 outputs are written.  Returns
    (Op_c, Op_n, LSEp_c, LSEp_n)."""
    torch = _torch()
    _check_inputs(Qc, Kc, Vc, Qn, Kn, Vn)
    L, Hq, Hkv, d = _shape(Qc, Kc)
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    if out is None:
        out = (torch.zeros((L, Hq, d), dtype=torch.float32, device=Qc.device),
               torch.zeros((L, Hq, d), dtype=torch.float32, device=Qc.device),
               torch.full((Hq, L), float("-inf"), dtype=torch.float32, device=Qc.device),
               torch.full((Hq, L), float("-inf"), dtype=torch.float32, device=Qc.device))
    ws = _workspace(OP_FWD_SHARD, L, B, Hq, Hkv, d, Qc.device, workspace)
    _check(load_library().bdlm_attn_fwd_shard_rows(
        _ptr(Qc), _ptr(Kc), _ptr(Vc), _ptr(Qn), _ptr(Kn), _ptr(Vn), L, B, Hq, Hkv, d, scale,
        kv_begin, kv_end, int(bool(include_local)), int(rows_c[0]), int(rows_c[1]), int(rows_n[0]), int(rows_n[1]),
        *[_ptr(t) for t in out], _ptr(ws), ws.numel(), _stream(stream)))
    return out


def bdlm_attn_bwd_shard_rows(Qc, Kc, Vc, Qn, Kn, Vn, dOc, dOn, LSEc, LSEn, Dc, Dn, B: int, kv_begin: int,
                             kv_end: int, include_local: bool, rows_c, rows_n, dQc_acc, dQn_acc, dKc_acc, dVc_acc,
                             dKn_acc, dVn_acc, scale: float | None = None, workspace=None, stream=None):
    """One rank's rows of the sharded backward: adds the rows' dQ and their
    contributions to the call's keys' dK, dV into the fp32 accumulators."""
    _check_inputs(Qc, Kc, Vc, Qn, Kn, Vn, dOc, dOn)
    L, Hq, Hkv, d = _shape(Qc, Kc)
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    ws = _workspace(OP_BWD_SHARD, L, B, Hq, Hkv, d, Qc.device, workspace)
    _check(load_library().bdlm_attn_bwd_shard_rows(
        _ptr(Qc), _ptr(Kc), _ptr(Vc), _ptr(Qn), _ptr(Kn), _ptr(Vn), _ptr(dOc), _ptr(dOn), _ptr(LSEc), _ptr(LSEn),
        _ptr(Dc), _ptr(Dn), L, B, Hq, Hkv, d, scale, kv_begin, kv_end, int(bool(include_local)),
        int(rows_c[0]), int(rows_c[1]), int(rows_n[0]), int(rows_n[1]),
        _ptr(dQc_acc), _ptr(dQn_acc), _ptr(dKc_acc), _ptr(dVc_acc), _ptr(dKn_acc), _ptr(dVn_acc),
        _ptr(ws), ws.numel(), _stream(stream)))


def _held(t, n, name):
    """A rank-local tensor must hold exactly n rows."""
    if t.shape[0] != n:
        raise ValueError(f"{name} holds {t.shape[0]} rows, the call's range has {n}")


def _ptr_held(t, spare):
    """A tensor with no rows is not read: a spare buffer stands in for its (null) address."""
    return _ptr(t) if t.numel() > 0 else _ptr(spare)


def bdlm_attn_fwd_rank(Qc, Kc, Vc, Qn, Kn, Vn, L: int, B: int, kv_begin: int, kv_end: int, include_local: bool,
                       rows_c, rows_n, scale: float | None = None, out=None, workspace=None, stream=None):
    """One rank's rows with rank-local tensors: Qc holds clean rows
    ``rows_c`` = (begin, end) only, Qn / Kn / Vn the corrupted rows
    ``rows_n`` only, Kc / Vc the clean keys [kv_begin, kv_end) only; L is the
    full length.  Returns the partial (Op_c, Op_n, LSEp_c, LSEp_n) of those
    rows (fp32, [rows, Hq, d] and [Hq, rows])."""
    torch = _torch()
    _check_inputs(Qc, Kc, Vc, Qn, Kn, Vn)
    nc, nn = rows_c[1] - rows_c[0], rows_n[1] - rows_n[0]
    for t, n, name in ((Qc, nc, "Qc"), (Qn, nn, "Qn"), (Kn, nn, "Kn"), (Vn, nn, "Vn"),
                       (Kc, kv_end - kv_begin, "Kc"), (Vc, kv_end - kv_begin, "Vc")):
        _held(t, n, name)
    Hq, d, Hkv = Qc.shape[1], Qc.shape[2], Kn.shape[1]
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    dev = Qc.device
    if out is None:
        out = (torch.zeros((nc, Hq, d), dtype=torch.float32, device=dev),
               torch.zeros((nn, Hq, d), dtype=torch.float32, device=dev),
               torch.full((Hq, nc), float("-inf"), dtype=torch.float32, device=dev),
               torch.full((Hq, nn), float("-inf"), dtype=torch.float32, device=dev))
    ws = _workspace(OP_FWD_SHARD, L, B, Hq, Hkv, d, dev, workspace)
    spare = torch.empty(256, dtype=torch.uint8, device=dev)
    _check(load_library().bdlm_attn_fwd_rank(
        *[_ptr_held(t, spare) for t in (Qc, Kc, Vc, Qn, Kn, Vn)], L, B, Hq, Hkv, d, scale, kv_begin, kv_end,
        int(bool(include_local)), int(rows_c[0]), int(rows_c[1]), int(rows_n[0]), int(rows_n[1]),
        *[_ptr_held(t, spare) for t in out], _ptr(ws), ws.numel(), _stream(stream)))
    return out


def bdlm_attn_bwd_rank(Qc, Kc, Vc, Qn, Kn, Vn, dOc, dOn, LSEc, LSEn, Dc, Dn, L: int, B: int, kv_begin: int,
                       kv_end: int, include_local: bool, rows_c, rows_n, dQc_acc, dQn_acc, dKc_acc, dVc_acc,
                       dKn_acc, dVn_acc, scale: float | None = None, workspace=None, stream=None):
    """One rank's rows of the backward with rank-local tensors (as
    bdlm_attn_fwd_rank; LSE, D of its rows as [Hq, rows]): adds the rows' dQ
    and their contributions to the call's keys' dK, dV into the fp32
    accumulators ([rows, Hq, d] for dQ, [keys, Hkv, d] for dK / dV)."""
    torch = _torch()
    _check_inputs(Qc, Kc, Vc, Qn, Kn, Vn, dOc, dOn)
    nc, nn, nk = rows_c[1] - rows_c[0], rows_n[1] - rows_n[0], kv_end - kv_begin
    for t, n, name in ((Qc, nc, "Qc"), (dOc, nc, "dOc"), (dQc_acc, nc, "dQc_acc"), (Qn, nn, "Qn"), (Kn, nn, "Kn"),
                       (Vn, nn, "Vn"), (dOn, nn, "dOn"), (dQn_acc, nn, "dQn_acc"), (dKn_acc, nn, "dKn_acc"),
                       (dVn_acc, nn, "dVn_acc"), (Kc, nk, "Kc"), (Vc, nk, "Vc"), (dKc_acc, nk, "dKc_acc"),
                       (dVc_acc, nk, "dVc_acc")):
        _held(t, n, name)
    Hq, d, Hkv = Qc.shape[1], Qc.shape[2], Kn.shape[1]
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    dev = Qc.device
    ws = _workspace(OP_BWD_SHARD, L, B, Hq, Hkv, d, dev, workspace)
    spare = torch.empty(256, dtype=torch.uint8, device=dev)
    ts = (Qc, Kc, Vc, Qn, Kn, Vn, dOc, dOn, LSEc, LSEn, Dc, Dn)
    acc = (dQc_acc, dQn_acc, dKc_acc, dVc_acc, dKn_acc, dVn_acc)
    _check(load_library().bdlm_attn_bwd_rank(
        *[_ptr_held(t, spare) for t in ts], L, B, Hq, Hkv, d, scale, kv_begin, kv_end, int(bool(include_local)),
        int(rows_c[0]), int(rows_c[1]), int(rows_n[0]), int(rows_n[1]), *[_ptr_held(t, spare) for t in acc],
        _ptr(ws), ws.numel(), _stream(stream)))


def bdlm_worklist(L: int, B: int, Hq: int, Hkv: int, tile_q: int = 256, tile_k: int = 128,
                  kv_begin: int = 0, kv_end: int | None = None, include_local: bool = True):
    """The forward work list as a list of 8-tuples (host only, no GPU)."""
    kv_end = L if kv_end is None else kv_end
    lib = load_library()
    n = lib.bdlm_worklist(L, B, Hq, Hkv, tile_q, tile_k, kv_begin, kv_end, int(include_local), None, 0)
    if n < 0:
        raise BdlmError(2, "invalid work-list shape")
    buf = (ctypes.c_int32 * (8 * n))()
    lib.bdlm_worklist(L, B, Hq, Hkv, tile_q, tile_k, kv_begin, kv_end, int(include_local),
                      ctypes.cast(buf, ctypes.c_void_p), n)
    return [tuple(buf[8 * i:8 * i + 8]) for i in range(n)]


def _offsets(seq_lens):
    """Host int64 array of the n + 1 row offsets of packed sequences."""
    lens = [int(x) for x in seq_lens]
    arr = (ctypes.c_int64 * (len(lens) + 1))()
    acc = 0
    for i, n in enumerate(lens):
        arr[i] = acc
        acc += n
    arr[len(lens)] = acc
    return arr, len(lens), acc


def bdlm_workspace_size_varlen(op: int, seq_lens, Hq: int, Hkv: int, d: int) -> int:
    arr, n, _ = _offsets(seq_lens)
    return load_library().bdlm_workspace_size_varlen(op, ctypes.cast(arr, ctypes.c_void_p), n, Hq, Hkv, d)


def _workspace_varlen(op, seq_lens, Hq, Hkv, d, device, ws):
    torch = _torch()
    need = bdlm_workspace_size_varlen(op, seq_lens, Hq, Hkv, d)
    if ws is None:
        ws = torch.empty(max(need, 256), dtype=torch.uint8, device=device)
    return ws


def bdlm_attn_fwd_varlen(Qc, Kc, Vc, Qn, Kn, Vn, seq_lens, B: int, scale: float | None = None, o_dtype=None,
                         out=None, workspace=None, stream=None):
    """Packed batch: sequences of the given lengths stored back to back along
    the token dimension ([T, H, d], T = sum of the lengths).  Returns
    (Oc, On, LSEc, LSEn) with LSE as [Hq, T]."""
    torch = _torch()
    _check_inputs(Qc, Kc, Vc, Qn, Kn, Vn)
    T, Hq, Hkv, d = _shape(Qc, Kc)
    arr, n, tot = _offsets(seq_lens)
    if tot != T:
        raise ValueError(f"sequence lengths sum to {tot}, tensors hold {T} rows")
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    o_dtype = torch.bfloat16 if o_dtype is None else o_dtype
    if out is None:
        out = (torch.empty((T, Hq, d), dtype=o_dtype, device=Qc.device),
               torch.empty((T, Hq, d), dtype=o_dtype, device=Qc.device),
               torch.empty((Hq, T), dtype=torch.float32, device=Qc.device),
               torch.empty((Hq, T), dtype=torch.float32, device=Qc.device))
    Oc, On, LSEc, LSEn = out
    ws = _workspace_varlen(OP_FWD, seq_lens, Hq, Hkv, d, Qc.device, workspace)
    _check(load_library().bdlm_attn_fwd_varlen(
        _ptr(Qc), _ptr(Kc), _ptr(Vc), _ptr(Qn), _ptr(Kn), _ptr(Vn), ctypes.cast(arr, ctypes.c_void_p), n, B,
        Hq, Hkv, d, scale, _ptr(Oc), _ptr(On), _dt(Oc.dtype), _ptr(LSEc), _ptr(LSEn), _ptr(ws), ws.numel(),
        _stream(stream)))
    return Oc, On, LSEc, LSEn


def bdlm_attn_bwd_varlen(Qc, Kc, Vc, Qn, Kn, Vn, Oc, On, dOc, dOn, LSEc, LSEn, seq_lens, B: int,
                         scale: float | None = None, g_dtype=None, out=None, workspace=None, stream=None):
    """Gradients of a packed batch.  Returns (dQc, dKc, dVc, dQn, dKn, dVn)."""
    torch = _torch()
    _check_inputs(Qc, Kc, Vc, Qn, Kn, Vn, dOc, dOn)
    T, Hq, Hkv, d = _shape(Qc, Kc)
    arr, n, tot = _offsets(seq_lens)
    if tot != T:
        raise ValueError(f"sequence lengths sum to {tot}, tensors hold {T} rows")
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    g_dtype = torch.bfloat16 if g_dtype is None else g_dtype
    if out is None:
        mk = lambda H: torch.empty((T, H, d), dtype=g_dtype, device=Qc.device)
        out = (mk(Hq), mk(Hkv), mk(Hkv), mk(Hq), mk(Hkv), mk(Hkv))
    dQc, dKc, dVc, dQn, dKn, dVn = out
    ws = _workspace_varlen(OP_BWD, seq_lens, Hq, Hkv, d, Qc.device, workspace)
    _check(load_library().bdlm_attn_bwd_varlen(
        _ptr(Qc), _ptr(Kc), _ptr(Vc), _ptr(Qn), _ptr(Kn), _ptr(Vn), _ptr(Oc), _ptr(On), _ptr(dOc), _ptr(dOn),
        _ptr(LSEc), _ptr(LSEn), ctypes.cast(arr, ctypes.c_void_p), n, B, Hq, Hkv, d, scale,
        _ptr(dQc), _ptr(dKc), _ptr(dVc), _ptr(dQn), _ptr(dKn), _ptr(dVn), _dt(dQc.dtype), _ptr(ws), ws.numel(),
        _stream(stream)))
    return out


def bdlm_sync_status(workspace, stream=None):
    """Synchronises and raises BdlmError(BDLM_ERR_TIMEOUT) if a kernel's
    bounded wait expired since the last call on this workspace."""
    _check(load_library().bdlm_sync_status(_ptr(workspace), _stream(stream)))


def bdlm_sync_status_noalloc(stream=None):
    """Synchronises and raises BdlmError(BDLM_ERR_TIMEOUT) if a kernel of an
    allocation-free call gave up on a device wait since the last check."""
    _check(load_library().bdlm_sync_status_noalloc(_stream(stream)))


def bdlm_watchdog_selftest_noalloc(limit_us: int = 20000, stream=None) -> int:
    """The watchdog self-test on the allocation-free array's status word;
    returns the status code (7 = the wait ran out and was reported)."""
    return int(load_library().bdlm_watchdog_selftest_noalloc(limit_us, _stream(stream)))


def bdlm_watchdog_selftest(workspace, limit_us: int = 20000, stream=None) -> int:
    """Runs the watchdog self-test; returns the status code (7 = the bounded
    wait expired and was reported, the expected outcome)."""
    return int(load_library().bdlm_watchdog_selftest(_ptr(workspace), workspace.numel(), limit_us,
                                                      _stream(stream)))
