"""The allocation-free backward entry point.

bdlm_attn_bwd_noalloc exists for callers that cannot allocate device memory
(plugin hosts that only pass inputs and outputs, runtimes that reserve all
device memory up front, latency-critical code that avoids cudaMalloc).  It
runs the ordinary backward with its workspace in a fixed array of device
memory the library declares.  This file is collected last so that a run that
stops at the first failure has already run every other test.
"""
from __future__ import annotations

import math

import pytest

from structured_mask_attention_gb300.inputs import make_numpy
from tests.parity_util import check_rel, to_dev, to_np

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

NAMES = ("Qc", "Kc", "Vc", "Qn", "Kn", "Vn")


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import structured_mask_attention_gb300 as m
    m.load_library()
    return m


def test_noalloc_backward_matches_workspace_backward(lib):
    """Two allocation-free calls in a row give the same gradients as the
    ordinary backward with a caller workspace.  Both run the same
    deterministic kernels on the same inputs, so the results are bitwise
    equal (which also meets the parity tolerance); the second call reuses
    the array the first one left behind."""
    m = lib
    L, B, Hq, Hkv, d = 1280, 128, 4, 2, 128
    X = make_numpy(L, Hq, Hkv, d, seed=31)
    dev = {k: to_dev(v, torch) for k, v in X.items()}
    ins = [dev[k] for k in NAMES]
    sc = 1.0 / math.sqrt(d)
    Oc, On, LSEc, LSEn = m.bdlm_attn_fwd(*ins, B, sc)
    ref = m.bdlm_attn_bwd(*ins, Oc, On, dev["dOc"], dev["dOn"], LSEc, LSEn, B, sc, g_dtype=torch.float32)
    names = ("dQc", "dKc", "dVc", "dQn", "dKn", "dVn")
    for call in range(2):
        got = m.bdlm_attn_bwd_noalloc(*ins, Oc, On, dev["dOc"], dev["dOn"], LSEc, LSEn, B, sc,
                                      g_dtype=torch.float32)
        torch.cuda.synchronize()
        for name, g, r in zip(names, got, ref):
            check_rel(f"{name} (call {call})", to_np(g), to_np(r))
            assert torch.equal(g, r), f"{name} (call {call}) differs from the workspace backward"


def test_noalloc_status_word_reports_a_device_timeout(lib):
    """A device wait that runs out while using the allocation-free array is
    reported through bdlm_sync_status_noalloc (a wait nobody ends, limited to
    20 ms); the status word is cleared after the report, so the next
    allocation-free backward checks clean."""
    m = lib
    assert m.bdlm_watchdog_selftest_noalloc(20000) == 7
    m.bdlm_sync_status_noalloc()  # cleared by the report
    L, B, Hq, Hkv, d = 256, 64, 2, 1, 64
    X = make_numpy(L, Hq, Hkv, d, seed=5)
    dev = {k: to_dev(v, torch) for k, v in X.items()}
    ins = [dev[k] for k in NAMES]
    f = m.bdlm_attn_fwd(*ins, B)
    m.bdlm_attn_bwd_noalloc(*ins, f[0], f[1], dev["dOc"], dev["dOn"], f[2], f[3], B, check_status=True)


def test_noalloc_rejects_shapes_beyond_the_array(lib):
    m = lib
    # 8 * Hq * L + 256 bytes exceed the 32 MiB array; rejected before any launch
    # (null pointers would also be rejected, so nothing can reach the device)
    st = m.load_library().bdlm_attn_bwd_noalloc(*([None] * 12), 1 << 20, 1024, 8, 4, 128, 0.088,
                                                *([None] * 6), 0, None)
    assert st == 4
    assert "4194272" in m.bdlm_last_error()
