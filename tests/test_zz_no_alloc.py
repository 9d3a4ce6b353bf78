"""qhead_fwd_noalloc: the forward for callers that cannot allocate device memory
(engines running inside a pre-sized memory arena, plugins whose host forbids
allocation after start-up, loops that must not enter the allocator).  It runs
the same kernels on the same plan as qhead_fwd with a caller-allocated
workspace, so it must give the same results bit for bit, call after call,
although every call reuses the library's one fixed scratch array.

This file is collected last on purpose, so a run that stops at its first
failure has already run every other test.  It builds and loads the library
itself, so it also passes when run alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

from parity import to_dev
from verify_vocab_blocked_gb300 import build as qbuild
from verify_vocab_blocked_gb300 import qhead, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    qbuild.build()
    return qhead.lib()


def _workload(M, H, V, cap, seed, masked):
    head = synth.make_head(V, H, 4, softcap=cap, seed=seed)
    h = synth.make_hidden(M, H, seed=seed)
    t = synth.make_targets(M, V, seed=seed)
    mask = synth.make_mask(M, 16, 0.3) if masked else None
    return synth.Workload("noalloc", head, h, t, mask, np.ones(M, np.float32), {})


def _noalloc(L, head, h, t, mk):
    M = h.shape[0]
    dev = h.device
    logp = torch.full((M,), float("nan"), device=dev)
    lse = torch.full((M,), float("nan"), device=dev)
    am = torch.full((M,), -7, dtype=torch.int32, device=dev)
    rc = L.qhead_fwd_noalloc(ctypes.byref(head.c()), h.data_ptr(), M,
                             t.data_ptr() if t is not None else None,
                             mk.data_ptr() if mk is not None else None, logp.data_ptr(),
                             lse.data_ptr(), am.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == qhead.QHEAD_OK, qhead.last_error()
    return logp, lse, am


def _compare(a, b):
    torch.cuda.synchronize()
    for x, y in zip(a, b):  # logp, lse, argmax: identical bits
        assert torch.equal(x, y)


def test_noalloc_matches_workspace_forward_on_consecutive_calls(L):
    # Two different workloads back to back: the second call must not see
    # anything the first one left in the shared scratch.
    # The last case is the Gemma-class verify head (H = 2560, V = 262144,
    # cap 30) with 63 rows: the tensor-core forward (from 17 rows), whose
    # per-segment partials are the largest use of the scratch in these cases.
    for M, H, V, cap, seed, masked in [(5, 2560, 20000, 30.0, 1, False),
                                       (37, 1024, 7001, 0.0, 2, True),
                                       (5, 2560, 20000, 30.0, 1, False),
                                       (63, 2560, 262144, 30.0, 5, False)]:
        wl = _workload(M, H, V, cap, seed, masked)
        head, h, t, mk, _ = to_dev(wl)
        need = qhead.fwd_workspace(head, M)
        assert need <= (8 << 20)
        ws = qhead.alloc_workspace(need, h.device)
        ref = qhead.fwd(head, h, t, mk, workspace=ws)
        got1 = _noalloc(L, head, h, t, mk)
        _compare(got1, ref)
        got2 = _noalloc(L, head, h, t, mk)
        _compare(got2, ref)


def test_noalloc_rejects_more_rows_than_the_scratch_holds(L):
    wl = _workload(4096, 2560, 1000, 0.0, 3, False)
    head, h, t, mk, _ = to_dev(wl)
    assert qhead.fwd_workspace(head, 4096) > (8 << 20)
    lse = torch.zeros(4096, device="cuda")
    rc = L.qhead_fwd_noalloc(ctypes.byref(head.c()), h.data_ptr(), 4096, None, None, None,
                             lse.data_ptr(), None, None)
    assert rc == qhead.QHEAD_EINVAL
    assert "scratch" in qhead.last_error()
    torch.cuda.synchronize()
    assert float(lse.abs().max()) == 0.0  # nothing was launched


def test_rejected_call_leaves_no_hook_armed(L):
    # A call rejected by the size check ends before any kernel: the one-shot
    # stall switch armed before it must not carry over to the next call
    # (which would then come back NaN after its waits expire).
    wl = _workload(4096, 2560, 1000, 0.0, 6, False)
    head, h, t, mk, _ = to_dev(wl)
    lse = torch.zeros(4096, device="cuda")
    qhead.test_stall_next_call(True)
    rc = L.qhead_fwd_noalloc(ctypes.byref(head.c()), h.data_ptr(), 4096, None, None, None,
                             lse.data_ptr(), None, None)
    assert rc == qhead.QHEAD_EINVAL
    small = _workload(5, 256, 300, 0.0, 7, False)
    head, h, t, mk, _ = to_dev(small)
    logp, lse5, am = _noalloc(L, head, h, t, mk)
    torch.cuda.synchronize()
    assert torch.isfinite(lse5).all() and torch.isfinite(logp).all()


def test_noalloc_reports_bad_arguments(L):
    wl = _workload(5, 256, 100, 0.0, 4, False)
    head, h, t, mk, _ = to_dev(wl)
    bad = head.c()
    bad.bits = 3
    rc = L.qhead_fwd_noalloc(ctypes.byref(bad), h.data_ptr(), 5, None, None, None, None, None,
                             None)
    assert rc == qhead.QHEAD_EUNSUPPORTED
