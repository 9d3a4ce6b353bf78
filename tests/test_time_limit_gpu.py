"""GPU tests of the kernels' time limits, without a fault.

The library's one-shot test switch makes the next call's TMA producer issue no
loads, so the consumers' bounded waits find a barrier that nothing completes.
After the 2 s limit the kernel must wind down by itself: active rows come back
NaN (argmax -1), inactive rows keep their defined values, nothing faults, and
the very next call on the same context is correct again.
"""
import time

import numpy as np
import pytest
import torch

from parity import check_dh, check_fwd, gpu_fwd, to_dev
from verify_vocab_blocked_gb300 import build as qbuild
from verify_vocab_blocked_gb300 import qhead, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    qbuild.build()
    qhead.lib()


def _workload(M, H, V, bits, cap, seed, mask=None):
    head = synth.make_head(V, H, bits, softcap=cap, seed=seed)
    h = synth.make_hidden(M, H, seed=seed)
    t = synth.make_targets(M, V, seed=seed)
    g = synth.make_dlogp(M, seed=seed)
    return synth.Workload("custom", head, h, t, mask, g, dict(M=M, H=H, V=V, bits=bits))


def _stalled_fwd(wl):
    head, h, t, mk, _ = to_dev(wl)
    torch.cuda.synchronize()
    t0 = time.monotonic()
    qhead.test_stall_next_call(True)
    logp, lse, am = gpu_fwd(head, h, t, mk)
    return time.monotonic() - t0, logp, lse, am


def _assert_poisoned_fwd(wl, logp, lse, am):
    act = np.ones(wl.M, bool) if wl.mask is None else wl.mask.astype(bool)
    assert act.any()
    assert np.all(np.isnan(lse[act])) and np.all(np.isnan(logp[act]))
    assert np.all(am[act] == -1)
    assert np.all(lse[~act] == 0.0) and np.all(logp[~act] == 0.0) and np.all(am[~act] == -1)


@pytest.mark.parametrize("M,H,V,bits,cap,masked", [
    (5, 256, 3000, 4, 30.0, False),    # weight-streaming kernel (scales by cp.async)
    (5, 2560, 1200, 4, 30.0, False),   # weight-streaming kernel, TMA-staged scales
    (200, 256, 2000, 8, 0.0, True),    # tensor-core kernel, some rows inactive
    (300, 512, 3000, 4, 30.0, True),   # tensor-core kernel, TMA-staged scale and bias boxes
])
def test_forward_wait_expires_then_recovers(M, H, V, bits, cap, masked):
    mask = synth.make_mask(M, 16, 0.3) if masked else None
    wl = _workload(M, H, V, bits, cap, seed=M + V, mask=mask)
    took, logp, lse, am = _stalled_fwd(wl)
    assert took >= 1.5, f"call ended after {took:.2f} s: the waits did not run to their limit"
    assert took < 60.0
    _assert_poisoned_fwd(wl, logp, lse, am)
    # The switch is one-shot and the context is intact: the next call is exact.
    head, h, t, mk, _ = to_dev(wl)
    logp, lse, am = gpu_fwd(head, h, t, mk)
    check_fwd(wl, np.arange(wl.M), logp, lse, am)


@pytest.mark.parametrize("M", [160, 5])  # every M runs the pipelined tensor-core backward
def test_backward_wait_expires_then_recovers(M):
    mask = synth.make_mask(M, 16, 0.3) if M > 16 else None
    wl = _workload(M, 256, 2500, 4, 30.0, seed=41, mask=mask)
    head, h, t, mk, g = to_dev(wl)
    logp, lse, am = gpu_fwd(head, h, t, mk)
    check_fwd(wl, np.arange(M), logp, lse, am)
    lse_d = torch.from_numpy(lse).cuda()
    qhead.test_stall_next_call(True)
    dh = qhead.bwd(head, h, t, lse_d, g, mk)
    torch.cuda.synchronize()
    dh = dh.cpu().numpy()
    act = mask.astype(bool) if mask is not None else np.ones(M, bool)
    assert np.all(np.isnan(dh[act]))
    assert np.all(dh[~act] == 0.0)
    dh = qhead.bwd(head, h, t, lse_d, g, mk)
    torch.cuda.synchronize()
    check_dh(wl, np.arange(M), dh.cpu().numpy())


def test_disarmed_switch_has_no_effect():
    wl = _workload(70, 128, 900, 4, 0.0, seed=5)
    qhead.test_stall_next_call(True)
    qhead.test_stall_next_call(False)
    head, h, t, mk, _ = to_dev(wl)
    logp, lse, am = gpu_fwd(head, h, t, mk)
    check_fwd(wl, np.arange(wl.M), logp, lse, am)


def test_head_gradient_wait_expires_then_recovers():
    M = 150
    mask = synth.make_mask(M, 16, 0.3)
    wl = _workload(M, 256, 2200, 4, 30.0, seed=43, mask=mask)
    head, h, t, mk, g = to_dev(wl)
    lse = qhead.fwd(head, h, t, mk)[1]
    qhead.test_stall_next_call(True)
    _, dw = qhead.bwd_dw(head, h, t, lse, g, mk)
    torch.cuda.synchronize()
    assert torch.isnan(dw).all()
    _, dw = qhead.bwd_dw(head, h, t, lse, g, mk)
    torch.cuda.synchronize()
    assert torch.isfinite(dw).all()
