"""The head gradient (qhead_bwd_dw) against the oracle's grad_head.

Every vocab row of dW must be within 2e-3 (rel-L2) of the oracle, measured
against the larger of the row's norm and the size of its terms,
sum_m |dlogp_m| (onehot + p) sech2 |h_m| (rows with no target are sums of
small softmax terms of both signs; the GPU rounds each term's coefficient and
h once to fp16).  Shapes cover 256- and 128-column tiles, 4 and 8 bits, the
soft cap on and off, a masked batch, rows sharing a target, several vocab
chunks, a 5-row batch, bf16 and fp32 scales and biases, and a batch with no
active row.
"""
import numpy as np
import pytest
import torch

import oracle
from parity import DH_REL_TOL, oracle_head, to_dev
from verify_vocab_blocked_gb300 import build as qbuild
from verify_vocab_blocked_gb300 import qhead, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    qbuild.build()
    qhead.lib()


def _workload(M, H, V, bits, cap, seed, mask=None, shared=False, sb_dtype="f16"):
    head = synth.make_head(V, H, bits, softcap=cap, seed=seed, sb_dtype=sb_dtype)
    h = synth.make_hidden(M, H, seed=seed)
    t = synth.make_targets(M, V, seed=seed)
    if shared:
        t[1::3] = t[0]  # every third row shares row 0's target
    g = np.random.default_rng(seed).uniform(-2.0, 2.0, size=M).astype(np.float32)
    return synth.Workload("dw", head, h, t, mask, g, {})


def _term_size(wl, oh):
    """sum_m |dlogp_m| (onehot + p) sech2 |h_m| per vocab row (active rows)."""
    f = oracle.forward(wl.h, oh, wl.targets, wl.mask, keep_raw=True)
    cap = wl.head.softcap
    act = np.ones(wl.M, bool) if wl.mask is None else wl.mask.astype(bool)
    raw = f.raw[act]
    th = np.tanh(raw / cap) if cap > 0 else None
    z = cap * th if cap > 0 else raw
    sech2 = 1.0 - th * th if cap > 0 else 1.0
    p = np.exp(z - f.lse[act][:, None])
    onehot = np.zeros_like(p)
    onehot[np.arange(p.shape[0]), wl.targets[act]] = 1.0
    hn = np.linalg.norm(oracle.widen_bf16(wl.h)[act], axis=1)
    w = np.abs(wl.dlogp[act].astype(np.float64)) * hn
    return ((onehot + p) * sech2 * w[:, None]).sum(axis=0)


def _check_dw(wl, dw):
    oh = oracle_head(wl.head)
    ref = oracle.grad_head(wl.h, oh, wl.targets, wl.dlogp.astype(np.float64), wl.mask)
    got = dw.astype(np.float64)
    assert np.isfinite(got).all()
    den = np.maximum(np.linalg.norm(ref, axis=1), _term_size(wl, oh))
    rel = np.linalg.norm(got - ref, axis=1) / np.maximum(den, 1e-30)
    worst = float(rel.max())
    assert worst <= DH_REL_TOL, f"dW rel-L2 {worst:.3e} at vocab row {int(rel.argmax())}"
    return worst


def _run(wl, want_dh=False):
    head, h, t, mk, g = to_dev(wl)
    lse = qhead.fwd(head, h, t, mk)[1]
    dh, dw = qhead.bwd_dw(head, h, t, lse, g, mk, want_dh=want_dh)
    torch.cuda.synchronize()
    return head, (h, t, mk, g, lse), dh, dw


@pytest.mark.parametrize("M,H,V,bits,cap,masked,shared,sbt", [
    (150, 256, 1800, 4, 30.0, True, False, "f16"),   # 256-column tiles, partial vocab unit
    (130, 384, 2100, 8, 0.0, False, True, "f16"),    # 128-column tiles, 8 bits, shared targets
    (5, 256, 3000, 4, 30.0, False, False, "f16"),    # a 5-row batch
    (70, 512, 1025, 8, 5.0, True, True, "f16"),
    (150, 256, 1800, 4, 30.0, True, True, "bf16"),
    (70, 384, 2100, 8, 5.0, False, False, "f32"),
])
def test_dw_parity(M, H, V, bits, cap, masked, shared, sbt):
    mask = synth.make_mask(M, 16, 0.3) if masked else None
    wl = _workload(M, H, V, bits, cap, seed=M + V, mask=mask, shared=shared, sb_dtype=sbt)
    _, _, _, dw = _run(wl)
    _check_dw(wl, dw.cpu().numpy())


def test_dw_several_chunks():
    # 2048 rows: chunks of 24576 vocab rows, so V = 30000 spans two (the
    # second partial); the one-hot lists cross the chunk boundary.
    wl = _workload(2048, 256, 30000, 4, 2.0, seed=31, shared=True)
    _, _, _, dw = _run(wl)
    _check_dw(wl, dw.cpu().numpy())


def test_dw_with_dh_matches_bwd_and_is_deterministic():
    wl = _workload(160, 256, 2600, 4, 30.0, seed=32, mask=synth.make_mask(160, 16, 0.3))
    head, (h, t, mk, g, lse), dh, dw = _run(wl, want_dh=True)
    dh_plain = qhead.bwd(head, h, t, lse, g, mk)
    dh2, dw2 = qhead.bwd_dw(head, h, t, lse, g, mk, want_dh=True)
    torch.cuda.synchronize()
    assert torch.equal(dh, dh_plain)
    assert torch.equal(dh, dh2) and torch.equal(dw, dw2)
    _check_dw(wl, dw.cpu().numpy())


def test_dw_no_active_row_is_zero():
    wl = _workload(100, 256, 1500, 4, 30.0, seed=33, mask=np.zeros(100, np.uint8))
    _, _, _, dw = _run(wl)
    assert torch.count_nonzero(dw).item() == 0


def test_dw_column_sums_vanish_without_cap():
    # No cap: sum_v dW[v, :] = sum_m dlogp_m (1 - sum_v p_v) h_m = 0 up to rounding.
    wl = _workload(256, 256, 4000, 4, 0.0, seed=34)
    _, _, _, dw = _run(wl)
    dw = dw.double()
    assert dw.sum(0).abs().max().item() <= 2e-3 * dw.abs().max().item()
