"""The blockMax early exit (qhead_fwd_blockmax, qhead_bwd_blockskip) against
the oracle.

* block_max: every active row's per-tile maximum of z within 2e-3 of the
  oracle's, plus 2e-4 |z| (the peaked rows' logits reach ~40, where the fp16
  weights' relative error shows in absolute terms); masked rows untouched;
* eps = 0 is the exact backward, bit for bit;
* on peaked synthetic data (a few hot vocab rows dominate every softmax,
  most targets are hot), the approximate dh matches the oracle's approximate
  dh -- which takes its skip decisions from the same block_max and lse --
  and the exact dh the exact oracle, both within the 2e-3 dh tolerance
  measured against the terms (the "peaked" cancellation case of the parity
  rule), and the approximate dh lies within |dlogp| * eps * sum_v |w_v| plus
  that tolerance of the exact one.
"""
import numpy as np
import pytest
import torch

import oracle
from parity import DH_REL_TOL, LSE_TOL, oracle_head, to_dev
from verify_vocab_blocked_gb300 import build as qbuild
from verify_vocab_blocked_gb300 import qhead, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    qbuild.build()
    qhead.lib()


def _peaked(M, H, V, bits, cap, seed, hot_frac=0.9, mask=None, bias_shift=0.3, sb_dtype="f16"):
    head, hot = synth.make_peaked_head(V, H, bits, n_hot=8, bias_shift=bias_shift, softcap=cap,
                                       seed=seed, sb_dtype=sb_dtype)
    h = synth.make_hidden(M, H, seed=seed, mean=0.5)
    t = synth.make_targets(M, V, seed=seed)
    rng = np.random.default_rng(seed)
    pick = rng.random(M) < hot_frac
    t[pick] = hot[rng.integers(0, len(hot), size=int(pick.sum()))]
    g = rng.uniform(-2.0, 2.0, size=M).astype(np.float32)
    return synth.Workload("peaked", head, h, t, mask, g, {})


def _rel_rows(got, ref, scale):
    return np.linalg.norm(got - ref, axis=1) / np.maximum(scale, 1e-30)


@pytest.mark.parametrize("M,H,V,bits,cap,masked", [
    (200, 256, 20000, 4, 30.0, True),
    (40, 256, 9000, 8, 0.0, False),   # below the tensor-core threshold
])
def test_block_max_matches_oracle(M, H, V, bits, cap, masked):
    mask = synth.make_mask(M, 20, 0.3) if masked else None
    wl = _peaked(M, H, V, bits, cap, seed=M + V, mask=mask)
    head, h, t, mk, g = to_dev(wl)
    logp, lse, am, bm = qhead.fwd_blockmax(head, h, t, mk)
    torch.cuda.synchronize()
    ref = oracle.block_max(wl.h, oracle_head(wl.head), mask=wl.mask)
    act = np.ones(M, bool) if mask is None else mask.astype(bool)
    bm = bm.cpu().numpy()
    # The peaked rows' logits reach ~40 (no cap): the fp16 weights' relative
    # error then shows in absolute terms, so the bound grows with |z|.
    assert (np.abs(bm[act] - ref[act]) <= LSE_TOL + 2e-4 * np.abs(ref[act])).all()
    assert np.isneginf(bm[~act]).all()
    f = oracle.forward(wl.h, oracle_head(wl.head), wl.targets, wl.mask)
    lse_g = lse.cpu().numpy()[act]
    assert (np.abs(lse_g - f.lse[act]) <= LSE_TOL + 2e-4 * np.abs(f.lse[act])).all()


def test_eps_zero_is_the_exact_backward():
    wl = _peaked(300, 256, 12000, 4, 30.0, seed=51, mask=synth.make_mask(300, 50, 0.2))
    head, h, t, mk, g = to_dev(wl)
    _, lse, _, bm = qhead.fwd_blockmax(head, h, t, mk)
    exact = qhead.bwd(head, h, t, lse, g, mk)
    approx = qhead.bwd_blockskip(head, h, t, lse, g, bm, 0.0, mk)
    torch.cuda.synchronize()
    assert torch.equal(exact, approx)


@pytest.mark.parametrize("M,H,V,bits,cap,eps,sbt", [
    (300, 256, 20000, 4, 30.0, 1e-6, "f16"),
    (170, 384, 15000, 8, 0.0, 1e-5, "f16"),
    (20, 256, 9000, 4, 30.0, 1e-6, "f16"),   # a 20-row batch
    (260, 256, 12000, 4, 30.0, 1e-6, "bf16"),
    (150, 384, 9000, 8, 0.0, 1e-5, "f32"),
])
def test_peaked_blockskip(M, H, V, bits, cap, eps, sbt):
    mask = synth.make_mask(M, 20, 0.25)
    wl = _peaked(M, H, V, bits, cap, seed=M * 3 + V, mask=mask, sb_dtype=sbt)
    head, h, t, mk, g = to_dev(wl)
    _, lse, _, bm = qhead.fwd_blockmax(head, h, t, mk)
    approx = qhead.bwd_blockskip(head, h, t, lse, g, bm, eps, mk)
    exact = qhead.bwd(head, h, t, lse, g, mk)
    torch.cuda.synchronize()
    approx, exact = approx.cpu().numpy().astype(np.float64), exact.cpu().numpy().astype(np.float64)
    oh = oracle_head(wl.head)
    lse_n, bm_n = lse.cpu().numpy().astype(np.float64), bm.cpu().numpy().astype(np.float64)
    # the oracle's own lse for the coefficients; the GPU's bm and lse for the
    # skip decisions (both sides drop the same blocks)
    ref_approx = oracle.backward_blockskip(wl.h, oh, wl.targets, wl.dlogp.astype(np.float64),
                                           bm_n, eps, mask=wl.mask, lse_decide=lse_n)
    ref_exact = oracle.backward(wl.h, oh, wl.targets, wl.dlogp.astype(np.float64), mask=wl.mask)
    act = mask.astype(bool)
    assert (approx[~act] == 0.0).all()
    # the dh scale of the "peaked" cancellation case of the parity rule:
    # max(|dh|, |dlogp| |w_target|) (the hot targets hold most of the mass)
    w = oracle.dequant(oh)
    scale = np.maximum(np.linalg.norm(ref_exact, axis=1),
                       np.abs(wl.dlogp) * np.linalg.norm(w[wl.targets], axis=1))
    rel_exact = _rel_rows(exact[act], ref_exact[act], scale[act])
    rel = _rel_rows(approx[act], ref_approx[act], scale[act])
    print(f"peaked blockskip: exact path {rel_exact.max():.3e}, approximate {rel.max():.3e}")
    assert rel_exact.max() <= DH_REL_TOL, f"exact dh rel-L2 {rel_exact.max():.3e}"
    assert rel.max() <= DH_REL_TOL, f"approx dh rel-L2 {rel.max():.3e}"
    bound = np.abs(wl.dlogp[act]) * eps * np.linalg.norm(w, axis=1).sum()
    diff = np.linalg.norm(approx[act] - ref_exact[act], axis=1)
    assert (diff <= bound + DH_REL_TOL * scale[act]).all()


def test_skipping_changes_the_result():
    # A milder peak: the non-hot probabilities (~1e-6 .. 1e-5) survive the fp16
    # coefficients but lie below eps = 1e-4, so the skipped blocks' terms were
    # nonzero in the exact backward.
    M, V = 200, 16000
    wl = _peaked(M, 256, V, 4, 30.0, seed=61, bias_shift=0.1)
    head, h, t, mk, g = to_dev(wl)
    _, lse, _, bm = qhead.fwd_blockmax(head, h, t, mk)
    approx = qhead.bwd_blockskip(head, h, t, lse, g, bm, 1e-4, mk)
    exact = qhead.bwd(head, h, t, lse, g, mk)
    torch.cuda.synchronize()
    d = (approx - exact).abs().max().item()
    assert d > 0.0
    w = oracle.dequant(oracle_head(wl.head))
    bound = float(np.abs(wl.dlogp).max()) * 1e-4 * float(np.linalg.norm(w, axis=1).sum())
    assert d <= bound
