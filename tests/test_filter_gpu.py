"""The coefficient filter (qhead_bwd_filter) against the oracle.

* eps = 0 is the exact backward, bit for bit, with no block cold;
* eps = +inf: exactly the blocks that hold no row's target are cold (a
  decision free of rounding), and dh matches the oracle's;
* on peaked synthetic data the GPU's block decisions equal the oracle's
  wherever the oracle's largest softmax term of the block lies more than 5 %
  away from eps (closer blocks may go either way: the kernel decides in fp32
  on its own logits); the approximate dh matches the oracle's approximate dh
  taken with the GPU's decisions, and the exact dh the exact oracle, both
  within the 2e-3 dh tolerance measured against the terms (the "peaked"
  cancellation case of the parity rule), and the approximate dh lies within
  eps * sum_v |w_v| plus that tolerance of the exact one; several vocab chunks, a mask,
  8-bit heads, M below the tensor-core threshold and zero cotangents;
* dropping blocks changes the result, within the bound.
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


def _active(wl):
    return np.ones(len(wl.targets), bool) if wl.mask is None else wl.mask.astype(bool)


def _run(wl, eps):
    head, h, t, mk, g = to_dev(wl)
    _, lse, _ = qhead.fwd(head, h, t, mk)
    approx, cold = qhead.bwd_filter(head, h, t, lse, g, eps, mk, want_cold=True)
    exact = qhead.bwd(head, h, t, lse, g, mk)
    torch.cuda.synchronize()
    return approx, exact, cold


def _scale(wl, ref_exact, w):
    # the dh scale of the "peaked" cancellation case of the parity rule:
    # max(|dh|, |dlogp| |w_target|) (the hot targets hold most of the mass)
    return np.maximum(np.linalg.norm(ref_exact, axis=1),
                      np.abs(wl.dlogp) * np.linalg.norm(w[wl.targets], axis=1))


def _rel_rows(got, ref, scale):
    return np.linalg.norm(got - ref, axis=1) / np.maximum(scale, 1e-30)


def test_eps_zero_is_the_exact_backward():
    wl = _peaked(300, 256, 12000, 4, 30.0, seed=71, mask=synth.make_mask(300, 50, 0.2))
    approx, exact, cold = _run(wl, 0.0)
    assert torch.equal(exact, approx)
    n_rb = (int(_active(wl).sum()) + 31) // 32
    cold = cold.cpu().numpy()
    assert (cold[:n_rb] == 0).all() and (cold[n_rb:] == 1).all()


def test_infinite_eps_keeps_exactly_the_target_blocks():
    wl = _peaked(150, 256, 9000, 4, 30.0, seed=72, mask=synth.make_mask(150, 30, 0.3))
    approx, exact, cold = _run(wl, float("inf"))
    oh = oracle_head(wl.head)
    ref, dec = oracle.backward_filter(wl.h, oh, wl.targets, wl.dlogp.astype(np.float64),
                                      float("inf"), mask=wl.mask)
    n_rb = dec.cold.shape[0]
    cold = cold.cpu().numpy().astype(bool)
    assert np.array_equal(cold[:n_rb], dec.cold)
    assert np.array_equal(dec.cold, ~dec.has_target)
    ref_exact = oracle.backward(wl.h, oh, wl.targets, wl.dlogp.astype(np.float64), mask=wl.mask)
    act = _active(wl)
    w = oracle.dequant(oh)
    scale = _scale(wl, ref_exact, w)
    exact = exact.cpu().numpy().astype(np.float64)
    rel_exact = _rel_rows(exact[act], ref_exact[act], scale[act])
    rel = _rel_rows(approx.cpu().numpy().astype(np.float64)[act], ref[act], scale[act])
    print(f"filter eps=inf: exact path {rel_exact.max():.3e}, approximate {rel.max():.3e}")
    assert rel_exact.max() <= DH_REL_TOL, f"exact dh rel-L2 {rel_exact.max():.3e}"
    assert rel.max() <= DH_REL_TOL, f"rel-L2 {rel.max():.3e}"


@pytest.mark.parametrize("M,H,V,bits,cap,eps,masked,sbt", [
    (300, 256, 20000, 4, 30.0, 1e-6, True, "f16"),
    (170, 384, 15000, 8, 0.0, 1e-5, True, "f16"),
    (20, 256, 9000, 4, 30.0, 1e-6, False, "f16"),     # a 20-row batch
    (3200, 128, 33000, 4, 30.0, 1e-6, False, "f16"),  # three vocab chunks
    (260, 256, 12000, 4, 30.0, 1e-6, True, "bf16"),
    (150, 384, 9000, 8, 0.0, 1e-5, False, "f32"),
])
def test_peaked_filter(M, H, V, bits, cap, eps, masked, sbt):
    mask = synth.make_mask(M, 20, 0.25) if masked else None
    wl = _peaked(M, H, V, bits, cap, seed=M * 7 + V, mask=mask, sb_dtype=sbt)
    wl.dlogp[::17] = 0.0  # rows that hold nothing warm
    approx, exact, cold = _run(wl, eps)
    approx = approx.cpu().numpy().astype(np.float64)
    exact = exact.cpu().numpy().astype(np.float64)
    cold = cold.cpu().numpy().astype(bool)
    oh = oracle_head(wl.head)
    g64 = wl.dlogp.astype(np.float64)
    _, dec = oracle.backward_filter(wl.h, oh, wl.targets, g64, eps, mask=wl.mask)
    n_rb = dec.cold.shape[0]
    assert (cold[n_rb:]).all()
    gcold = cold[:n_rb]
    clear = np.abs(dec.cmax - eps) > 0.05 * eps
    assert np.array_equal(gcold[clear], dec.cold[clear])
    assert gcold.sum() > 0 and (~gcold).sum() > 0
    ref_approx, _ = oracle.backward_filter(wl.h, oh, wl.targets, g64, eps, mask=wl.mask,
                                           cold=gcold)
    ref_exact = oracle.backward(wl.h, oh, wl.targets, g64, mask=wl.mask)
    act = _active(wl)
    assert (approx[~act] == 0.0).all()
    w = oracle.dequant(oh)
    scale = _scale(wl, ref_exact, w)
    rel_exact = _rel_rows(exact[act], ref_exact[act], scale[act])
    rel = _rel_rows(approx[act], ref_approx[act], scale[act])
    print(f"peaked filter: exact path {rel_exact.max():.3e}, approximate {rel.max():.3e}")
    assert rel_exact.max() <= DH_REL_TOL, f"exact dh rel-L2 {rel_exact.max():.3e}"
    assert rel.max() <= DH_REL_TOL, f"approx dh rel-L2 {rel.max():.3e}"
    bound = eps * np.linalg.norm(w, axis=1).sum()
    diff = np.linalg.norm(approx[act] - ref_exact[act], axis=1)
    assert (diff <= bound + DH_REL_TOL * scale[act]).all()


def test_filtering_changes_the_result():
    # A milder peak: the non-hot softmax terms (~1e-6 .. 1e-5) survive the fp16
    # coefficients but lie below eps = 1e-4, so the cold blocks' terms were
    # nonzero in the exact backward.
    wl = _peaked(200, 256, 16000, 4, 30.0, seed=73, bias_shift=0.1)
    approx, exact, cold = _run(wl, 1e-4)
    d = (approx - exact).abs().max().item()
    assert d > 0.0 and cold.sum().item() > 0
    w = oracle.dequant(oracle_head(wl.head))
    assert d <= 1e-4 * float(np.linalg.norm(w, axis=1).sum())


def test_workspace_and_its_size_check():
    wl = _peaked(100, 256, 3000, 4, 30.0, seed=74)
    head, h, t, mk, g = to_dev(wl)
    need = qhead._ws_size("qhead_bwd_filter_workspace", head, 100)
    assert need > qhead.bwd_workspace(head, 100)  # the tensor-core plan plus the cold map
    _, lse, _ = qhead.fwd(head, h, t, mk)
    small = qhead.alloc_workspace(need - 256, h.device)
    with pytest.raises(qhead.QheadError, match="workspace"):
        qhead.bwd_filter(head, h, t, lse, g, 1e-5, mk, workspace=small)
