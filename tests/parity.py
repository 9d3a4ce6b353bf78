"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI
binding and compare it with the fp64 oracle.

Tolerances (from the method's accuracy bar):
  |lse_gpu - lse_oracle| <= 2e-3,  |logp_gpu - logp_oracle| <= 2e-3;
  argmax identical wherever the oracle's top-2 gap of z exceeds 1e-3, and
  otherwise the GPU's pick must be a valid maximum (its z within 2e-3 of max z);
  dh: L2 error per row <= 2e-3 x max(|dh_oracle|, |dlogp| * |w_target|); masked
  rows exactly 0.  dh is the difference of the one-hot term dlogp*sech2*w_target
  and the softmax average; where the two nearly cancel (V = 1, a peaked
  softmax) the error is relative to the terms, not to their tiny difference.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from verify_vocab_blocked_gb300 import qhead, synth

LSE_TOL = 2e-3
LOGP_TOL = 2e-3
GAP_TOL = 1e-3
DH_REL_TOL = 2e-3


def to_dev(wl: synth.Workload, device="cuda"):
    head = qhead.Head.from_numpy(wl.head.wq, wl.head.scales, wl.head.biases, wl.head.bits,
                                 wl.head.group, wl.head.softcap, device=device)
    h = torch.from_numpy(wl.h.astype(np.int16)).view(torch.bfloat16).to(device)
    t = torch.from_numpy(wl.targets).to(device) if wl.targets is not None else None
    mk = torch.from_numpy(wl.mask).to(device) if wl.mask is not None else None
    g = torch.from_numpy(wl.dlogp).to(device)
    return head, h, t, mk, g


def oracle_head(sh: synth.SynthHead) -> oracle.Head:
    return oracle.Head(sh.wq, sh.scales, sh.biases, sh.bits, sh.group, sh.softcap)


def gpu_fwd(head, h, t, mk):
    logp, lse, am = qhead.fwd(head, h, t, mk)
    torch.cuda.synchronize()
    return ((logp.cpu().numpy() if logp is not None else None), lse.cpu().numpy(),
            am.cpu().numpy())


def check_fwd(wl: synth.Workload, rows, g_logp, g_lse, g_am, threads=0):
    """Compare GPU forward outputs (full-M arrays) with the oracle on `rows`."""
    rows = np.asarray(rows)
    oh = oracle_head(wl.head)
    tg = wl.targets[rows] if wl.targets is not None else None
    mk = wl.mask[rows] if wl.mask is not None else None
    ref = oracle.forward(wl.h[rows], oh, tg, mk, threads=threads, keep_raw=True)
    act = np.ones(len(rows), bool) if mk is None else mk.astype(bool)
    cap = wl.head.softcap
    # masked rows: exact sentinels
    assert np.all(g_lse[rows][~act] == 0.0)
    assert np.all(g_am[rows][~act] == -1)
    if g_logp is not None:
        assert np.all(g_logp[rows][~act] == 0.0)
    if not act.any():
        return ref
    d_lse = np.abs(g_lse[rows][act] - ref.lse[act])
    assert d_lse.max() <= LSE_TOL, f"lse err {d_lse.max():.3e}"
    if g_logp is not None:
        d_logp = np.abs(g_logp[rows][act] - ref.logp[act])
        assert d_logp.max() <= LOGP_TOL, f"logp err {d_logp.max():.3e}"
    am = g_am[rows]
    for k in np.nonzero(act)[0]:
        if ref.gap[k] > GAP_TOL:
            assert am[k] == ref.argmax[k], (rows[k], am[k], ref.argmax[k], ref.gap[k])
        else:
            assert 0 <= am[k] < wl.head.V
            zr = ref.raw[k, am[k]]
            z = cap * np.tanh(zr / cap) if cap > 0 else zr
            assert z >= ref.zmax[k] - LOGP_TOL
    return ref


def check_dh(wl: synth.Workload, rows, g_dh, lse_ref=None, threads=0):
    rows = np.asarray(rows)
    oh = oracle_head(wl.head)
    mk = wl.mask[rows] if wl.mask is not None else None
    ref = oracle.backward(wl.h[rows], oh, wl.targets[rows], wl.dlogp[rows].astype(np.float64),
                          mk, threads=threads)
    act = np.ones(len(rows), bool) if mk is None else mk.astype(bool)
    got = g_dh[rows].astype(np.float64)
    assert np.all(got[~act] == 0.0), "masked dh rows must be exactly 0"
    sub = oracle.Head(wl.head.wq[wl.targets[rows]], wl.head.scales[wl.targets[rows]],
                      wl.head.biases[wl.targets[rows]], wl.head.bits, wl.head.group,
                      wl.head.softcap)
    wt_norm = np.linalg.norm(oracle.dequant(sub), axis=1)
    worst = 0.0
    for k in np.nonzero(act)[0]:
        den = max(np.linalg.norm(ref[k]), abs(float(wl.dlogp[rows[k]])) * wt_norm[k])
        rel = np.linalg.norm(got[k] - ref[k]) / max(den, 1e-30)
        worst = max(worst, rel)
    assert worst <= DH_REL_TOL, f"dh rel-L2 {worst:.3e}"
    return worst
