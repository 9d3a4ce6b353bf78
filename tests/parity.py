"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI
binding and compare it with the fp64 oracle.

Tolerances (from the method's accuracy bar):
  |lse_gpu - lse_oracle| <= 2e-3,  |logp_gpu - logp_oracle| <= 2e-3;
  argmax identical wherever the oracle's top-2 gap of z exceeds 1e-3, and
  otherwise the GPU's pick must be a valid maximum (its z within 2e-3 of max z);
  dh: relative L2 error <= 2e-3 per row, ||dh_gpu - dh_oracle|| / ||dh_oracle||,
  and over all compared rows together; masked rows exactly 0.

The plain per-row rule has no meaning where dh itself is a cancellation: dh is
the difference of the one-hot term dlogp * sech2 * w_target and the softmax
average of the weights, and where the softmax puts (nearly) all its mass on
the target the two agree to many digits (V = 1: dh = 0 exactly).  Only the
cases named in TERMS_RELATIVE measure the error against the size of the
terms, max(||dh_oracle||, |dlogp| * ||w_target||), and a test opts into one by
name.
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
                                 wl.head.group, wl.head.softcap, device=device,
                                 sb_dtype=wl.head.sb_dtype)
    h = torch.from_numpy(wl.h.astype(np.int16)).view(torch.bfloat16).to(device)
    t = torch.from_numpy(wl.targets).to(device) if wl.targets is not None else None
    mk = torch.from_numpy(wl.mask).to(device) if wl.mask is not None else None
    g = torch.from_numpy(wl.dlogp).to(device)
    return head, h, t, mk, g


def oracle_head(sh: synth.SynthHead) -> oracle.Head:
    return oracle.Head(sh.wq, sh.scales, sh.biases, sh.bits, sh.group, sh.softcap, sh.sb_dtype)


def gpu_fwd(head, h, t, mk):
    logp, lse, am = qhead.fwd(head, h, t, mk)
    torch.cuda.synchronize()
    return ((logp.cpu().numpy() if logp is not None else None), lse.cpu().numpy(),
            am.cpu().numpy())


BATCH = 128  # oracle rows per call: bounds its [rows, V] fp64 logits (268 MB at V = 262144)


def check_fwd(wl: synth.Workload, rows, g_logp, g_lse, g_am, threads=0):
    """Compare GPU forward outputs (full-M arrays) with the oracle on `rows`
    (in batches of BATCH rows).  Returns the number of active rows compared."""
    rows = np.asarray(rows)
    n_act = 0
    for b0 in range(0, len(rows), BATCH):
        n_act += _check_fwd_batch(wl, rows[b0:b0 + BATCH], g_logp, g_lse, g_am, threads)
    return n_act


def _check_fwd_batch(wl, rows, g_logp, g_lse, g_am, threads):
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
        return 0
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
    return int(act.sum())


# Cases where dh is a cancellation of its two terms, so the error is measured
# against the terms (see the module docstring).  Each entry names the case
# and why it cancels.
TERMS_RELATIVE = {
    "V=1": "a one-row vocabulary: softmax = onehot, dh = 0 exactly",
    "peaked": "a peaked softmax whose mass sits on the target: onehot - p ~ 0",
}


def check_dh(wl: synth.Workload, rows, g_dh, threads=0, case: str | None = None,
             label: str = ""):
    """Compare GPU dh rows (a full-M array) with the oracle on `rows`.
    Returns (worst per-row rel-L2, rel-L2 over all compared active rows)."""
    if case is not None and case not in TERMS_RELATIVE:
        raise ValueError(f"unknown cancellation case {case!r}")
    rows = np.asarray(rows)
    errs, dens, idx = [], [], []
    for b0 in range(0, len(rows), BATCH):
        e, d, r = _dh_batch(wl, rows[b0:b0 + BATCH], g_dh, threads, case)
        errs.append(e)
        dens.append(d)
        idx.append(r)
    err, den, act_rows = np.concatenate(errs), np.concatenate(dens), np.concatenate(idx)
    if not len(err):
        return 0.0, 0.0
    rel = err / np.maximum(den, 1e-300)
    worst = float(rel.max())
    glob = float(np.linalg.norm(err) / max(np.linalg.norm(den), 1e-300))
    print(f"dh{(' ' + label) if label else ''}: {len(err)} rows, worst row rel-L2 "
          f"{worst:.3e} (row {int(act_rows[rel.argmax()])}), over all rows {glob:.3e}"
          + (f" [terms-relative: {case}]" if case else ""))
    assert worst <= DH_REL_TOL, f"dh rel-L2 {worst:.3e} at row {int(act_rows[rel.argmax()])}"
    assert glob <= DH_REL_TOL, f"dh rel-L2 over all rows {glob:.3e}"
    return worst, glob


def _dh_batch(wl, rows, g_dh, threads, case):
    """Per active row of the batch: the L2 error and the denominator."""
    oh = oracle_head(wl.head)
    mk = wl.mask[rows] if wl.mask is not None else None
    ref = oracle.backward(wl.h[rows], oh, wl.targets[rows], wl.dlogp[rows].astype(np.float64),
                          mk, threads=threads)
    act = np.ones(len(rows), bool) if mk is None else mk.astype(bool)
    got = g_dh[rows].astype(np.float64)
    assert np.all(got[~act] == 0.0), "masked dh rows must be exactly 0"
    err = np.linalg.norm(got[act] - ref[act], axis=1)
    den = np.linalg.norm(ref[act], axis=1)
    if case is not None and act.any():
        tg = wl.targets[rows][act]
        sub = oracle.Head(wl.head.wq[tg], wl.head.scales[tg], wl.head.biases[tg], wl.head.bits,
                          wl.head.group, wl.head.softcap, wl.head.sb_dtype)
        wt_norm = np.linalg.norm(oracle.dequant(sub), axis=1)
        den = np.maximum(den, np.abs(wl.dlogp[rows][act].astype(np.float64)) * wt_norm)
    return err, den, rows[act]
