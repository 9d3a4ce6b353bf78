"""Pins for the fp64 oracle, each against something other than the oracle itself.

* the packed layout against hand-packed words (tests/golden/pack_layout.txt);
* fp16 / bf16 widening against numpy's and torch's own conversions, on every
  bit pattern;
* hand-derivable worked examples (closed forms for lse, logp, argmax, dh,
  with and without the soft cap);
* special cases: V = 1, identical vocab rows, a very large cap equals no cap,
  a shared bias shift leaves logp / argmax / dh unchanged;
* a naive second fp64 path on the tiny shapes (codes by integer division,
  unshifted log-sum-exp, a scanned first maximum, dh from its definition);
* a library cross-check: torch fp64 log_softmax / logsumexp / argmax and
  autograd's dh on an independently unpacked head;
* finite differences of sum_m dlogp_m * logp_m against dh;
* invariants: logp <= 0, max z <= lse <= max z + ln V, z at the argmax is the
  row maximum;
* the head gradient dW: torch fp64 autograd with respect to the dense head,
  finite differences with respect to a group's bias and scale, a two-row
  closed form, vanishing column sums without the cap, V = 1 and masking;
* the blockMax early exit: tile maxima against the row maxima of the C row
  statistics and a hand example, the approximate dh equal to the exact one at
  eps = 0 and within |dlogp| eps sum_v |w_v| of it otherwise, and a hand
  derivation of a row whose tile keeps only its own target's vocab tile;
* the coefficient filter: block decisions and block maxima against plain
  loops over torch's softmax terms, the approximate dh against autograd's
  exact dh plus the dropped terms, equality with the exact dh at eps = 0, the
  eps sum_v |w_v| bound, and a hand derivation of a row whose block keeps
  only its own target's 32 vocab rows.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from verify_vocab_blocked_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_layout():
    rows = []
    with open(os.path.join(GOLDEN, "pack_layout.txt")) as f:
        for line in f:
            if not line.strip() or line.startswith("#"):
                continue
            bits, words, codes = line.rstrip("\n").split("\t")
            rows.append((int(bits), [int(w, 16) for w in words.split()],
                         [int(c) for c in codes.split()]))
    return rows


@pytest.mark.parametrize("case", _read_layout())
def test_pack_layout_golden(case):
    bits, words, expect = case
    wq = np.array([words], dtype=np.uint32)
    H = len(words) * 32 // bits
    got = oracle.codes(wq, H, bits)[0]
    assert got.tolist() == expect


def _unpack_independent(wq: np.ndarray, bits: int) -> np.ndarray:
    """Unpack through the little-endian bit string of each row (np.unpackbits),
    not through shifts and masks."""
    V, wpr = wq.shape
    b = np.unpackbits(wq.astype("<u4").view(np.uint8).reshape(V, wpr * 4), axis=1,
                      bitorder="little")
    fields = b.reshape(V, wpr * 32 // bits, bits).astype(np.int64)
    return (fields * (1 << np.arange(bits))).sum(axis=2)


@pytest.mark.parametrize("bits", [4, 8])
def test_unpack_matches_bitstring_expansion(bits):
    head = synth.make_head(37, 128, bits, seed=3)
    assert np.array_equal(oracle.codes(head.wq, 128, bits), _unpack_independent(head.wq, bits))


def test_widen_f16_all_patterns():
    pats = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ours = oracle.widen_f16(pats)
    ref = pats.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


def test_widen_bf16_all_patterns():
    pats = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ours = oracle.widen_bf16(pats)
    ref = torch.from_numpy(pats.astype(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


# ------------------------------------------------------------ worked examples

def _const_code_head(codes_per_row, H=64, scale=1.0 / 64, bias=0.0, softcap=0.0):
    """Row v has every 4-bit code equal to codes_per_row[v] (word = c * 0x11111111)."""
    V = len(codes_per_row)
    wq = np.array([[c * 0x11111111] * (H // 8) for c in codes_per_row], dtype=np.uint32)
    s = np.full((V, H // 64), scale, dtype=np.float64)
    b = np.full((V, H // 64), bias, dtype=np.float64)
    return oracle.Head(wq, s, b, 4, 64, softcap)


def test_worked_example_no_cap():
    # h = ones(64), w_v = c_v / 64 everywhere, so raw = [0, 1, 2].
    head = _const_code_head([0, 1, 2])
    h = np.ones((1, 64), dtype=np.float64)
    f = oracle.forward(h, head, targets=[1], keep_raw=True)
    assert np.allclose(f.raw[0], [0.0, 1.0, 2.0], atol=1e-15)
    lse = math.log(1 + math.e + math.e ** 2)
    assert abs(f.lse[0] - lse) < 1e-14
    assert abs(f.logp[0] - (1.0 - lse)) < 1e-14
    assert f.argmax[0] == 2
    assert abs(f.gap[0] - 1.0) < 1e-14
    # dh = sum_v (onehot_v - p_v) w_v = (c_t - E_p[c]) / 64 in every column.
    p = np.exp(np.array([0.0, 1.0, 2.0]) - lse)
    expect = (1.0 - (p * [0, 1, 2]).sum()) / 64
    dh = oracle.backward(h, head, [1], 1.0)
    assert np.allclose(dh, expect, atol=1e-15, rtol=1e-13)
    # The sign follows d(dlogp * logp)/dh: a negative cotangent flips it.
    dh_neg = oracle.backward(h, head, [1], -2.5)
    assert np.allclose(dh_neg, -2.5 * expect, atol=1e-15, rtol=1e-13)


def test_worked_example_softcap():
    # cap = 1: z = tanh(raw); sech2 = 1 - tanh(raw)^2 scales every coefficient.
    head = _const_code_head([0, 1, 2], softcap=1.0)
    h = np.ones((1, 64), dtype=np.float64)
    f = oracle.forward(h, head, targets=[2])
    z = np.tanh([0.0, 1.0, 2.0])
    lse = math.log(np.exp(z).sum())
    assert abs(f.lse[0] - lse) < 1e-14
    assert abs(f.logp[0] - (z[2] - lse)) < 1e-14
    assert f.argmax[0] == 2
    assert abs(f.gap[0] - (z[2] - z[1])) < 1e-14
    p = np.exp(z - lse)
    sech2 = 1 - z ** 2
    coeff = (np.array([0.0, 0.0, 1.0]) - p) * sech2
    expect = (coeff * np.array([0, 1, 2]) / 64).sum()
    dh = oracle.backward(h, head, [2], 1.0)
    assert np.allclose(dh, expect, atol=1e-15, rtol=1e-12)


def test_worked_example_group_scales():
    # Two groups with different scales and biases; h = ones(128); row 0 has code 3
    # in group 0 and code 5 in group 1, row 1 is all zeros.
    wq = np.zeros((2, 16), dtype=np.uint32)
    wq[0, :8] = 3 * 0x11111111
    wq[0, 8:] = 5 * 0x11111111
    s = np.array([[0.25, 0.5], [1.0, 1.0]])
    b = np.array([[-0.5, 0.125], [0.0, -0.25]])
    head = oracle.Head(wq, s, b, 4, 64, 0.0)
    raw = oracle.logits(np.ones((1, 128)), head)[0]
    assert np.allclose(raw, [64 * (0.25 * 3 - 0.5) + 64 * (0.5 * 5 + 0.125),
                             64 * 0.0 + 64 * (-0.25)], atol=1e-12)


# -------------------------------------------------------------- special cases

@pytest.mark.parametrize("cap", [0.0, 30.0])
def test_single_vocab_row(cap):
    head = synth.make_head(1, 128, 4, softcap=cap, seed=1)
    ohead = oracle.Head(head.wq, head.scales, head.biases, 4, 64, cap)
    h = synth.make_hidden(3, 128, seed=1)
    f = oracle.forward(h, ohead, targets=[0, 0, 0], keep_raw=True)
    z = cap * np.tanh(f.raw[:, 0] / cap) if cap else f.raw[:, 0]
    assert np.allclose(f.lse, z, atol=1e-13)
    assert np.allclose(f.logp, 0.0, atol=1e-13)
    assert (f.argmax == 0).all()
    dh = oracle.backward(h, ohead, [0, 0, 0], 1.0)
    assert np.abs(dh).max() < 1e-13


@pytest.mark.parametrize("cap", [0.0, 5.0])
def test_identical_rows(cap):
    base = synth.make_head(1, 128, 4, seed=2)
    V = 7
    head = oracle.Head(np.repeat(base.wq, V, 0), np.repeat(base.scales, V, 0),
                       np.repeat(base.biases, V, 0), 4, 64, cap)
    h = synth.make_hidden(4, 128, seed=2)
    t = np.array([0, 3, 6, 2])
    f = oracle.forward(h, head, targets=t)
    assert np.allclose(f.logp, -math.log(V), atol=1e-13)
    assert (f.argmax == 0).all()
    assert np.allclose(f.gap, 0.0)
    dh = oracle.backward(h, head, t, 1.0)
    assert np.abs(dh).max() < 1e-13


def test_huge_cap_equals_no_cap():
    wl = synth.make_workload("tiny")
    h0 = oracle.Head(wl.head.wq, wl.head.scales, wl.head.biases, 4, 64, 0.0)
    h1 = oracle.Head(wl.head.wq, wl.head.scales, wl.head.biases, 4, 64, 1e9)
    f0 = oracle.forward(wl.h, h0, wl.targets)
    f1 = oracle.forward(wl.h, h1, wl.targets)
    assert np.allclose(f0.lse, f1.lse, atol=1e-9)
    assert np.allclose(f0.logp, f1.logp, atol=1e-9)
    assert np.array_equal(f0.argmax, f1.argmax)
    d0 = oracle.backward(wl.h, h0, wl.targets, 1.0)
    d1 = oracle.backward(wl.h, h1, wl.targets, 1.0)
    assert np.allclose(d0, d1, atol=1e-9)


def test_shared_bias_shift_invariance():
    # Adding delta to every bias shifts every logit of token m by delta * sum_d h[m,d]:
    # lse shifts by that amount, logp / argmax / dh (no cap) are unchanged.
    wl = synth.make_workload("tiny")
    s = oracle.widen_f16(wl.head.scales).reshape(wl.head.scales.shape)
    b = oracle.widen_f16(wl.head.biases).reshape(wl.head.biases.shape)
    delta = 0.0371
    ha = oracle.Head(wl.head.wq, s, b, 4, 64, 0.0)
    hb = oracle.Head(wl.head.wq, s, b + delta, 4, 64, 0.0)
    fa = oracle.forward(wl.h, ha, wl.targets)
    fb = oracle.forward(wl.h, hb, wl.targets)
    hsum = oracle.widen_bf16(wl.h).sum(axis=1)
    assert np.allclose(fb.lse - fa.lse, delta * hsum, atol=1e-10)
    assert np.allclose(fa.logp, fb.logp, atol=1e-10)
    assert np.array_equal(fa.argmax, fb.argmax)
    g = synth.make_dlogp(wl.M, seed=4)
    da = oracle.backward(wl.h, ha, wl.targets, g)
    db = oracle.backward(wl.h, hb, wl.targets, g)
    assert np.allclose(da, db, atol=1e-10)


# --------------------------------------------------------- naive second path

def _naive_codes(wq: np.ndarray, H: int, bits: int) -> np.ndarray:
    """Codes by integer division: field j of a word is (w // 2^(bits j)) mod 2^bits."""
    per = 32 // bits
    base = 1 << bits
    q = np.empty((wq.shape[0], H), dtype=np.int64)
    w64 = wq.astype(np.int64)
    for d in range(H):
        q[:, d] = (w64[:, d // per] // (base ** (d % per))) % base
    return q


@pytest.mark.parametrize("bits,cap", [(4, 0.0), (4, 30.0), (8, 0.0)])
def test_against_a_naive_second_path(bits, cap):
    # A second fp64 path on the tiny configuration's shapes: codes by integer
    # division, bf16 widened by placing its bits in the high half of a
    # binary32, logsumexp as log(sum(exp(z))) with no shift (|z| is small),
    # the first maximum by a Python scan, and dh from the definition.
    M, H, V = 16, 256, 2048
    head = synth.make_head(V, H, bits, softcap=cap, seed=31 + bits)
    oh = oracle.Head(head.wq, head.scales, head.biases, bits, 64, cap)
    hb = synth.make_hidden(M, H, seed=31)
    t = synth.make_targets(M, V, seed=31)
    g = synth.make_dlogp(M, seed=31).astype(np.float64)
    h = (hb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    q = _naive_codes(head.wq, H, bits)
    s = np.repeat(head.scales.astype(np.float64), 64, axis=1)
    b = np.repeat(head.biases.astype(np.float64), 64, axis=1)
    w = s * q + b
    raw = h @ w.T
    z = cap * np.tanh(raw / cap) if cap > 0 else raw
    lse = np.log(np.exp(z).sum(axis=1))
    logp = z[np.arange(M), t] - lse
    am = np.empty(M, dtype=np.int64)
    for m in range(M):
        best = 0
        for v in range(1, V):
            if raw[m, v] > raw[m, best]:
                best = v
        am[m] = best
    sech2 = 1.0 - np.tanh(raw / cap) ** 2 if cap > 0 else np.ones_like(raw)
    onehot = np.zeros_like(raw)
    onehot[np.arange(M), t] = 1.0
    dh = (g[:, None] * (onehot - np.exp(z - lse[:, None])) * sech2) @ w

    f = oracle.forward(hb, oh, t)
    assert np.allclose(f.lse, lse, rtol=0, atol=1e-12)
    assert np.allclose(f.logp, logp, rtol=0, atol=1e-12)
    assert np.array_equal(f.argmax, am)
    got = oracle.backward(hb, oh, t, g)
    assert np.abs(got - dh).max() <= 1e-12 * max(1.0, np.abs(dh).max())


# ----------------------------------------------------- library cross-check

def _torch_reference(h64, head: oracle.Head, targets, dlogp):
    """torch fp64: dense head from the bit-string unpack, log_softmax, autograd."""
    q = torch.from_numpy(_unpack_independent(head.wq, head.bits)).double()

    def widen(x):  # torch's own conversions, independent of the oracle's C widening
        if head.sb_dtype == "bf16":
            return torch.from_numpy(x.astype(np.uint16).view(np.int16)).view(torch.bfloat16).double()
        return torch.from_numpy(x).double()

    s, b = widen(head.scales), widen(head.biases)
    w = q * s.repeat_interleave(head.group, 1) + b.repeat_interleave(head.group, 1)
    h = torch.from_numpy(h64).clone().requires_grad_(True)
    raw = h @ w.T
    z = head.softcap * torch.tanh(raw / head.softcap) if head.softcap > 0 else raw
    lp = torch.log_softmax(z, dim=1)
    t = torch.from_numpy(np.asarray(targets, dtype=np.int64))
    logp = lp.gather(1, t[:, None])[:, 0]
    (torch.from_numpy(np.asarray(dlogp, dtype=np.float64)) * logp).sum().backward()
    return (logp.detach().numpy(), torch.logsumexp(z, 1).detach().numpy(),
            torch.argmax(raw, 1).numpy(), h.grad.numpy())


@pytest.mark.parametrize("name,V,cap,sbt", [("tiny", None, None, "f16"),
                                            ("gemma512", 4096, None, "f16"),
                                            ("mid8", 2048, None, "f16"),
                                            ("gemma512", 1500, 0.0, "f16"),
                                            ("gemma512", 1500, None, "bf16"),
                                            ("mid8", 1000, None, "bf16"),
                                            ("gemma512", 1500, None, "f32"),
                                            ("mid8", 1000, None, "f32")])
def test_against_torch_autograd(name, V, cap, sbt):
    cfg = synth.CONFIGS[name]
    V = V or cfg["V"]
    cap = cfg["softcap"] if cap is None else cap
    head = synth.make_head(V, cfg["H"], cfg["bits"], softcap=cap, seed=11, sb_dtype=sbt)
    ohead = oracle.Head(head.wq, head.scales, head.biases, cfg["bits"], 64, cap, sbt)
    M = 6
    h = synth.make_hidden(M, cfg["H"], seed=11)
    t = synth.make_targets(M, V, seed=11)
    g = synth.make_dlogp(M, seed=11).astype(np.float64)
    f = oracle.forward(h, ohead, t)
    dh = oracle.backward(h, ohead, t, g)
    r_logp, r_lse, r_am, r_dh = _torch_reference(oracle.widen_bf16(h), ohead, t, g)
    assert np.allclose(f.logp, r_logp, atol=1e-10, rtol=0)
    assert np.allclose(f.lse, r_lse, atol=1e-10, rtol=0)
    assert np.array_equal(f.argmax, r_am)
    assert np.abs(dh - r_dh).max() <= 1e-10 * max(1.0, np.abs(r_dh).max())


# ---------------------------------------------------------- finite differences

@pytest.mark.parametrize("cap", [0.0, 2.0])
def test_finite_differences(cap):
    head = synth.make_head(300, 128, 4, softcap=cap, seed=5)
    ohead = oracle.Head(head.wq, head.scales, head.biases, 4, 64, cap)
    M = 5
    h = oracle.widen_bf16(synth.make_hidden(M, 128, seed=5)) * 3.0
    t = synth.make_targets(M, 300, seed=5)
    g = synth.make_dlogp(M, seed=5).astype(np.float64)
    mask = np.array([1, 0, 1, 1, 0], dtype=np.uint8)
    dh = oracle.backward(h, ohead, t, g, mask=mask)
    assert np.all(dh[mask == 0] == 0.0)

    def f(x):
        return float((g * oracle.forward(x, ohead, t, mask=mask).logp).sum())

    rng = np.random.default_rng(0)
    for _ in range(3):
        u = rng.standard_normal(h.shape)
        eps = 1e-5
        fd = (f(h + eps * u) - f(h - eps * u)) / (2 * eps)
        an = float((dh * u).sum())
        assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (fd, an)


# ------------------------------------------------------------------ invariants

@pytest.mark.parametrize("name", ["tiny", "gemma512"])
def test_invariants(name):
    cfg = synth.CONFIGS[name]
    V = min(cfg["V"], 8192)
    head = synth.make_head(V, cfg["H"], cfg["bits"], softcap=cfg["softcap"], seed=9)
    ohead = oracle.Head(head.wq, head.scales, head.biases, cfg["bits"], 64, cfg["softcap"])
    M = 8
    h = synth.make_hidden(M, cfg["H"], seed=9)
    t = synth.make_targets(M, V, seed=9)
    mask = np.array([1, 1, 0, 1, 1, 1, 0, 1], dtype=np.uint8)
    f = oracle.forward(h, ohead, t, mask=mask, keep_raw=True)
    act = mask == 1
    assert (f.logp[act] <= 0).all()
    assert (f.lse[act] >= f.zmax[act]).all()
    assert (f.lse[act] <= f.zmax[act] + math.log(V) + 1e-12).all()
    cap = cfg["softcap"]
    z = cap * np.tanh(f.raw / cap) if cap else f.raw
    for m in np.nonzero(act)[0]:
        assert abs(z[m, f.argmax[m]] - f.zmax[m]) <= 1e-12
        assert f.argmax[m] == int(np.argmax(f.raw[m]))
    assert (f.argmax[~act] == -1).all() and (f.logp[~act] == 0).all()


# ------------------------------------------------- head gradient (dW) pins

def _torch_dw(h64, head: oracle.Head, targets, dlogp, mask=None):
    """torch fp64 autograd with respect to the dense head (independent unpack)."""
    q = torch.from_numpy(_unpack_independent(head.wq, head.bits)).double()
    s = torch.from_numpy(np.asarray(head.scales, dtype=np.float64))
    b = torch.from_numpy(np.asarray(head.biases, dtype=np.float64))
    w = (q * s.repeat_interleave(head.group, 1) + b.repeat_interleave(head.group, 1))
    w = w.clone().requires_grad_(True)
    h = torch.from_numpy(h64)
    raw = h @ w.T
    z = head.softcap * torch.tanh(raw / head.softcap) if head.softcap > 0 else raw
    lp = torch.log_softmax(z, dim=1)
    t = torch.from_numpy(np.asarray(targets, dtype=np.int64))
    logp = lp.gather(1, t[:, None])[:, 0]
    g = torch.from_numpy(np.asarray(dlogp, dtype=np.float64))
    if mask is not None:
        g = g * torch.from_numpy(np.asarray(mask, dtype=np.float64))
    (g * logp).sum().backward()
    return w.grad.numpy()


@pytest.mark.parametrize("bits,cap", [(4, 30.0), (8, 0.0), (4, 2.0)])
def test_dw_against_torch_autograd(bits, cap):
    V, H, M = 700, 128, 9
    head = synth.make_head(V, H, bits, softcap=cap, seed=21)
    ohead = oracle.Head(head.wq, head.scales, head.biases, bits, 64, cap)
    h = synth.make_hidden(M, H, seed=21)
    t = synth.make_targets(M, V, seed=21)
    t[4] = t[1]  # two rows share a target
    g = synth.make_dlogp(M, seed=21).astype(np.float64)
    mask = np.array([1, 1, 0, 1, 1, 1, 0, 1, 1], dtype=np.uint8)
    dw = oracle.grad_head(h, ohead, t, g, mask=mask)
    ohead64 = oracle.Head(head.wq, oracle.widen_f16(head.scales).reshape(head.scales.shape),
                          oracle.widen_f16(head.biases).reshape(head.biases.shape), bits, 64, cap)
    ref = _torch_dw(oracle.widen_bf16(h), ohead64, t, g, mask)
    assert np.abs(dw - ref).max() <= 1e-10 * max(1.0, np.abs(ref).max())


def test_dw_finite_differences_of_group_bias_and_scale():
    # A group's bias moves every element of the group: d/db = sum_d dW[v,d];
    # its scale moves element d by q[v,d]: d/ds = sum_d q[v,d] dW[v,d].
    V, H, M, cap = 200, 128, 5, 3.0
    head = synth.make_head(V, H, 4, softcap=cap, seed=22)
    s = oracle.widen_f16(head.scales).reshape(head.scales.shape)
    b = oracle.widen_f16(head.biases).reshape(head.biases.shape)
    h = oracle.widen_bf16(synth.make_hidden(M, H, seed=22)) * 2.0
    t = synth.make_targets(M, V, seed=22)
    g = synth.make_dlogp(M, seed=22).astype(np.float64)
    dw = oracle.grad_head(h, oracle.Head(head.wq, s, b, 4, 64, cap), t, g)
    q = oracle.codes(head.wq, H, 4).astype(np.float64)

    def loss(ss, bb):
        return float((g * oracle.forward(h, oracle.Head(head.wq, ss, bb, 4, 64, cap), t).logp).sum())

    eps = 1e-6
    for v, grp in [(int(t[0]), 0), (int(t[2]), 1), (17, 1), (150, 0)]:
        sl = slice(64 * grp, 64 * grp + 64)
        db = b.copy(); db[v, grp] += eps
        bm = b.copy(); bm[v, grp] -= eps
        fd_b = (loss(s, db) - loss(s, bm)) / (2 * eps)
        assert abs(fd_b - dw[v, sl].sum()) <= 1e-6 * max(1.0, abs(fd_b)), (v, grp)
        ds = s.copy(); ds[v, grp] += eps
        sm = s.copy(); sm[v, grp] -= eps
        fd_s = (loss(ds, b) - loss(sm, b)) / (2 * eps)
        an_s = (q[v, sl] * dw[v, sl]).sum()
        assert abs(fd_s - an_s) <= 1e-6 * max(1.0, abs(fd_s)), (v, grp)


def test_dw_worked_example_two_rows():
    # One token, two vocab rows, no cap: raw = (a, b), p = softmax(raw),
    # target 0: dW[0] = g (1 - p0) h, dW[1] = -g p1 h.
    wq = np.zeros((2, 16), dtype=np.uint32)
    wq[0, :] = 0x11111111        # codes 1
    wq[1, :] = 0x22222222        # codes 2
    s = np.array([[0.01, 0.01], [0.01, 0.01]])
    b = np.zeros((2, 2))
    head = oracle.Head(wq, s, b, 4, 64, 0.0)
    h = np.linspace(-1.0, 1.0, 128)[None, :]
    hs = h.sum()
    a0, a1 = 0.01 * hs, 0.02 * hs
    p0 = 1.0 / (1.0 + math.exp(a1 - a0))
    g = 0.75
    dw = oracle.grad_head(h, head, [0], g)
    assert np.allclose(dw[0], g * (1 - p0) * h[0], atol=1e-14)
    assert np.allclose(dw[1], -g * (1 - p0) * h[0], atol=1e-14)


def test_dw_column_sums_vanish_without_cap():
    # No cap: sum_v (1[v = t] - p_v) = 0 for every row, so sum_v dW[v, :] = 0.
    wl = synth.make_workload("tiny")
    head = oracle.Head(wl.head.wq, wl.head.scales, wl.head.biases, 4, 64, 0.0)
    g = synth.make_dlogp(wl.M, seed=23)
    dw = oracle.grad_head(wl.h, head, wl.targets, g)
    assert np.abs(dw.sum(axis=0)).max() <= 1e-12 * max(1.0, np.abs(dw).max())
    # ...and a soft cap breaks it (the sech2 factors differ per vocab row)
    capped = oracle.Head(wl.head.wq, wl.head.scales, wl.head.biases, 4, 64, 2.0)
    assert np.abs(oracle.grad_head(wl.h, capped, wl.targets, g).sum(axis=0)).max() > 1e-6


def test_dw_single_vocab_row_and_mask():
    head = synth.make_head(1, 128, 4, seed=24)
    oh = oracle.Head(head.wq, head.scales, head.biases, 4, 64, 30.0)
    h = synth.make_hidden(3, 128, seed=24)
    assert np.abs(oracle.grad_head(h, oh, [0, 0, 0], 1.0)).max() < 1e-13
    # masked rows contribute nothing: equal to the gradient of the active rows alone
    head = synth.make_head(300, 128, 8, seed=25)
    oh = oracle.Head(head.wq, head.scales, head.biases, 8, 64, 0.0)
    h = synth.make_hidden(6, 128, seed=25)
    t = synth.make_targets(6, 300, seed=25)
    g = synth.make_dlogp(6, seed=25)
    mask = np.array([0, 1, 1, 0, 1, 0], dtype=np.uint8)
    act = mask == 1
    a = oracle.grad_head(h, oh, t, g, mask=mask)
    b = oracle.grad_head(h[act], oh, t[act], g[act])
    assert np.allclose(a, b, atol=1e-13, rtol=0)


# ------------------------------------------- blockMax early exit (approximate)

def test_block_max_pins():
    # The maximum over a row's tiles is the row's maximum capped logit (from
    # the C row statistics), every tile maximum lies below lse, and a hand
    # example: V = 3 rows in one tile of 2 and one of 1.
    head = synth.make_head(700, 128, 4, softcap=30.0, seed=26)
    oh = oracle.Head(head.wq, head.scales, head.biases, 4, 64, 30.0)
    h = synth.make_hidden(6, 128, seed=26)
    mask = np.array([1, 1, 0, 1, 1, 1], np.uint8)
    bm = oracle.block_max(h, oh, mask=mask)
    f = oracle.forward(h, oh, mask=mask)
    act = mask == 1
    assert bm.shape == (6, 3)
    assert np.allclose(bm[act].max(axis=1), f.zmax[act], atol=1e-13)
    assert (bm[act] <= f.lse[act, None]).all()
    assert np.isneginf(bm[~act]).all()
    wq = np.zeros((3, 16), np.uint32)
    wq[1, :] = 0x11111111
    wq[2, :] = 0x33333333
    small = oracle.Head(wq, np.full((3, 2), 0.01), np.zeros((3, 2)), 4, 64, 0.0)
    x = np.ones((1, 128))
    assert np.allclose(oracle.block_max(x, small, tile=2)[0], [1.28, 3.84], atol=1e-12)


def test_blockskip_reduces_to_exact_and_obeys_its_bound():
    # one row tile of 40 rows over 32 vocab tiles: most tiles hold no target
    V = 8192
    head, hot = synth.make_peaked_head(V, 128, 4, n_hot=4, bias_shift=0.3, softcap=30.0,
                                       seed=27)
    oh = oracle.Head(head.wq, head.scales, head.biases, 4, 64, 30.0)
    M = 40
    h = synth.make_hidden(M, 128, seed=27, mean=0.5)
    t = synth.make_targets(M, V, seed=27)
    g = synth.make_dlogp(M, seed=27).astype(np.float64)
    mask = synth.make_mask(M, 20, 0.2)
    f = oracle.forward(h, oh, t, mask=mask)
    bm = oracle.block_max(h, oh, mask=mask)
    exact = oracle.backward(h, oh, t, g, mask=mask)
    # eps = 0 drops nothing
    assert np.array_equal(oracle.backward_blockskip(h, oh, t, g, bm, 0.0, mask=mask, lse=f.lse),
                          exact)
    # eps > 0 drops blocks: every dropped coefficient is below |dlogp| eps (sech2 <= 1),
    # so per row the change is at most |dlogp| eps sum_v |w_v|
    eps = 1e-4
    approx = oracle.backward_blockskip(h, oh, t, g, bm, eps, mask=mask, lse=f.lse)
    wnorm = np.linalg.norm(oracle.dequant(oh), axis=1).sum()
    act = mask == 1
    diff = np.linalg.norm(approx - exact, axis=1)
    assert (diff[act] <= np.abs(g[act]) * eps * wnorm + 1e-12).all()
    assert diff[act].max() > 0.0           # something was dropped...
    assert (approx[~act] == 0.0).all()      # ...and masked rows stay exact zeros


def test_blockskip_keeps_target_tiles_and_decides_per_row_tile():
    # 129 active rows: two row tiles (128 + 1).  With an enormous eps every
    # vocab tile is below it, so only the tiles holding one of the row tile's
    # targets survive: row 128 (alone in its tile) keeps exactly its own
    # target's tile.
    head = synth.make_head(1024, 128, 4, seed=28)
    oh = oracle.Head(head.wq, head.scales, head.biases, 4, 64, 0.0)
    M = 129
    h = synth.make_hidden(M, 128, seed=28)
    t = synth.make_targets(M, 1024, seed=28)
    t[128] = 700                                  # tile 2
    t[:128] = np.where(t[:128] // 256 == 2, 5, t[:128])  # no other row targets tile 2
    g = np.ones(M)
    f = oracle.forward(h, oh, t)
    bm = oracle.block_max(h, oh)
    approx = oracle.backward_blockskip(h, oh, t, g, bm, 1e300, lse=f.lse)
    # row 128: dh = (onehot - p) sech2 . W restricted to vocab tile 2
    raw = oracle.logits(h[128:], oh)[0]
    p = np.exp(raw - f.lse[128])
    c = -p
    c[700] += 1.0
    c[:512] = 0.0
    c[768:] = 0.0
    w = oracle.dequant(oh)
    assert np.allclose(approx[128], c @ w, atol=1e-12)


# ---------------------------------------------- coefficient filter (approximate)

def _torch_softmax_terms(h64, head: oracle.Head):
    """torch fp64 on the independently unpacked dense head: p[m, v] and
    sech2[m, v] (1 without a cap), and the dense head itself."""
    q = torch.from_numpy(_unpack_independent(head.wq, head.bits)).double()

    def widen(x):  # torch's own conversions, independent of the oracle's C widening
        if head.sb_dtype == "bf16":
            return torch.from_numpy(x.astype(np.uint16).view(np.int16)).view(torch.bfloat16).double()
        return torch.from_numpy(x).double()

    s, b = widen(head.scales), widen(head.biases)
    w = q * s.repeat_interleave(head.group, 1) + b.repeat_interleave(head.group, 1)
    raw = torch.from_numpy(h64) @ w.T
    if head.softcap > 0:
        th = torch.tanh(raw / head.softcap)
        z, sech2 = head.softcap * th, 1.0 - th * th
    else:
        z, sech2 = raw, torch.ones_like(raw)
    return torch.softmax(z, dim=1).numpy(), sech2.numpy(), w.numpy()


def _filter_case(seed=41, bits=4, cap=30.0, V=640):
    # 52 of 70 rows active: row blocks of 32 and 20; V = 640: 20 vocab blocks;
    # peaked logits so that some blocks are cold and others warm
    H, M = 128, 70
    head, hot = synth.make_peaked_head(V, H, bits, n_hot=6, bias_shift=0.3, softcap=cap,
                                       seed=seed)
    oh = oracle.Head(head.wq, head.scales, head.biases, bits, 64, cap)
    h = synth.make_hidden(M, H, seed=seed, mean=0.5)
    t = synth.make_targets(M, V, seed=seed)
    g = synth.make_dlogp(M, seed=seed).astype(np.float64)
    mask = np.ones(M, np.uint8)
    mask[[0, 3, 4, 9, 17, 18, 19, 25, 33, 40, 41, 44, 50, 51, 60, 61, 62, 69]] = 0
    return oh, h, t, g, mask


def _brute_decisions(oh, h, t, g, mask, eps):
    """Block decisions by plain loops over torch's softmax terms."""
    p, sech2, _ = _torch_softmax_terms(oracle._as_f64_h(h), oh)
    act = [m for m in range(len(mask)) if mask[m]]
    V = p.shape[1]
    nrb, nvb = (len(act) + 31) // 32, (V + 31) // 32
    cold = np.zeros((nrb, nvb), bool)
    cmax = np.zeros((nrb, nvb))
    for j in range(nrb):
        rows = act[32 * j:32 * j + 32]
        for k in range(nvb):
            best, target_here = 0.0, False
            for m in rows:
                for v in range(32 * k, min(32 * k + 32, V)):
                    if v == t[m]:
                        target_here = True
                        continue
                    best = max(best, abs(g[m]) * p[m, v] * sech2[m, v])
            cmax[j, k] = best
            cold[j, k] = best < eps and not target_here
    return cold, cmax, p, sech2, act


@pytest.mark.parametrize("seed,bits,cap,V", [(41, 4, 30.0, 640), (45, 8, 0.0, 600),
                                            (46, 4, 0.0, 333)])
def test_filter_decisions_match_brute_force(seed, bits, cap, V):
    oh, h, t, g, mask = _filter_case(seed, bits, cap, V)
    dec0 = oracle.filter_blocks(np.zeros((70, V)), t, 1.0, mask)  # shape only
    assert dec0.cold.shape == (2, (V + 31) // 32)
    _, dec = oracle.backward_filter(h, oh, t, g, 0.0, mask=mask)
    eps = float(np.median(dec.cmax))
    cold_b, cmax_b, *_ = _brute_decisions(oh, h, t, g, mask, eps)
    _, dec = oracle.backward_filter(h, oh, t, g, eps, mask=mask)
    assert np.allclose(dec.cmax, cmax_b, rtol=1e-10, atol=1e-300)
    assert np.array_equal(dec.cold, cold_b)
    assert 0 < dec.cold.sum() < dec.cold.size  # both kinds of block occur


def test_filter_dh_against_torch_autograd():
    # dh with the filter = the exact autograd dh plus the dropped softmax terms
    # (a dropped coefficient is -dlogp p sech2, so dropping it adds
    # dlogp p sech2 w_v back), with the brute-force decisions
    oh, h, t, g, mask = _filter_case(seed=42)
    _, dec = oracle.backward_filter(h, oh, t, g, 0.0, mask=mask)
    eps = float(np.quantile(dec.cmax, 0.6))
    cold_b, _, p, sech2, act = _brute_decisions(oh, h, t, g, mask, eps)
    h64 = oracle._as_f64_h(h)
    act_idx = np.array(act)
    *_, dh_exact = _torch_reference(h64[act_idx], oh, t[act_idx], g[act_idx])
    _, _, w = _torch_softmax_terms(h64, oh)
    want = np.zeros((70, 128))
    want[act_idx] = dh_exact
    for j, k in zip(*np.nonzero(cold_b)):
        for m in act[32 * j:32 * j + 32]:
            cols = slice(32 * k, 32 * k + 32)
            want[m] += (g[m] * p[m, cols] * sech2[m, cols]) @ w[cols]
    got, dec = oracle.backward_filter(h, oh, t, g, eps, mask=mask)
    assert np.array_equal(dec.cold, cold_b)
    assert np.allclose(got, want, rtol=0, atol=1e-10)


def test_filter_reduces_to_exact_and_obeys_its_bound():
    oh, h, t, g, mask = _filter_case(seed=43)
    exact = oracle.backward(h, oh, t, g, mask=mask)
    got0, dec0 = oracle.backward_filter(h, oh, t, g, 0.0, mask=mask)
    assert not dec0.cold.any()
    assert np.array_equal(got0, exact)
    eps = float(np.quantile(dec0.cmax, 0.5))
    got, dec = oracle.backward_filter(h, oh, t, g, eps, mask=mask)
    # every dropped coefficient is below eps, so per row the change is at
    # most eps sum_v |w_v|
    wnorm = np.linalg.norm(oracle.dequant(oh), axis=1).sum()
    diff = np.linalg.norm(got - exact, axis=1)
    act = mask == 1
    assert (diff <= eps * wnorm + 1e-12).all()
    assert diff[act].max() > 0.0
    assert (got[~act] == 0.0).all()


def test_filter_keeps_target_blocks():
    # With an enormous eps every block is cold except those holding a target:
    # the 33rd active row, alone in its row block, keeps exactly its own
    # target's 32 vocab rows.
    head = synth.make_head(256, 128, 4, softcap=30.0, seed=44)
    oh = oracle.Head(head.wq, head.scales, head.biases, 4, 64, 30.0)
    M = 33
    h = synth.make_hidden(M, 128, seed=44)
    t = synth.make_targets(M, 256, seed=44)
    t[32] = 77                                       # vocab block 2
    g = np.full(M, -1.5)
    got, dec = oracle.backward_filter(h, oh, t, g, 1e300)
    assert dec.cold[1].sum() == 7 and not dec.cold[1, 2]
    f = oracle.forward(h[32:], oh)
    raw = oracle.logits(h[32:], oh)[0]
    th = np.tanh(raw / 30.0)
    p = np.exp(30.0 * th - f.lse[0])
    onehot = (np.arange(256) == 77).astype(np.float64)
    c = -1.5 * (onehot - p) * (1.0 - th * th)
    c[:64] = 0.0
    c[96:] = 0.0
    assert np.allclose(got[32], c @ oracle.dequant(oh), atol=1e-12)


# ------------------------------------------------- scale / bias element types

def test_bf16_scales_equal_the_fp16_head_they_round_to():
    # bf16 values of magnitude in [2^-14, 65504] have 8 significant bits and
    # are exactly fp16 values too: the bf16 head and the fp16 head holding the
    # same numbers must give identical results (the fp16 path is pinned above).
    hb = synth.make_head(700, 256, 4, softcap=30.0, seed=31, sb_dtype="bf16")
    sv, bv = oracle.widen_bf16(hb.scales), oracle.widen_bf16(hb.biases)
    assert (np.abs(sv) >= 2.0 ** -14).all() and (np.abs(bv) >= 2.0 ** -14).all()
    s16, b16 = sv.astype(np.float16), bv.astype(np.float16)
    assert np.array_equal(s16.astype(np.float64), sv) and np.array_equal(b16.astype(np.float64), bv)
    o_bf = oracle.Head(hb.wq, hb.scales, hb.biases, 4, 64, 30.0, "bf16")
    o_16 = oracle.Head(hb.wq, s16, b16, 4, 64, 30.0, "f16")
    h = synth.make_hidden(7, 256, seed=31)
    t = synth.make_targets(7, 700, seed=31)
    g = synth.make_dlogp(7, seed=31).astype(np.float64)
    fa, fb = oracle.forward(h, o_bf, t), oracle.forward(h, o_16, t)
    assert np.array_equal(fa.lse, fb.lse) and np.array_equal(fa.logp, fb.logp)
    assert np.array_equal(oracle.backward(h, o_bf, t, g), oracle.backward(h, o_16, t, g))


def test_f32_scales_are_used_unrounded():
    # A scale no fp16 (or bf16) can hold: 1/64 * (1 + 2^-20).  With every code
    # 15 and h = ones(64), raw = 64 * (15 s + b) exactly (fp64 holds it).
    s = np.float32(1.0 / 64) * np.float32(1.0 + 2.0 ** -20)
    b = np.float32(-0.1)
    wq = np.full((1, 8), 0xFFFFFFFF, dtype=np.uint32)
    head = oracle.Head(wq, np.array([[s]], np.float32), np.array([[b]], np.float32), 4, 64, 0.0,
                       "f32")
    raw = oracle.logits(np.ones((1, 64)), head)
    assert raw[0, 0] == 64.0 * (15.0 * float(s) + float(b))
    assert float(s) != float(np.float16(s))
