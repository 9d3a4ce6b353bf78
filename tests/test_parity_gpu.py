"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Small cases are compared on every row.  The full-size workloads run whole on
the GPU and are compared on every forward row (all five workloads), and dh
on 256 seeded rows plus rows 0 and M - 1 and every row next to a mask
boundary: rows are independent, so a compared row is an exact check of that
row.  Properties that hold at any size are checked on every row besides.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from parity import check_dh, check_fwd, gpu_fwd, oracle_head, to_dev
from verify_vocab_blocked_gb300 import build as qbuild
from verify_vocab_blocked_gb300 import qhead, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="session", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    qbuild.build()
    qhead.lib()


def _custom(M, H, V, bits, cap, seed=0, mask=None, targets=None, dlogp=None, sb_dtype="f16"):
    head = synth.make_head(V, H, bits, softcap=cap, seed=seed, sb_dtype=sb_dtype)
    h = synth.make_hidden(M, H, seed=seed)
    t = synth.make_targets(M, V, seed=seed) if targets is None else np.asarray(targets, np.int32)
    g = synth.make_dlogp(M, seed=seed) if dlogp is None else np.asarray(dlogp, np.float32)
    return synth.Workload("custom", head, h, t, mask, g, dict(M=M, H=H, V=V, bits=bits))


def _run_all(wl, bwd=True, case=None):
    head, h, t, mk, g = to_dev(wl)
    logp, lse, am = gpu_fwd(head, h, t, mk)
    rows = np.arange(wl.M)
    check_fwd(wl, rows, logp, lse, am)
    if bwd:
        lse_d = torch.from_numpy(lse).cuda()
        dh = qhead.bwd(head, h, t, lse_d, g, mk)
        torch.cuda.synchronize()
        check_dh(wl, rows, dh.cpu().numpy(), case=case)


def test_tiny_config():
    wl = synth.make_workload("tiny")
    wl.dlogp = np.ones(wl.M, np.float32)
    _run_all(wl)


def test_tiny_random_cotangent():
    wl = synth.make_workload("tiny", seed=3)
    wl.dlogp = synth.make_dlogp(wl.M, seed=3)
    _run_all(wl)


EDGE = [
    # M, H, V, bits, cap
    (1, 256, 2048, 4, 0.0),
    (2, 256, 2048, 4, 30.0),
    (3, 256, 2048, 8, 0.0),
    (4, 128, 1000, 4, 5.0),
    (5, 384, 4099, 4, 30.0),
    (7, 128, 130, 8, 0.0),
    (8, 256, 127, 4, 0.0),
    (9, 512, 3000, 8, 30.0),
    (17, 128, 1, 4, 0.0),
    (33, 256, 16, 4, 2.0),
    (127, 128, 777, 8, 0.0),
    (128, 256, 515, 4, 30.0),
    (129, 128, 2049, 4, 0.0),
]


@pytest.mark.parametrize("M,H,V,bits,cap", EDGE)
def test_edge_shapes(M, H, V, bits, cap):
    # V = 1: softmax = onehot, so dh = 0 exactly and only the terms-relative
    # error is defined.
    _run_all(_custom(M, H, V, bits, cap, seed=M + V), case="V=1" if V == 1 else None)


# Shapes on the tensor-core forward (M >= 17): partial 256-row units, vocab
# sizes that are not multiples of the 256-row tile or of the 32-column argmax
# chunk, 4 and 8 bits, cap on and off.
TC_SHAPES = [
    (17, 256, 2000, 4, 30.0),   # the fewest rows that take the tensor-core forward
    (40, 2560, 1500, 4, 0.0),
    (64, 256, 1000, 4, 30.0),
    (128, 128, 256, 4, 0.0),
    (130, 384, 4099, 8, 30.0),
    (200, 256, 257, 8, 0.0),
    (300, 512, 3000, 4, 5.0),
    (257, 128, 31, 4, 0.0),
]


# Shapes on the weight-streaming forward (M <= 16) whose tiles span 5 or 20
# stages and whose scale table has 8k groups: the variant with compile-time
# ring slots and TMA-staged scales (4 and 8 bits, vocab sizes off the 256-row
# tile, one and two token groups); H = 1280 (20 groups) takes the other one.
STREAM_SHAPES = [
    (5, 2560, 3001, 4, 30.0),
    (13, 2560, 2000, 8, 0.0),
    (16, 2560, 1500, 4, 0.0),
    (6, 1280, 2500, 4, 30.0),
]


@pytest.mark.parametrize("M,H,V,bits,cap", STREAM_SHAPES)
def test_stream_forward_shapes(M, H, V, bits, cap):
    _run_all(_custom(M, H, V, bits, cap, seed=M * 11 + V))


@pytest.mark.parametrize("M,H,V,bits,cap", TC_SHAPES)
def test_tensor_core_forward_shapes(M, H, V, bits, cap):
    _run_all(_custom(M, H, V, bits, cap, seed=M * 7 + V))


# The largest hidden sizes the library accepts (H up to 8192): the
# weight-streaming forward with its shallowest ring (the staged h rows take
# most of shared memory), the tensor-core forward with 128 K steps per unit,
# and the backward with the finalize's widest rows.
MAX_H_SHAPES = [
    (5, 8192, 700, 4, 30.0),
    (9, 4096, 900, 8, 0.0),
    (40, 8192, 600, 8, 30.0),
    (130, 4096, 1100, 4, 5.0),
]


@pytest.mark.parametrize("M,H,V,bits,cap", MAX_H_SHAPES)
def test_max_hidden_sizes(M, H, V, bits, cap):
    _run_all(_custom(M, H, V, bits, cap, seed=M * 13 + V))


# Vocabularies of about a million rows (indices past 2^20; the streaming
# forward's splits and the tensor-core forward's 256-row tiles both ragged).
@pytest.mark.parametrize("M,H,V,bits,cap", [
    (5, 128, 1_000_003, 4, 30.0),
    (20, 128, 600_001, 8, 0.0),
])
def test_large_vocabularies(M, H, V, bits, cap):
    _run_all(_custom(M, H, V, bits, cap, seed=M + 17))


# Scales and biases in bf16 and fp32 (the page widens any float type): the
# weight-streaming forward (TMA-staged scales at H = 2560, cp.async at 1280)
# and the tensor-core forward, each with the tensor-core backward.
SB_SHAPES = [
    (5, 2560, 3001, 4, 30.0, "bf16"),
    (13, 1280, 2000, 8, 0.0, "f32"),
    (40, 256, 1500, 4, 30.0, "f32"),
    (130, 384, 4099, 8, 30.0, "bf16"),
    (300, 512, 3000, 4, 5.0, "f32"),
    (257, 256, 2049, 4, 0.0, "bf16"),
]


@pytest.mark.parametrize("M,H,V,bits,cap,sbt", SB_SHAPES)
def test_scale_bias_types(M, H, V, bits, cap, sbt):
    mask = synth.make_mask(M, 32, 0.25) if M > 100 else None
    _run_all(_custom(M, H, V, bits, cap, seed=M * 5 + V, mask=mask, sb_dtype=sbt))


def test_tensor_core_forward_masked():
    M = 333
    mask = synth.make_mask(M, 64, 0.4)
    _run_all(_custom(M, 256, 2000, 4, 30.0, seed=21, mask=mask))


@pytest.mark.parametrize("pattern", ["all", "none", "alternate", "spans"])
def test_masks(pattern):
    M = 40
    mask = {"all": np.zeros(M, np.uint8), "none": np.ones(M, np.uint8),
            "alternate": (np.arange(M) % 2).astype(np.uint8),
            "spans": synth.make_mask(M, 16, 0.3)}[pattern]
    _run_all(_custom(M, 256, 1500, 4, 30.0, seed=7, mask=mask))


def test_target_at_both_ends():
    M, V = 6, 3001
    _run_all(_custom(M, 256, V, 4, 30.0, seed=8, targets=[0, V - 1, 0, V - 1, 5, V - 2]))


def test_tied_rows_pick_lowest_index():
    # Vocab rows 17, 250 and 251 are identical and carry a bias large enough to
    # make them every token's maximum with one shared value: the argmax must be
    # the lowest of the tied indices, 17.  (Only the tie rule is asserted: with
    # all-positive h and repeated weights this head is outside the error model
    # of the workloads the lse tolerance is stated for.)
    M, H, V = 12, 256, 300
    wl = _custom(M, H, V, 4, 0.0, seed=9)
    hh = wl.head
    hh.biases[17] = np.float16(0.05)
    for r in (250, 251):
        hh.wq[r] = hh.wq[17]
        hh.scales[r] = hh.scales[17]
        hh.biases[r] = hh.biases[17]
    wl.h = synth.f32_to_bf16_bits(np.abs(oracle.widen_bf16(wl.h)).astype(np.float32))
    ref = oracle.forward(wl.h, oracle_head(wl.head), wl.targets)
    assert (ref.argmax == 17).all()
    head, h, t, mk, g = to_dev(wl)
    logp, lse, am = gpu_fwd(head, h, t, mk)
    assert (am == 17).all()


def test_verify_no_targets():
    wl = _custom(5, 512, 5000, 4, 30.0, seed=10)
    wl.targets = None
    head, h, t, mk, g = to_dev(wl)
    logp, lse, am = qhead.fwd(head, h, None, None)
    assert logp is None
    check_fwd(wl, np.arange(5), None, lse.cpu().numpy(), am.cpu().numpy())


def test_invalid_target_gives_nan_not_a_fault():
    wl = _custom(4, 256, 1000, 4, 0.0, seed=11, targets=[0, 1000, -3, 999])
    head, h, t, mk, g = to_dev(wl)
    logp, lse, am = gpu_fwd(head, h, t, mk)
    assert np.isnan(logp[1]) and np.isnan(logp[2])
    assert np.isfinite(logp[0]) and np.isfinite(logp[3])


def test_empty_batch_every_entry_point():
    # M = 0: every entry point returns empty results (and a zero head
    # gradient) without launching anything that could read past the inputs.
    wl = _custom(3, 256, 1000, 4, 30.0, seed=14)
    head, *_ = to_dev(wl)
    h = torch.empty(0, 256, dtype=torch.bfloat16, device="cuda")
    t = torch.empty(0, dtype=torch.int32, device="cuda")
    f = torch.empty(0, dtype=torch.float32, device="cuda")
    logp, lse, am = qhead.fwd(head, h, t)
    assert logp.numel() == 0 and lse.numel() == 0 and am.numel() == 0
    assert qhead.bwd(head, h, t, f, f).shape == (0, 256)
    dh, dw = qhead.bwd_dw(head, h, t, f, f, want_dh=True)
    torch.cuda.synchronize()
    assert dh.shape == (0, 256) and dw.shape == (1000, 256)
    assert torch.count_nonzero(dw).item() == 0
    dh, cold = qhead.bwd_filter(head, h, t, f, f, 1e-5)
    assert dh.shape == (0, 256)
    _, lse, _, bm = qhead.fwd_blockmax(head, h, t)
    assert bm.shape[0] == 0
    assert qhead.bwd_blockskip(head, h, t, f, f, bm, 1e-5).shape == (0, 256)
    n_acc, nxt, am, _ = qhead.verify(head, h, 5, torch.empty(0, 4, dtype=torch.int32, device="cuda"))
    assert n_acc.numel() == 0 and nxt.numel() == 0 and am.numel() == 0


def test_deterministic():
    wl = _custom(70, 256, 4000, 4, 30.0, seed=12, mask=synth.make_mask(70, 32, 0.25))
    head, h, t, mk, g = to_dev(wl)
    a = qhead.fwd(head, h, t, mk)
    b = qhead.fwd(head, h, t, mk)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    d1 = qhead.bwd(head, h, t, a[1], g, mk)
    d2 = qhead.bwd(head, h, t, a[1], g, mk)
    assert torch.equal(d1, d2)


def test_workspace_too_small_is_rejected():
    wl = _custom(9, 256, 2048, 4, 0.0, seed=13)
    head, h, t, mk, g = to_dev(wl)
    need = qhead.fwd_workspace(head, 9)
    ws = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(qhead.QheadError) as e:
        qhead.fwd(head, h, t, mk, workspace=ws)
    assert e.value.code == qhead.QHEAD_EINVAL


def test_workspace_sizes_of_the_variants():
    # Each variant's workspace covers its plan: the tensor-core plan for every
    # M where the variant needs it (tile maxima, skip maps, dW), a superset of
    # the exact backward's at M >= 64.
    wl = _custom(100, 256, 3000, 4, 30.0, seed=14)
    head = to_dev(wl)[0]
    c = ctypes.byref(head.c())
    L = qhead.lib()
    bad = ctypes.c_size_t(-1).value
    for m in (8, 100):
        f, b = L.qhead_fwd_workspace(c, m), L.qhead_bwd_workspace(c, m)
        for name in ("qhead_fwd_blockmax_workspace", "qhead_bwd_blockskip_workspace",
                     "qhead_bwd_filter_workspace", "qhead_bwd_dw_workspace"):
            assert getattr(L, name)(c, m) not in (0, bad), name
        assert f not in (0, bad) and b not in (0, bad)
        assert L.qhead_fwd_blockmax_workspace(c, m) >= f
    for name in ("qhead_bwd_blockskip_workspace", "qhead_bwd_filter_workspace",
                 "qhead_bwd_dw_workspace"):
        assert getattr(L, name)(c, 100) >= L.qhead_bwd_workspace(c, 100), name
        assert getattr(L, name)(c, 0) == 0, name


# ------------------------------------------------------------ full-size configs

_FULL = {}


def _full(name):
    if name not in _FULL:
        wl = synth.make_workload(name, seed=0)
        _FULL[name] = (wl, to_dev(wl))
    return _FULL[name]


def _sample_rows(wl, n, seed=0):
    """n seeded active rows, rows 0 and M - 1, and both sides of every mask
    boundary of every sequence."""
    rng = np.random.default_rng(seed)
    act = np.arange(wl.M) if wl.mask is None else np.nonzero(wl.mask)[0]
    rows = set(rng.choice(act, size=min(n, len(act)), replace=False).tolist())
    rows |= {0, wl.M - 1}
    n_boundary = 0
    if wl.mask is not None:
        for i in np.nonzero(np.diff(wl.mask.astype(int)))[0]:
            rows |= {int(i), int(i) + 1}
            n_boundary += 1
    return np.array(sorted(rows)), n_boundary


def test_full_verify_window():
    wl, (head, h, t, mk, g) = _full("verify")
    logp, lse, am = qhead.fwd(head, h, None, None)
    torch.cuda.synchronize()
    assert check_fwd(wl, np.arange(wl.M), None, lse.cpu().numpy(), am.cpu().numpy()) == wl.M


@pytest.mark.parametrize("sbt", ["bf16", "f32"])
def test_full_verify_window_bf16_and_f32_scales(sbt):
    # The verify head with its scales and biases in bf16 or fp32 (the
    # streaming kernel reads their per-call fp16 copy, the finalize the
    # caller's values): every position against the oracle.
    cfg = synth.CONFIGS["verify"]
    head = synth.make_head(cfg["V"], cfg["H"], cfg["bits"], softcap=cfg["softcap"], seed=0,
                           sb_dtype=sbt)
    wl = synth.Workload(
        "verify", head, synth.make_hidden(cfg["M"], cfg["H"], seed=0), None, None,
        np.ones(cfg["M"], np.float32), cfg)
    dhead, h, t, mk, g = to_dev(wl)
    logp, lse, am = qhead.fwd(dhead, h, None, None)
    torch.cuda.synchronize()
    assert check_fwd(wl, np.arange(wl.M), None, lse.cpu().numpy(), am.cpu().numpy()) == wl.M


def _full_step(name):
    """The workload's forward and backward on the GPU, exactly as the bench
    runs them, with the every-row properties checked."""
    wl, (head, h, t, mk, g) = _full(name)
    logp, lse, am = qhead.fwd(head, h, t, mk)
    dh = qhead.bwd(head, h, t, lse, g, mk)
    torch.cuda.synchronize()
    logp, lse_h, am = logp.cpu().numpy(), lse.cpu().numpy(), am.cpu().numpy()
    dh_h = dh.cpu().numpy()
    act = np.ones(wl.M, bool) if wl.mask is None else wl.mask.astype(bool)
    # properties on every row
    assert np.all(np.isfinite(logp)) and np.all(logp[act] <= 1e-6)
    assert np.all(np.isfinite(lse_h)) and np.all(lse_h[~act] == 0.0)
    assert np.all((am[act] >= 0) & (am[act] < wl.head.V)) and np.all(am[~act] == -1)
    assert np.all(dh_h[~act] == 0.0) and np.all(np.isfinite(dh_h))
    return wl, logp, lse_h, am, dh_h


def test_full_gemma512_every_forward_row():
    wl, logp, lse, am, dh = _full_step("gemma512")
    assert check_fwd(wl, np.arange(wl.M), logp, lse, am) == 512
    rows, _ = _sample_rows(wl, 256, seed=1)
    assert len(rows) >= 256
    check_dh(wl, rows, dh, label="gemma512")


def test_full_mid8_every_forward_row():
    wl, logp, lse, am, dh = _full_step("mid8")
    assert check_fwd(wl, np.arange(wl.M), logp, lse, am) == 8192
    rows, _ = _sample_rows(wl, 256, seed=2)
    check_dh(wl, rows, dh, label="mid8")


def test_full_gemma8k_masked_every_forward_row():
    wl, logp, lse, am, dh = _full_step("gemma8k_masked")
    # every row: the 5736 active ones against the oracle, the masked ones
    # against their sentinels
    assert check_fwd(wl, np.arange(wl.M), logp, lse, am) == 5736
    rows, n_boundary = _sample_rows(wl, 256, seed=3)
    assert n_boundary == 2 * 8 - 1  # prompt/response and response/next-prompt edges
    check_dh(wl, rows, dh, label="gemma8k_masked")
