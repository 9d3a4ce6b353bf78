"""The fused verify + accept step (qhead_verify) against the oracle.

CPU: the oracle's accept loop pinned by hand-worked windows and by an
independent formulation (a cumulative product of matches).  GPU: qhead_verify
returns the argmax qhead_fwd returns, and its accepted-prefix lengths and next
tokens equal the oracle's accept loop applied to that argmax (exactly), and to
the oracle's own argmax wherever every decisive position has a top-2 gap
above 1e-3.
"""
import numpy as np
import pytest
import torch

import oracle
from parity import GAP_TOL, oracle_head, to_dev
from verify_vocab_blocked_gb300 import build as qbuild
from verify_vocab_blocked_gb300 import qhead, synth


# ---------------------------------------------------------------- CPU pins

@pytest.mark.parametrize("argmax,draft,n,nxt", [
    ([7, 3, 9, 4, 2], [7, 3, 9, 4], 4, 2),   # every draft token accepted: bonus token
    ([7, 3, 9, 4, 2], [7, 3, 8, 4], 2, 9),   # first mismatch at k = 2
    ([7, 3, 9, 4, 2], [1, 3, 9, 4], 0, 7),   # rejected at once
    ([5], [], 0, 5),                          # gamma = 0: the target's own token
    ([7, -1, 9], [7, 1], 1, -1),              # a masked position (argmax -1) never matches
])
def test_accept_worked_windows(argmax, draft, n, nxt):
    W = len(argmax)
    got_n, got_next = oracle.accept_prefix(np.array(argmax), np.array(draft, np.int64), W)
    assert got_n.tolist() == [n] and got_next.tolist() == [nxt]


def test_accept_matches_cumulative_product():
    rng = np.random.default_rng(11)
    B, W = 200, 9
    argmax = rng.integers(0, 4, size=(B, W))
    draft = np.where(rng.random((B, W - 1)) < 0.8, argmax[:, :-1], rng.integers(0, 4, (B, W - 1)))
    n, nxt = oracle.accept_prefix(argmax.ravel(), draft, W)
    n2 = np.cumprod(draft == argmax[:, :-1], axis=1).sum(axis=1)
    assert np.array_equal(n, n2)
    assert np.array_equal(nxt, argmax[np.arange(B), n2])


def test_accept_on_oracle_argmax():
    # Drafts built from the oracle's own argmax of a tiny head: a draft equal
    # to the argmax is accepted whole; changing token j stops the prefix at j.
    head = synth.make_head(300, 128, 4, softcap=30.0, seed=4)
    h = synth.make_hidden(3 * 4, 128, seed=4)
    am = oracle.forward(h, oracle_head(head)).argmax.reshape(3, 4)
    draft = am[:, :3].copy()
    draft[1, 2] = (draft[1, 2] + 1) % 300
    draft[2, 0] = (draft[2, 0] + 1) % 300
    n, nxt = oracle.accept_prefix(am.ravel(), draft, 4)
    assert n.tolist() == [3, 2, 0]
    assert nxt.tolist() == [am[0, 3], am[1, 2], am[2, 0]]


# ---------------------------------------------------------------- GPU parity

@pytest.fixture(scope="module")
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    qbuild.build()
    qhead.lib()


def _windows(B, W, H, V, bits, cap, seed, mask=None):
    head = synth.make_head(V, H, bits, softcap=cap, seed=seed)
    h = synth.make_hidden(B * W, H, seed=seed)
    return synth.Workload("verify", head, h, None, mask, np.ones(B * W, np.float32), {})


@pytest.mark.gpu
@pytest.mark.parametrize("B,W,H,V,bits,cap", [
    (4, 5, 256, 3000, 4, 30.0),      # the gamma = 4 window, weight-streaming path
    (3, 33, 256, 2000, 4, 0.0),      # windows longer than a warp
    (20, 5, 384, 1500, 8, 30.0),     # 100 rows: tensor-core path
    (1, 1, 128, 700, 4, 0.0),        # gamma = 0
])
def test_verify_accept_parity(_gpu, B, W, H, V, bits, cap):
    wl = _windows(B, W, H, V, bits, cap, seed=B * 31 + W)
    ref = oracle.forward(wl.h, oracle_head(wl.head))
    am_ref = ref.argmax.reshape(B, W)
    rng = np.random.default_rng(B + W)
    # Drafts: the oracle argmax with one token changed at a random position
    # (or none) per window.
    draft = am_ref[:, :-1].copy()
    cut = rng.integers(0, W, size=B)  # cut == W - 1 keeps the whole draft
    for b in range(B):
        if cut[b] < W - 1:
            draft[b, cut[b]] = (draft[b, cut[b]] + 1) % V
    head, h, _, _, _ = to_dev(wl)
    d = torch.from_numpy(draft.astype(np.int32)).cuda() if W > 1 else None
    n, nxt, am, lse = qhead.verify(head, h, W, d, want_lse=True)
    torch.cuda.synchronize()
    n, nxt, am, lse = n.cpu().numpy(), nxt.cpu().numpy(), am.cpu().numpy(), lse.cpu().numpy()
    # same argmax and lse as the plain forward
    _, lse_f, am_f = qhead.fwd(head, h)
    torch.cuda.synchronize()
    assert np.array_equal(am, am_f.cpu().numpy())
    assert np.array_equal(lse, lse_f.cpu().numpy())
    # the accept step applied to the GPU's own argmax, exactly
    n_own, nxt_own = oracle.accept_prefix(am, draft, W)
    assert np.array_equal(n, n_own) and np.array_equal(nxt, nxt_own)
    # and the oracle's decision wherever the decisive positions are not near-ties
    gap = ref.gap.reshape(B, W)
    n_ref, nxt_ref = oracle.accept_prefix(ref.argmax, draft, W)
    for b in range(B):
        decisive = gap[b, : n_ref[b] + 1]
        if np.all(decisive > GAP_TOL):
            assert n[b] == n_ref[b] and nxt[b] == nxt_ref[b], b


@pytest.mark.gpu
def test_verify_masked_position_stops_the_prefix(_gpu):
    B, W = 2, 5
    mask = np.ones(B * W, np.uint8)
    mask[1 * W + 2] = 0  # window 1, position 2
    wl = _windows(B, W, 256, 2500, 4, 30.0, seed=77, mask=mask)
    head, h, _, mk, _ = to_dev(wl)
    _, _, am_full = qhead.fwd(head, h)
    am_full = am_full.cpu().numpy().reshape(B, W)
    draft = torch.from_numpy(am_full[:, :-1].astype(np.int32).copy()).cuda()
    n, nxt, am, _ = qhead.verify(head, h, W, draft, mk)
    torch.cuda.synchronize()
    am = am.cpu().numpy()
    assert am[1 * W + 2] == -1
    assert n.cpu().tolist() == [W - 1, 2]
    assert nxt.cpu().tolist()[1] == -1
