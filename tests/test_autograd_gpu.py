"""The torch.autograd wrapper: its forward is qhead_fwd's logp, its backward
is qhead_bwd's dh for the incoming cotangent, and both match the oracle."""
import numpy as np
import pytest
import torch

import oracle
from parity import check_dh, to_dev
from verify_vocab_blocked_gb300 import build as qbuild
from verify_vocab_blocked_gb300 import qhead, synth
from verify_vocab_blocked_gb300.autograd import head_logp

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    qbuild.build()
    qhead.lib()


@pytest.mark.parametrize("M,H,V,bits,cap,masked", [
    (12, 256, 2000, 4, 30.0, False),   # weight-streaming forward, CUDA-core backward
    (150, 256, 1800, 8, 0.0, True),    # tensor-core forward and backward
])
def test_autograd_matches_library_and_oracle(M, H, V, bits, cap, masked):
    mask = synth.make_mask(M, 16, 0.3) if masked else None
    head_np = synth.make_head(V, H, bits, softcap=cap, seed=M)
    h_np = synth.make_hidden(M, H, seed=M)
    t_np = synth.make_targets(M, V, seed=M)
    w = np.random.default_rng(M).uniform(-1.0, 1.0, size=M).astype(np.float32)
    wl = synth.Workload("autograd", head_np, h_np, t_np, mask, w, {})
    head, h, t, mk, _ = to_dev(wl)
    hx = h.clone().requires_grad_(True)
    logp = head_logp(hx, head, t, mk)
    # the forward is qhead_fwd's logp
    ref_logp, lse, _ = qhead.fwd(head, h, t, mk)
    assert torch.equal(logp.detach(), ref_logp)
    # loss = sum_m w[m] logp[m]  ->  dh = qhead_bwd(dlogp = w), cast to bf16
    wt = torch.from_numpy(w).cuda()
    (logp * wt).sum().backward()
    dh_lib = qhead.bwd(head, h, t, lse, wt, mk)
    torch.cuda.synchronize()
    assert hx.grad.dtype == torch.bfloat16
    assert torch.equal(hx.grad, dh_lib.to(torch.bfloat16))
    # and the library's fp32 dh matches the oracle for this cotangent
    check_dh(wl, np.arange(M), dh_lib.cpu().numpy())
