"""Host-side checks of the Python binding's argument validation: every entry
point rejects, before it reaches the C library, per-row arguments whose dtype,
length or layout the kernels would misread (int64 token ids read as int32
pairs, a short tensor read past its end) and hidden states whose width is not
the head's H.  CPU tensors only; nothing here calls the library."""
import pytest
import torch

from verify_vocab_blocked_gb300 import autograd, qhead

M, H, V, BITS = 6, 256, 1000, 4


def _head():
    return qhead.Head(torch.zeros(V, H * BITS // 32, dtype=torch.int32),
                      torch.zeros(V, H // 64, dtype=torch.float16),
                      torch.zeros(V, H // 64, dtype=torch.float16), BITS)


def _h(m=M, h=H):
    return torch.zeros(m, h, dtype=torch.bfloat16)


def _t(dtype=torch.int32, n=M):
    return torch.zeros(n, dtype=dtype)


def _f(n=M, dtype=torch.float32):
    return torch.zeros(n, dtype=dtype)


def test_int64_targets_are_rejected():
    with pytest.raises(ValueError, match="targets must be int32"):
        qhead.fwd(_head(), _h(), _t(torch.int64))
    with pytest.raises(ValueError, match="targets must be int32"):
        qhead.bwd(_head(), _h(), _t(torch.int64), _f(), _f())


def test_wrong_hidden_size_is_rejected():
    with pytest.raises(ValueError, match="hidden size"):
        qhead.fwd(_head(), _h(h=H + 128), _t())
    with pytest.raises(ValueError, match="hidden size"):
        qhead.bwd(_head(), _h(h=128), _t(), _f(), _f())
    with pytest.raises(ValueError, match="hidden size"):
        qhead.verify(_head(), _h(m=5, h=512), 5, _t(n=4))


def test_short_per_row_tensors_are_rejected():
    with pytest.raises(ValueError, match=r"targets must have shape \[6\]"):
        qhead.fwd(_head(), _h(), _t(n=M - 1))
    with pytest.raises(ValueError, match=r"mask must have shape \[6\]"):
        qhead.fwd(_head(), _h(), _t(), torch.ones(M - 2, dtype=torch.uint8))
    with pytest.raises(ValueError, match=r"lse must have shape \[6\]"):
        qhead.bwd(_head(), _h(), _t(), _f(M - 1), _f())
    with pytest.raises(ValueError, match=r"dlogp must have shape \[6\]"):
        qhead.bwd_dw(_head(), _h(), _t(), _f(), _f(M + 1))


def test_wrong_dtypes_of_lse_dlogp_and_mask_are_rejected():
    with pytest.raises(ValueError, match="lse must be float32"):
        qhead.bwd(_head(), _h(), _t(), _f(dtype=torch.float64), _f())
    with pytest.raises(ValueError, match="dlogp must be float32"):
        qhead.bwd_filter(_head(), _h(), _t(), _f(), _f(dtype=torch.float16), 1e-5)
    with pytest.raises(ValueError, match="mask must be uint8 or bool"):
        qhead.fwd(_head(), _h(), _t(), torch.ones(M, dtype=torch.int32))


def test_non_contiguous_targets_are_rejected():
    t = torch.zeros(2 * M, dtype=torch.int32)[::2]
    with pytest.raises(ValueError, match="contiguous"):
        qhead.fwd(_head(), _h(), t)


def test_missing_targets_for_the_backward_are_rejected():
    with pytest.raises(ValueError, match="targets is required"):
        qhead.bwd(_head(), _h(), None, _f(), _f())


def test_block_max_shape_is_checked():
    bm = torch.zeros(M, 3, dtype=torch.float32)  # V = 1000 needs 4 vocab tiles
    with pytest.raises(ValueError, match="block_max"):
        qhead.bwd_blockskip(_head(), _h(), _t(), _f(), _f(), bm, 1e-5)


def test_autograd_wrapper_validates_through_the_binding():
    h = _h().requires_grad_(True)
    with pytest.raises(ValueError, match="targets must be int32"):
        autograd.head_logp(h, _head(), _t(torch.int64))


def test_scale_types_map_to_the_abi_codes():
    for dt, code in ((torch.float16, qhead.QHEAD_SB_F16), (torch.bfloat16, qhead.QHEAD_SB_BF16),
                     (torch.float32, qhead.QHEAD_SB_F32)):
        hd = qhead.Head(torch.zeros(V, H * BITS // 32, dtype=torch.int32),
                        torch.zeros(V, H // 64, dtype=dt), torch.zeros(V, H // 64, dtype=dt), BITS)
        assert hd.c().sb_dtype == code
    mixed = qhead.Head(torch.zeros(V, H * BITS // 32, dtype=torch.int32),
                       torch.zeros(V, H // 64, dtype=torch.float16),
                       torch.zeros(V, H // 64, dtype=torch.float32), BITS)
    with pytest.raises(ValueError, match="share one type"):
        mixed.c()


def test_bf16_scales_from_numpy_keep_their_bits():
    from verify_vocab_blocked_gb300 import synth
    sh = synth.make_head(300, 128, 4, seed=2, sb_dtype="bf16")
    hd = qhead.Head.from_numpy(sh.wq, sh.scales, sh.biases, 4, device="cpu", sb_dtype="bf16")
    assert hd.scales.dtype == torch.bfloat16
    assert (hd.scales.view(torch.int16).numpy().view("uint16") == sh.scales).all()
