"""The seeded synthetic inputs follow the stated recipe (they stand in for the
real heads and training data of the pages): field-uniform packed codes, the
scale and bias distributions of the 4- and 8-bit heads, N(0, 1) hidden
states rounded to bf16, uniform targets, masked prompt spans, the workload
shapes, and the logit scale that makes the flat workloads' softmax flat.
These check the generator only; none of the method's arithmetic is here."""
import numpy as np
import pytest

from verify_vocab_blocked_gb300 import synth


def _fields(wq: np.ndarray, bits: int) -> np.ndarray:
    per = 32 // bits
    w = wq.astype(np.uint64)
    return np.stack([(w >> np.uint64(bits * k)) & np.uint64((1 << bits) - 1)
                     for k in range(per)], axis=-1).reshape(-1)


@pytest.mark.parametrize("bits", [4, 8])
def test_codes_are_uniform_in_every_field(bits):
    head = synth.make_head(4096, 256, bits, seed=5)
    q = _fields(head.wq, bits).astype(np.int64)
    n = 1 << bits
    counts = np.bincount(q, minlength=n)
    assert counts.size == n
    # chi-square with n - 1 degrees of freedom, far inside its 1e-6 tail
    exp = q.size / n
    chi2 = float(((counts - exp) ** 2 / exp).sum())
    assert chi2 < (n - 1) + 12 * np.sqrt(2 * (n - 1))
    # and within every field position of a word (LSB-first packing)
    per = 32 // bits
    by_field = q.reshape(-1, per)
    assert np.allclose(by_field.mean(axis=0), (n - 1) / 2, atol=0.02 * n)


def test_four_bit_scales_and_biases():
    head = synth.make_head(8192, 256, 4, seed=6)
    s = head.scales.astype(np.float64)
    b = head.biases.astype(np.float64)
    assert head.scales.dtype == np.float16 and head.biases.dtype == np.float16
    assert s.min() >= 1e-3 * (1 - 2 ** -10) and s.max() <= 1e-2 * (1 + 2 ** -10)
    assert abs(s.mean() - 5.5e-3) < 1e-4                      # U(1e-3, 1e-2)
    resid = b + 8.0 * s                                        # = N(0, 1e-3) + rounding
    assert abs(resid.mean()) < 5e-5 and abs(resid.std() - 1e-3) < 5e-5


def test_eight_bit_scales_and_biases():
    head = synth.make_head(8192, 256, 8, seed=7)
    s = head.scales.astype(np.float64)
    b = head.biases.astype(np.float64)
    assert s.min() >= 1e-4 * (1 - 2 ** -10) and s.max() <= 1e-3 * (1 + 2 ** -10)
    assert abs(s.mean() - 5.5e-4) < 1e-5
    # bias = -128 scale before the fp16 rounding of each
    assert np.all(np.abs(b + 128.0 * s) <= 128.0 * s * 2 ** -10)


def test_hidden_states_targets_and_cotangents():
    h = synth.make_hidden(64, 2560, seed=8)
    assert h.dtype == np.uint16
    x = (h.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1.0) < 0.01
    hm = (synth.make_hidden(64, 2560, seed=8, mean=0.5).astype(np.uint32) << 16).view(np.float32)
    assert abs(float(hm.mean()) - 0.5) < 0.01
    t = synth.make_targets(200000, 1000, seed=9)
    assert t.dtype == np.int32 and t.min() >= 0 and t.max() < 1000
    assert np.bincount(t, minlength=1000).min() > 100
    g = synth.make_dlogp(100000, seed=9)
    assert g.min() >= -2.0 and g.max() <= 2.0 and abs(float(g.mean())) < 0.02


def test_masked_prompt_spans():
    mask = synth.make_mask(8192, 1024, 0.3)
    assert mask.sum() == 8 * (1024 - 307) == 5736
    for s0 in range(0, 8192, 1024):
        assert (mask[s0:s0 + 307] == 0).all() and (mask[s0 + 307:s0 + 1024] == 1).all()


def test_workload_shapes():
    want = {"tiny": (16, 256, 2048, 4, 0.0), "verify": (5, 2560, 262144, 4, 30.0),
            "mid8": (8192, 1536, 131072, 8, 0.0), "gemma512": (512, 2560, 262144, 4, 30.0),
            "gemma8k_masked": (8192, 2560, 262144, 4, 30.0)}
    for name, (M, H, V, bits, cap) in want.items():
        c = synth.CONFIGS[name]
        assert (c["M"], c["H"], c["V"], c["bits"], c["softcap"], c["group"]) == \
            (M, H, V, bits, cap, 64), name
    assert synth.CONFIGS["verify"]["bwd"] is False
    assert synth.CONFIGS["gemma8k_masked"]["mask"] == (1024, 0.3)


def test_logit_scale_of_the_flat_workloads():
    # std of h . w over random rows: sqrt(H E[w^2]) = 1.43 at H = 2560 (4-bit)
    # and 1.76 at H = 1536 (8-bit), so the softmax over 2^17..2^18 rows is flat
    for bits, H, want in ((4, 2560, 1.43), (8, 1536, 1.76)):
        head = synth.make_head(512, H, bits, seed=10)
        q = _fields(head.wq, bits).reshape(512, H).astype(np.float64)
        s = np.repeat(head.scales.astype(np.float64), 64, axis=1)
        b = np.repeat(head.biases.astype(np.float64), 64, axis=1)
        w = s * q + b
        x = (synth.make_hidden(64, H, seed=10).astype(np.uint32) << 16).view(np.float32)
        raw = x.astype(np.float64) @ w.T
        assert abs(raw.std() - want) < 0.05 * want, (bits, raw.std())


@pytest.mark.parametrize("sb_dtype", ["f16", "bf16", "f32"])
def test_peaked_head_raises_only_the_hot_rows_biases(sb_dtype):
    # The peaked head is make_head's head with the group biases of n_hot rows
    # raised by bias_shift, rounded to the scales' own type; nothing else moves.
    base = synth.make_head(3000, 256, 4, softcap=30.0, seed=41, sb_dtype=sb_dtype)
    head, hot = synth.make_peaked_head(3000, 256, 4, n_hot=8, bias_shift=0.3, softcap=30.0,
                                       seed=41, sb_dtype=sb_dtype)
    assert head.biases.dtype == base.biases.dtype and head.sb_dtype == sb_dtype
    assert (head.wq == base.wq).all() and (head.scales == base.scales).all()

    def as_f64(b):
        if sb_dtype == "bf16":
            return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        return b.astype(np.float64)

    diff = as_f64(head.biases) - as_f64(base.biases)
    changed = np.flatnonzero(np.abs(diff).max(axis=1) > 0)
    assert np.array_equal(changed, np.sort(hot)) and len(hot) == 8
    step = {"f16": 2.0 ** -10, "bf16": 2.0 ** -7, "f32": 2.0 ** -23}[sb_dtype]
    # raised by 0.3 up to one rounding of the sum (|bias| < 1 here)
    assert np.allclose(diff[hot], 0.3, atol=step)
