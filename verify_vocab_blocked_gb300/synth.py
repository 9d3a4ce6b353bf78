"""Seeded synthetic inputs for the fused quantized LM-head.

This module only draws random inputs; it holds none of the head's arithmetic
and imports nothing else from this package, so both the CUDA path and the CPU
oracle can be fed from it.  Everything is generated on the host with numpy's
Philox counter-based generator, one independent stream per tensor.

The workloads stand in for the Gemma-class (V=262144, H=2560) and
MiniCPM-class (H=1536) heads the pages train and decode with; real weights
and real training data are not used.

Recipes (per tensor):
  * packed codes: each code uniform on [0, 2^bits - 1], independent.  With
    32/bits fields per word that is exactly a uniform uint32 word, which is how
    it is drawn (fields are least-significant first by the format's
    definition, and uniformity makes the order irrelevant to the draw).
  * 4-bit heads: scale ~ U(1e-3, 1e-2); bias = -8*scale + N(0, 1e-3); both
    rounded to fp16 (round to nearest even) from the unrounded draws.
  * 8-bit heads: scale ~ U(1e-4, 1e-3); bias = -128*scale; both rounded to fp16.
  * hidden states: N(0, 1) drawn in float32, rounded to bf16 (nearest even).
  * targets: uniform on [0, V).
  * response mask (1 = token contributes, 0 = masked prompt token): sequences
    of `seq_len` tokens, each starting with a contiguous masked prompt span of
    round(masked_frac * seq_len) tokens.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

# Named workloads: shapes, bit widths and soft caps of the five cases the
# head is checked and measured on.
CONFIGS: dict[str, dict] = {
    "tiny": dict(M=16, H=256, V=2048, bits=4, group=64, softcap=0.0, mask=None,
                 bwd=True, desc="tiny correctness: M=16, H=256, V=2048, 4-bit, no cap"),
    "verify": dict(M=5, H=2560, V=262144, bits=4, group=64, softcap=30.0, mask=None,
                   bwd=False, targets=False,
                   desc="spec-decode verify window: M=5 (gamma=4 + 1), H=2560, V=262144, "
                        "4-bit, softcap 30, forward only"),
    "mid8": dict(M=8192, H=1536, V=131072, bits=8, group=64, softcap=0.0, mask=None,
                 bwd=True, desc="mid-size training head: M=8192, H=1536, V=131072, 8-bit"),
    "gemma512": dict(M=512, H=2560, V=262144, bits=4, group=64, softcap=30.0, mask=None,
                     bwd=True, desc="Gemma-class head, M=512, H=2560, V=262144, 4-bit, cap 30"),
    "gemma8k_masked": dict(M=8192, H=2560, V=262144, bits=4, group=64, softcap=30.0,
                           mask=(1024, 0.3), bwd=True,
                           desc="Gemma-class head, M=8192 with 30% masked prompt spans "
                                "(8 x 1024-token sequences), H=2560, V=262144, 4-bit, cap 30"),
    # A peaked softmax for the approximate blockMax early exit (not one of the
    # five parity workloads): 64 hot vocab rows with every group bias raised
    # by 0.03, hidden states of mean 0.5 (so the hot logits sit ~38 above the
    # rest before the cap), 90% of the targets hot.
    "gemma8k_peaked": dict(M=8192, H=2560, V=262144, bits=4, group=64, softcap=30.0,
                           mask=(1024, 0.3), bwd=True,
                           peaked=dict(n_hot=64, bias_shift=0.03, h_mean=0.5, hot_frac=0.9),
                           desc="Gemma-class head with a peaked softmax (64 hot vocab rows, "
                                "90% hot targets), M=8192 with 30% masked prompt spans, "
                                "H=2560, V=262144, 4-bit, cap 30"),
}

_STREAMS = {"wq": 1, "scales": 2, "bias_noise": 3, "h": 4, "targets": 5, "dlogp": 6, "hot": 7,
            "hot_targets": 8}


def _rng(seed: int, stream: str) -> np.random.Generator:
    return np.random.Generator(np.random.Philox(key=[seed, _STREAMS[stream]]))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); returns uint16 bits.
    Inputs must be finite."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float64 values to bf16 (nearest, ties to even, in one rounding);
    returns uint16 bits.  Inputs must be finite and within bf16's normal range
    or zero."""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)                     # x = m * 2^e, 0.5 <= |m| < 1
    q = np.round(m * 256.0) / 256.0        # 8 significant bits, ties to even
    return f32_to_bf16_bits(np.ldexp(q, e).astype(np.float32))


@dataclass
class SynthHead:
    wq: np.ndarray        # uint32 [V, H*bits/32]
    scales: np.ndarray    # [V, H/group]: float16, bf16 bits (uint16) or float32
    biases: np.ndarray    # [V, H/group], the same type as scales
    bits: int
    group: int
    softcap: float
    sb_dtype: str = "f16"

    @property
    def V(self) -> int:
        return int(self.wq.shape[0])

    @property
    def H(self) -> int:
        return int(self.wq.shape[1]) * 32 // self.bits


def make_head(V: int, H: int, bits: int, group: int = 64, softcap: float = 0.0,
              seed: int = 0, chunk_rows: int = 1 << 16, sb_dtype: str = "f16") -> SynthHead:
    """sb_dtype: the element type scales and biases are rounded to from their
    unrounded draws -- "f16" (float16 arrays), "bf16" (uint16 bit patterns)
    or "f32" (float32 arrays)."""
    if bits not in (4, 8):
        raise ValueError("bits must be 4 or 8")
    if H % group:
        raise ValueError("H must be a multiple of the group size")
    wpr = H * bits // 32
    G = H // group
    rw = _rng(seed, "wq")
    wq = np.empty((V, wpr), dtype=np.uint32)
    for r0 in range(0, V, chunk_rows):
        r1 = min(V, r0 + chunk_rows)
        wq[r0:r1] = rw.integers(0, 1 << 32, size=(r1 - r0, wpr), dtype=np.uint32)
    rs = _rng(seed, "scales")
    if bits == 4:
        s = rs.uniform(1e-3, 1e-2, size=(V, G))
        noise = _rng(seed, "bias_noise").normal(0.0, 1e-3, size=(V, G))
        b = -8.0 * s + noise
    else:
        s = rs.uniform(1e-4, 1e-3, size=(V, G))
        b = -128.0 * s
    if sb_dtype == "f16":
        sr, br = s.astype(np.float16), b.astype(np.float16)
    elif sb_dtype == "f32":
        sr, br = s.astype(np.float32), b.astype(np.float32)
    elif sb_dtype == "bf16":
        sr, br = f64_to_bf16_bits(s), f64_to_bf16_bits(b)
    else:
        raise ValueError("sb_dtype must be f16, bf16 or f32")
    return SynthHead(wq, sr, br, bits, group, float(softcap), sb_dtype)


def make_hidden(M: int, H: int, seed: int = 0, mean: float = 0.0) -> np.ndarray:
    """bf16 bit patterns (uint16 [M,H]) of N(mean,1) draws."""
    x = _rng(seed, "h").standard_normal(size=(M, H), dtype=np.float32)
    if mean:
        x = x + np.float32(mean)
    return f32_to_bf16_bits(x)


def make_peaked_head(V: int, H: int, bits: int, n_hot: int, bias_shift: float,
                     softcap: float = 0.0, seed: int = 0,
                     sb_dtype: str = "f16") -> tuple[SynthHead, np.ndarray]:
    """A head as make_head draws it, with every group bias of n_hot vocab rows
    (drawn uniformly without replacement) raised by bias_shift (rounded to
    the scales' type).  With hidden states of positive mean
    (make_hidden(mean=...)), those rows dominate every token's softmax: a
    peaked distribution, where most vocab tiles carry negligible probability.
    Returns (head, hot rows)."""
    head = make_head(V, H, bits, softcap=softcap, seed=seed, sb_dtype=sb_dtype)
    hot = np.sort(_rng(seed, "hot").choice(V, size=n_hot, replace=False))
    if sb_dtype == "bf16":
        b = (head.biases.astype(np.uint32) << 16).view(np.float32).copy()
    else:
        b = head.biases.astype(np.float32)
    b[hot] += np.float32(bias_shift)
    head.biases = (f32_to_bf16_bits(b) if sb_dtype == "bf16"
                   else b.astype(np.float32 if sb_dtype == "f32" else np.float16))
    return head, hot


def make_targets(M: int, V: int, seed: int = 0) -> np.ndarray:
    return _rng(seed, "targets").integers(0, V, size=M, dtype=np.int64).astype(np.int32)


def make_dlogp(M: int, seed: int = 0) -> np.ndarray:
    """A non-trivial per-token cotangent (uniform on [-2, 2]) for tests."""
    return _rng(seed, "dlogp").uniform(-2.0, 2.0, size=M).astype(np.float32)


def make_mask(M: int, seq_len: int, masked_frac: float) -> np.ndarray:
    """1 = response token (contributes), 0 = masked prompt token."""
    mask = np.ones(M, dtype=np.uint8)
    n_prompt = int(round(masked_frac * seq_len))
    for s0 in range(0, M, seq_len):
        mask[s0:min(M, s0 + n_prompt)] = 0
    return mask


@dataclass
class Workload:
    name: str
    head: SynthHead
    h: np.ndarray                 # uint16 bf16 bits [M,H]
    targets: np.ndarray | None    # int32 [M]
    mask: np.ndarray | None       # uint8 [M]
    dlogp: np.ndarray             # float32 [M]
    cfg: dict = field(default_factory=dict)

    @property
    def M(self) -> int:
        return int(self.h.shape[0])


def make_workload(name: str, seed: int = 0, M: int | None = None,
                  head: SynthHead | None = None) -> Workload:
    """The named workload.  `head`, if given, replaces the head this call would
    draw (it must be the one make_head draws for the same shape and seed, e.g.
    from another workload with the same head parameters)."""
    cfg = dict(CONFIGS[name])
    M = cfg["M"] if M is None else M
    pk = cfg.get("peaked")
    if head is not None:
        if pk or (head.V, head.H, head.bits, head.group, head.softcap) != (
                cfg["V"], cfg["H"], cfg["bits"], cfg["group"], cfg["softcap"]):
            raise ValueError(f"the given head does not have {name}'s parameters")
        h = make_hidden(M, cfg["H"], seed)
    elif pk:
        head, hot = make_peaked_head(cfg["V"], cfg["H"], cfg["bits"], pk["n_hot"],
                                     pk["bias_shift"], cfg["softcap"], seed)
        h = make_hidden(M, cfg["H"], seed, mean=pk["h_mean"])
    else:
        head = make_head(cfg["V"], cfg["H"], cfg["bits"], cfg["group"], cfg["softcap"], seed)
        h = make_hidden(M, cfg["H"], seed)
    targets = make_targets(M, cfg["V"], seed) if cfg.get("targets", True) else None
    if pk and targets is not None:
        rt = _rng(seed, "hot_targets")
        pick = rt.random(M) < pk["hot_frac"]
        targets[pick] = hot[rt.integers(0, len(hot), size=int(pick.sum()))].astype(np.int32)
    mask = make_mask(M, cfg["mask"][0], cfg["mask"][1]) if cfg["mask"] else None
    dlogp = np.ones(M, dtype=np.float32)
    return Workload(name, head, h, targets, mask, dlogp, cfg)
