"""fp64 CPU oracle for the fused quantized LM-head -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The CUDA
library never calls it and shares no code with it.

The arithmetic lives in ``qhead_oracle.c`` (plain C, fp64, OpenMP over
independent outputs); this module only builds that file with gcc, marshals
numpy arrays and strings the steps together in the order the method defines
them (page "mlx-bun 0.0.4 -> 0.0.6", src/train/flash-cce.ts):

1. dequantize  w[v,d] = scale[v,d//group] * q[v,d] + bias[v,d//group]
2. raw = h @ w.T
3. z = cap*tanh(raw/cap) if cap > 0 else raw
4. lse = logsumexp_v z;  logp = z[target] - lse;  argmax = first argmax of raw
5. dh = sum_v dlogp*(onehot - exp(z - lse))*sech2 * w[v,:]
6. (the head gradient, a variant the pages leave out because their head is
   frozen) dW[v,:] = sum_m dlogp*(onehot - exp(z - lse))*sech2 * h[m,:]
7. (the approximate blockMax early exit) per-vocab-tile maxima of z, and dh
   with the (row tile, vocab tile) blocks whose rows all lie below
   lse + ln(eps) and hold no target dropped

and the speculative-decode accept step (page "mlx-bun 0.0.8 -> 0.0.10",
src/spec/generate.ts): per window of gamma + 1 positions, the longest prefix of
the draft that the argmax reproduces, and the token after it.

Masked rows (mask == 0) are skipped: logp = lse = 0, argmax = -1, dh = 0.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qhead_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None

_f64p = ctypes.POINTER(ctypes.c_double)
_u32p = ctypes.POINTER(ctypes.c_uint32)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_i32p = ctypes.POINTER(ctypes.c_int32)
_i64p = ctypes.POINTER(ctypes.c_int64)
_u8p = ctypes.POINTER(ctypes.c_uint8)
_i64 = ctypes.c_int64
_int = ctypes.c_int


def build(force: bool = False) -> str:
    """Compile qhead_oracle.c into liboracle.so (gcc, -O2, OpenMP, no fast-math,
    no FMA contraction so x86 and Arm hosts give the same bits)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    lib.oracle_widen_bf16.argtypes = [_u16p, _f64p, _i64]
    lib.oracle_widen_f16.argtypes = [_u16p, _f64p, _i64]
    lib.oracle_codes.argtypes = [_u32p, _i64, _i64, _int, _u32p]
    lib.oracle_dequant.argtypes = [_u32p, _f64p, _f64p, _i64, _i64, _int, _int, _f64p]
    lib.oracle_logits.argtypes = [_i64, _i64, _i64, _int, _int, _f64p, _u32p, _f64p, _f64p,
                                  _f64p, _int]
    lib.oracle_row_stats.argtypes = [_i64, _i64, ctypes.c_double, _f64p, _i32p, _u8p, _f64p,
                                     _f64p, _i64p, _f64p, _f64p, _int]
    lib.oracle_coeff.argtypes = [_i64, _i64, ctypes.c_double, _f64p, _f64p, _i32p, _u8p,
                                 _f64p, _int]
    lib.oracle_dh.argtypes = [_i64, _i64, _i64, _int, _int, _u32p, _f64p, _f64p, _f64p,
                              _f64p, _int]
    lib.oracle_dw.argtypes = [_i64, _i64, _i64, _f64p, _f64p, _f64p, _int]
    lib.oracle_num_threads.argtypes = [_int]
    lib.oracle_num_threads.restype = _int
    _lib = lib
    return lib


def _ptr(a: np.ndarray | None, ctype):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(ctype)


def num_threads(threads: int = 0) -> int:
    """Threads the oracle's OpenMP loops use for ``threads`` (0 = all cores)."""
    return int(_load().oracle_num_threads(threads))


# ------------------------------------------------------------------ widening

def widen_bf16(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64, exactly."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(b.shape, dtype=np.float64)
    _load().oracle_widen_bf16(_ptr(b, _u16p), _ptr(out, _f64p), b.size)
    return out


def widen_f16(bits: np.ndarray) -> np.ndarray:
    """IEEE binary16 bit patterns (uint16, or a float16 array) -> float64, exactly."""
    b = np.ascontiguousarray(bits)
    if b.dtype == np.float16:
        b = b.view(np.uint16)
    b = np.ascontiguousarray(b.astype(np.uint16, copy=False))
    out = np.empty(b.shape, dtype=np.float64)
    _load().oracle_widen_f16(_ptr(b, _u16p), _ptr(out, _f64p), b.size)
    return out


def _as_f64_h(h: np.ndarray) -> np.ndarray:
    """Hidden states: uint16 arrays are bf16 bit patterns; float64 is taken as is."""
    if h.dtype == np.uint16:
        return widen_bf16(h)
    if h.dtype == np.float64:
        return np.ascontiguousarray(h)
    raise TypeError(f"oracle: h must be bf16 bits (uint16) or float64, got {h.dtype}")


def _as_f64_sb(x: np.ndarray, sb_dtype: str = "f16") -> np.ndarray:
    """Scales/biases widened exactly to float64 (the page casts any float type
    to f32 before the dequantization): float16 (or its uint16 bits, with
    sb_dtype "f16"), bf16 bit patterns (uint16, sb_dtype "bf16"), float32
    (every binary32 value is a binary64 value); float64 is taken as is."""
    if x.dtype == np.float64:
        return np.ascontiguousarray(x)
    if sb_dtype == "bf16":
        if x.dtype != np.uint16:
            raise TypeError(f"oracle: bf16 scales/biases are uint16 bit patterns, got {x.dtype}")
        return widen_bf16(x)
    if sb_dtype == "f32":
        if x.dtype != np.float32:
            raise TypeError(f"oracle: f32 scales/biases must be float32, got {x.dtype}")
        return np.ascontiguousarray(x, dtype=np.float64)
    if x.dtype in (np.float16, np.uint16):
        return widen_f16(x)
    raise TypeError(f"oracle: scales/biases must be float16, bf16 bits, float32 or float64, "
                    f"got {x.dtype}")


# -------------------------------------------------------------------- head

@dataclass
class Head:
    """The quantized head (FlashCceHead on the page): packed codes, per-group
    affine scale and bias, bit width, group size and the optional soft cap."""
    wq: np.ndarray          # uint32 [V, H*bits/32]
    scales: np.ndarray      # [V, H/group]: float16, bf16 bits (uint16), float32 or float64
    biases: np.ndarray      # [V, H/group], the same type as scales
    bits: int
    group: int = 64
    softcap: float = 0.0
    sb_dtype: str = "f16"   # "f16", "bf16" or "f32": how uint16 / float32 arrays are read

    def sb(self):
        """(scales, biases) widened exactly to float64."""
        return _as_f64_sb(self.scales, self.sb_dtype), _as_f64_sb(self.biases, self.sb_dtype)

    @property
    def V(self) -> int:
        return int(self.wq.shape[0])

    @property
    def H(self) -> int:
        return int(self.wq.shape[1]) * 32 // self.bits


def codes(wq: np.ndarray, H: int, bits: int) -> np.ndarray:
    """Unpacked codes q[v,d] (uint32 [V,H])."""
    wq = np.ascontiguousarray(wq, dtype=np.uint32)
    V = wq.shape[0]
    out = np.empty((V, H), dtype=np.uint32)
    _load().oracle_codes(_ptr(wq, _u32p), V, H, bits, _ptr(out, _u32p))
    return out


def dequant(head: Head) -> np.ndarray:
    """Dense fp64 head w[v,d] (for small heads only: V*H doubles)."""
    wq = np.ascontiguousarray(head.wq, dtype=np.uint32)
    s, b = head.sb()
    out = np.empty((head.V, head.H), dtype=np.float64)
    _load().oracle_dequant(_ptr(wq, _u32p), _ptr(s, _f64p), _ptr(b, _f64p), head.V, head.H,
                           head.bits, head.group, _ptr(out, _f64p))
    return out


def _check(head: Head, hf: np.ndarray):
    if head.bits not in (2, 4, 8):
        raise ValueError(f"oracle: bits={head.bits}")
    if head.H % head.group or head.group % (32 // head.bits):
        raise ValueError("oracle: H must be a multiple of group, group of 32/bits")
    if hf.ndim != 2 or hf.shape[1] != head.H:
        raise ValueError(f"oracle: h shape {hf.shape} vs H={head.H}")


def logits(h: np.ndarray, head: Head, threads: int = 0) -> np.ndarray:
    """raw[m,v] = sum_d h[m,d] w[v,d]  (fp64 [M,V])."""
    hf = _as_f64_h(h)
    _check(head, hf)
    wq = np.ascontiguousarray(head.wq, dtype=np.uint32)
    s, b = head.sb()
    M = hf.shape[0]
    raw = np.empty((M, head.V), dtype=np.float64)
    _load().oracle_logits(M, head.H, head.V, head.bits, head.group, _ptr(hf, _f64p),
                          _ptr(wq, _u32p), _ptr(s, _f64p), _ptr(b, _f64p), _ptr(raw, _f64p),
                          threads)
    return raw


@dataclass
class Forward:
    logp: np.ndarray | None  # float64 [M] (None when no targets)
    lse: np.ndarray          # float64 [M]
    argmax: np.ndarray       # int64 [M], -1 on masked rows
    gap: np.ndarray          # float64 [M], top-2 gap of the capped logits
    zmax: np.ndarray         # float64 [M]
    raw: np.ndarray | None   # float64 [M,V] when keep_raw


def _targets(targets, M):
    if targets is None:
        return None
    t = np.ascontiguousarray(targets, dtype=np.int32)
    if t.shape != (M,):
        raise ValueError("oracle: targets must be [M]")
    return t


def _mask(mask, M):
    if mask is None:
        return None
    mk = np.ascontiguousarray(mask, dtype=np.uint8)
    if mk.shape != (M,):
        raise ValueError("oracle: mask must be [M]")
    return mk


def forward(h: np.ndarray, head: Head, targets=None, mask=None, threads: int = 0,
            keep_raw: bool = False) -> Forward:
    """logp, lse, argmax (and the top-2 gap of z) for every row of h."""
    raw = logits(h, head, threads)
    M, V = raw.shape
    t = _targets(targets, M)
    if t is not None and M and (t.min() < 0 or t.max() >= V):
        raise ValueError("oracle: target out of range")
    mk = _mask(mask, M)
    logp = np.empty(M) if t is not None else None
    lse, gap, zmax = np.empty(M), np.empty(M), np.empty(M)
    am = np.empty(M, dtype=np.int64)
    _load().oracle_row_stats(M, V, float(head.softcap), _ptr(raw, _f64p), _ptr(t, _i32p),
                             _ptr(mk, _u8p), _ptr(logp, _f64p), _ptr(lse, _f64p),
                             _ptr(am, _i64p), _ptr(gap, _f64p), _ptr(zmax, _f64p), threads)
    return Forward(logp, lse, am, gap, zmax, raw if keep_raw else None)


def _coeff(h: np.ndarray, head: Head, targets, dlogp, mask, lse, threads: int):
    """coeff[m,v] = dlogp[m] (1[v = t_m] - p[m,v]) sech2[m,v]  (fp64 [M,V]; 0 on
    masked rows), the factor both gradients share."""
    raw = logits(h, head, threads)
    M, V = raw.shape
    t = _targets(targets, M)
    if t is None:
        raise ValueError("oracle: backward needs targets")
    mk = _mask(mask, M)
    if lse is None:
        tmp_lse, gap, zmax = np.empty(M), np.empty(M), np.empty(M)
        am = np.empty(M, dtype=np.int64)
        _load().oracle_row_stats(M, V, float(head.softcap), _ptr(raw, _f64p), None,
                                 _ptr(mk, _u8p), None, _ptr(tmp_lse, _f64p), _ptr(am, _i64p),
                                 _ptr(gap, _f64p), _ptr(zmax, _f64p), threads)
        lse = tmp_lse
    lse = np.ascontiguousarray(lse, dtype=np.float64)
    g = np.ascontiguousarray(np.broadcast_to(np.asarray(dlogp, dtype=np.float64), (M,)))
    _load().oracle_coeff(M, V, float(head.softcap), _ptr(raw, _f64p), _ptr(lse, _f64p),
                         _ptr(t, _i32p), _ptr(mk, _u8p), _ptr(g, _f64p), threads)
    return raw


def backward(h: np.ndarray, head: Head, targets, dlogp, mask=None, lse=None,
             threads: int = 0) -> np.ndarray:
    """dh = d(sum_m dlogp[m] * logp[m]) / dh  (fp64 [M,H]).  When ``lse`` is None
    it is recomputed by the forward definition (the same value the forward
    returns)."""
    raw = _coeff(h, head, targets, dlogp, mask, lse, threads)
    M, V = raw.shape
    wq = np.ascontiguousarray(head.wq, dtype=np.uint32)
    s, b = head.sb()
    dh = np.empty((M, head.H), dtype=np.float64)
    _load().oracle_dh(M, head.H, V, head.bits, head.group, _ptr(wq, _u32p), _ptr(s, _f64p),
                      _ptr(b, _f64p), _ptr(raw, _f64p), _ptr(dh, _f64p), threads)
    return dh


def grad_head(h: np.ndarray, head: Head, targets, dlogp, mask=None, lse=None,
              threads: int = 0) -> np.ndarray:
    """dW = d(sum_m dlogp[m] * logp[m]) / dW  (fp64 [V,H]) with respect to the
    dequantized head w[v,d] = s q + b: sum_m coeff[m,v] h[m,d], the classifier
    gradient of the Apple CCE reference (the pages' head is frozen and
    computes none).  Masked rows contribute nothing."""
    raw = _coeff(h, head, targets, dlogp, mask, lse, threads)
    M, V = raw.shape
    hf = _as_f64_h(h)
    dw = np.empty((V, head.H), dtype=np.float64)
    _load().oracle_dw(M, head.H, V, _ptr(raw, _f64p), _ptr(hf, _f64p), _ptr(dw, _f64p), threads)
    return dw


# ------------------------------------------------- blockMax early exit (approximate)

def block_max(h: np.ndarray, head: Head, mask=None, tile: int = 256, threads: int = 0) -> np.ndarray:
    """bm[m, k] = max of the capped logits z[m, v] over vocab tile k (rows
    k*tile .. k*tile + tile - 1), -inf on masked rows: the per-block maxima the
    vocab-parallel forward hands to its backward (page "mlx-bun 0.0.4 ->
    0.0.6", src/train/flash-cce.ts, blockMax), over fixed vocab tiles."""
    raw = logits(h, head, threads)
    M, V = raw.shape
    z = head.softcap * np.tanh(raw / head.softcap) if head.softcap > 0 else raw
    nt = (V + tile - 1) // tile
    zp = np.full((M, nt * tile), -np.inf)
    zp[:, :V] = z
    bm = zp.reshape(M, nt, tile).max(axis=2)
    mk = _mask(mask, M)
    if mk is not None:
        bm[mk == 0] = -np.inf
    return bm


def backward_blockskip(h: np.ndarray, head: Head, targets, dlogp, bm, eps: float,
                       mask=None, lse=None, lse_decide=None, tile_rows: int = 128,
                       tile: int = 256, threads: int = 0) -> np.ndarray:
    """The approximate dh of the blockMax early exit (same page, the
    backward's block skip): the active rows, in ascending order, form tiles
    of tile_rows; a (row tile, vocab tile) block is dropped -- its
    coefficients left out of dh = coeff . W -- when every row of the tile has
    exp(bm[m, k] - lse_decide[m]) < eps and no row's target lies in vocab
    tile k.  The coefficients use ``lse`` (None: recomputed, the forward
    definition); the decision uses the given bm and ``lse_decide`` (default:
    that lse) -- those the caller's forward returned, so that both sides
    drop the same blocks."""
    coeff = _coeff(h, head, targets, dlogp, mask, lse, threads)
    M, V = coeff.shape
    t = np.asarray(targets, dtype=np.int64)
    act = np.arange(M) if mask is None else np.nonzero(np.asarray(mask))[0]
    if lse_decide is None:
        if lse is None:
            lse_decide = forward(h, head, mask=mask, threads=threads).lse
        else:
            lse_decide = lse
    lse = np.asarray(lse_decide, dtype=np.float64)
    bm = np.asarray(bm, dtype=np.float64)
    for j0 in range(0, len(act), tile_rows):
        rows = act[j0:j0 + tile_rows]
        below = np.exp(bm[rows] - lse[rows, None]) < eps        # [rows, tiles]
        drop = below.all(axis=0)
        drop[t[rows] // tile] = False
        for k in np.nonzero(drop)[0]:
            coeff[rows, k * tile:(k + 1) * tile] = 0.0
    wq = np.ascontiguousarray(head.wq, dtype=np.uint32)
    s, b = head.sb()
    dh = np.empty((M, head.H), dtype=np.float64)
    _load().oracle_dh(M, head.H, V, head.bits, head.group, _ptr(wq, _u32p), _ptr(s, _f64p),
                      _ptr(b, _f64p), _ptr(coeff, _f64p), _ptr(dh, _f64p), threads)
    return dh


# ------------------------------------------- coefficient filter (approximate)

class FilterDecision:
    """Blocks of the coefficient filter: ``cold[j, k]`` for the block of active
    rows 32j .. 32j + 31 (ascending order) and vocab rows 32k .. 32k + 31;
    ``cmax[j, k]`` the block's largest softmax term |dlogp| p sech2 (over
    columns that hold no row's target); ``has_target[j, k]`` whether a row's
    target lies in the block's vocab range."""

    def __init__(self, cold, cmax, has_target):
        self.cold, self.cmax, self.has_target = cold, cmax, has_target


def filter_blocks(coeff: np.ndarray, targets, eps: float, mask=None, rows_per_block: int = 32,
                  cols_per_block: int = 32) -> FilterDecision:
    """The coefficient filter's decisions (page "mlx-bun 0.0.4 -> 0.0.6",
    src/train/flash-cce.ts, the backward's near-zero coefficient filter:
    phase 2 skips a coefficient tile whose largest |coeff| is below eps).
    Here a block is cold when no row's target lies in its vocab range and
    every coefficient in it, |dlogp (0 - p) sech2|, is below eps; a block
    that holds a target is always warm, because its one-hot term is carried
    whole (reading of the pages: they test the combined coefficient)."""
    M, V = coeff.shape
    t = np.asarray(targets, dtype=np.int64)
    act = np.arange(M) if mask is None else np.nonzero(np.asarray(mask))[0]
    nrb = (len(act) + rows_per_block - 1) // rows_per_block
    nvb = (V + cols_per_block - 1) // cols_per_block
    cmax = np.zeros((nrb, nvb))
    has_t = np.zeros((nrb, nvb), dtype=bool)
    for j in range(nrb):
        rows = act[j * rows_per_block:(j + 1) * rows_per_block]
        a = np.abs(coeff[rows])
        for r, m in enumerate(rows):
            if 0 <= t[m] < V:
                a[r, t[m]] = 0.0  # the target column holds the one-hot term
                has_t[j, t[m] // cols_per_block] = True
        pad = np.zeros((len(rows), nvb * cols_per_block))
        pad[:, :V] = a
        cmax[j] = pad.reshape(len(rows), nvb, cols_per_block).max(axis=(0, 2))
    cold = (cmax < eps) & ~has_t
    return FilterDecision(cold, cmax, has_t)


def backward_filter(h: np.ndarray, head: Head, targets, dlogp, eps: float, mask=None, lse=None,
                    cold=None, threads: int = 0):
    """The approximate dh of the coefficient filter: dh = coeff . W with the
    coefficients of every cold block (``filter_blocks``) set to 0.  ``cold``
    (bool [row blocks, vocab blocks]) overrides the decisions, so that a
    caller can apply the ones another implementation took.  Returns
    (dh, FilterDecision)."""
    coeff = _coeff(h, head, targets, dlogp, mask, lse, threads)
    M, V = coeff.shape
    dec = filter_blocks(coeff, targets, eps, mask)
    drop = dec.cold if cold is None else np.asarray(cold, dtype=bool)
    act = np.arange(M) if mask is None else np.nonzero(np.asarray(mask))[0]
    for j, k in zip(*np.nonzero(drop)):
        rows = act[32 * j:32 * (j + 1)]
        coeff[rows, 32 * k:32 * (k + 1)] = 0.0
    wq = np.ascontiguousarray(head.wq, dtype=np.uint32)
    s, b = head.sb()
    dh = np.empty((M, head.H), dtype=np.float64)
    _load().oracle_dh(M, head.H, V, head.bits, head.group, _ptr(wq, _u32p), _ptr(s, _f64p),
                      _ptr(b, _f64p), _ptr(coeff, _f64p), _ptr(dh, _f64p), threads)
    return dh, dec


# ------------------------------------------------------------ verify accept

def accept_prefix(argmax: np.ndarray, draft: np.ndarray, W: int):
    """Per window b of W = gamma + 1 rows: the number of leading draft tokens
    equal to the argmax at their positions (stop at the first mismatch, at
    most gamma), and argmax at that position -- the accept loop of the
    speculative decoder (page "mlx-bun 0.0.8 -> 0.0.10", src/spec/generate.ts),
    written as the plain loop."""
    argmax = np.asarray(argmax).reshape(-1, W)
    gamma = W - 1
    draft = np.asarray(draft).reshape(argmax.shape[0], gamma)
    n_accept = np.empty(argmax.shape[0], np.int64)
    nxt = np.empty(argmax.shape[0], np.int64)
    for b in range(argmax.shape[0]):
        k = 0
        while k < gamma and draft[b, k] == argmax[b, k]:
            k += 1
        n_accept[b] = k
        nxt[b] = argmax[b, k]
    return n_accept, nxt
