"""Thin ctypes binding of libqhead.so (include/qhead.h).

Argument marshalling only: every step of the head runs in the library's CUDA
kernels.  PyTorch provides device memory and the current stream.  If the
library has not been built, the first call raises -- there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libqhead.so")

QHEAD_OK, QHEAD_EINVAL, QHEAD_EUNSUPPORTED, QHEAD_ECUDA = 0, 1, 2, 3
QHEAD_SB_F16, QHEAD_SB_BF16, QHEAD_SB_F32 = 0, 1, 2
_SB_CODE = {torch.float16: QHEAD_SB_F16, torch.bfloat16: QHEAD_SB_BF16,
            torch.float32: QHEAD_SB_F32}

# Every symbol include/qhead.h declares.
EXPORTS = ("qhead_fwd_workspace", "qhead_bwd_workspace", "qhead_fwd", "qhead_bwd",
           "qhead_last_error", "qhead_version", "qhead_time_next_head_kernel",
           "qhead_fwd_noalloc", "qhead_test_stall_next_call", "qhead_verify",
           "qhead_bwd_dw_workspace", "qhead_bwd_dw", "qhead_fwd_blockmax_workspace",
           "qhead_fwd_blockmax", "qhead_bwd_blockskip_workspace", "qhead_bwd_blockskip",
           "qhead_bwd_filter_workspace", "qhead_bwd_filter")


class CHead(ctypes.Structure):
    _fields_ = [("wq", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("biases", ctypes.c_void_p), ("V", ctypes.c_int64), ("H", ctypes.c_int32),
                ("bits", ctypes.c_int32), ("group", ctypes.c_int32),
                ("sb_dtype", ctypes.c_int32), ("softcap", ctypes.c_float)]


class QheadError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"qhead error {code}: {msg}")
        self.code = code


_lib = None


def lib() -> ctypes.CDLL:
    """Load libqhead.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with "
                          "`python -m verify_vocab_blocked_gb300.build` (no CPU fallback exists)")
    L = ctypes.CDLL(LIB_PATH)
    vp, i64, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t
    hp = ctypes.POINTER(CHead)
    L.qhead_fwd_workspace.argtypes = [hp, i64]
    L.qhead_fwd_workspace.restype = sz
    L.qhead_bwd_workspace.argtypes = [hp, i64]
    L.qhead_bwd_workspace.restype = sz
    L.qhead_bwd_dw_workspace.argtypes = [hp, i64]
    L.qhead_bwd_dw_workspace.restype = sz
    L.qhead_fwd.argtypes = [hp, vp, i64, vp, vp, vp, vp, vp, vp, sz, vp]
    L.qhead_fwd.restype = ctypes.c_int
    L.qhead_bwd.argtypes = [hp, vp, i64, vp, vp, vp, vp, vp, vp, sz, vp]
    L.qhead_bwd.restype = ctypes.c_int
    L.qhead_bwd_dw.argtypes = [hp, vp, i64, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    L.qhead_bwd_dw.restype = ctypes.c_int
    for name in ("qhead_fwd_blockmax_workspace", "qhead_bwd_blockskip_workspace",
                 "qhead_bwd_filter_workspace"):
        getattr(L, name).argtypes = [hp, i64]
        getattr(L, name).restype = sz
    L.qhead_fwd_blockmax.argtypes = [hp, vp, i64, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    L.qhead_fwd_blockmax.restype = ctypes.c_int
    L.qhead_bwd_blockskip.argtypes = [hp, vp, i64, vp, vp, vp, vp, vp, ctypes.c_float, vp, vp,
                                      sz, vp]
    L.qhead_bwd_blockskip.restype = ctypes.c_int
    L.qhead_bwd_filter.argtypes = [hp, vp, i64, vp, vp, vp, vp, ctypes.c_float, vp, vp, vp, sz,
                                   vp]
    L.qhead_bwd_filter.restype = ctypes.c_int
    L.qhead_verify.argtypes = [hp, vp, i64, i64, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    L.qhead_verify.restype = ctypes.c_int
    L.qhead_last_error.argtypes = []
    L.qhead_last_error.restype = ctypes.c_char_p
    L.qhead_version.argtypes = []
    L.qhead_version.restype = ctypes.c_char_p
    L.qhead_time_next_head_kernel.argtypes = [vp, vp]
    L.qhead_time_next_head_kernel.restype = None
    L.qhead_test_stall_next_call.argtypes = [ctypes.c_int]
    L.qhead_test_stall_next_call.restype = None
    L.qhead_fwd_noalloc.argtypes = [hp, vp, i64, vp, vp, vp, vp, vp, vp]
    L.qhead_fwd_noalloc.restype = ctypes.c_int
    _lib = L
    return L


def test_stall_next_call(armed: bool = True) -> None:
    """Arm the library's one-shot stall switch on this thread: the next fwd/bwd
    call's pipelined head kernel gets no loads, its bounded waits expire and
    the call's active rows come back NaN (argmax -1)."""
    lib().qhead_test_stall_next_call(1 if armed else 0)


def time_next_head_kernel(start: torch.cuda.Event, stop: torch.cuda.Event) -> None:
    """Arm the library's one-shot hook: the next fwd/bwd call on this thread
    records `start` / `stop` around its head kernel on the call's stream.
    Both events must already exist (record them once beforehand)."""
    lib().qhead_time_next_head_kernel(start.cuda_event, stop.cuda_event)


def last_error() -> str:
    return lib().qhead_last_error().decode()


def _check(rc: int):
    if rc != QHEAD_OK:
        raise QheadError(rc, last_error())


@dataclass
class Head:
    """A quantized head resident on the GPU (FlashCceHead layout)."""
    wq: torch.Tensor        # int32 (uint32 bit patterns) [V, H*bits/32]
    scales: torch.Tensor    # float16, bfloat16 or float32 [V, H/group]
    biases: torch.Tensor    # the same type as scales, [V, H/group]
    bits: int
    group: int = 64
    softcap: float = 0.0

    @property
    def V(self) -> int:
        return int(self.wq.shape[0])

    @property
    def H(self) -> int:
        return int(self.wq.shape[1]) * 32 // self.bits

    def c(self) -> CHead:
        for t in (self.wq, self.scales, self.biases):
            if not t.is_contiguous():
                raise ValueError("head tensors must be contiguous")
        if self.scales.dtype not in _SB_CODE or self.biases.dtype != self.scales.dtype:
            raise ValueError("scales and biases must share one type: float16, bfloat16 or "
                             "float32")
        return CHead(self.wq.data_ptr(), self.scales.data_ptr(), self.biases.data_ptr(),
                     self.V, self.H, self.bits, self.group, _SB_CODE[self.scales.dtype],
                     float(self.softcap))

    @staticmethod
    def from_numpy(wq, scales, biases, bits, group=64, softcap=0.0, device="cuda",
                   sb_dtype: str = "f16"):
        """Scales and biases: float16 or float32 arrays, or uint16 bf16 bit
        patterns with sb_dtype="bf16"."""
        import numpy as np

        def sb(x):
            x = np.ascontiguousarray(x)
            if sb_dtype == "bf16":
                return torch.from_numpy(x.astype(np.uint16).view(np.int16)).view(
                    torch.bfloat16).to(device)
            want = {"f16": np.float16, "f32": np.float32}[sb_dtype]
            if x.dtype != want:
                raise ValueError(f"scales/biases are {x.dtype}, sb_dtype is {sb_dtype}")
            return torch.from_numpy(x).to(device)

        return Head(torch.from_numpy(np.ascontiguousarray(wq).view(np.int32)).to(device),
                    sb(scales), sb(biases), bits, group, softcap)


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _check_h(head: Head, h: torch.Tensor, what: str = "[M, H]") -> int:
    """h must be a contiguous bf16 matrix with head.H columns, on the head's
    device; returns M."""
    if not isinstance(h, torch.Tensor) or h.dtype != torch.bfloat16 or h.dim() != 2 \
            or not h.is_contiguous():
        raise ValueError(f"h must be a contiguous bf16 {what} tensor")
    if h.shape[1] != head.H:
        raise ValueError(f"h has {h.shape[1]} columns but the head's hidden size H is {head.H}")
    if head.wq.device != h.device:
        raise ValueError(f"h is on {h.device} but the head is on {head.wq.device}")
    return int(h.shape[0])


def _check_vec(name: str, t: torch.Tensor | None, n: int, dtypes, dev, required: bool = True):
    """A per-row argument: contiguous, shape [n], one of `dtypes`, on `dev`.
    Returns the tensor to pass (bool masks are passed as their uint8 bytes)."""
    if t is None:
        if required:
            raise ValueError(f"{name} is required")
        return None
    if not isinstance(t, torch.Tensor):
        raise ValueError(f"{name} must be a torch tensor")
    if t.dtype not in dtypes:
        names = " or ".join(str(d).replace("torch.", "") for d in dtypes)
        raise ValueError(f"{name} must be {names}, got {str(t.dtype).replace('torch.', '')}")
    if t.dim() != 1 or t.shape[0] != n:
        raise ValueError(f"{name} must have shape [{n}], got {list(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.device != dev:
        raise ValueError(f"{name} is on {t.device}, h on {dev}")
    return t.view(torch.uint8) if t.dtype == torch.bool else t


def _targets(t, M, dev, required):
    return _check_vec("targets", t, M, (torch.int32,), dev, required)


def _mask(mk, M, dev):
    return _check_vec("mask", mk, M, (torch.uint8, torch.bool), dev, required=False)


def _f32(name, t, M, dev):
    return _check_vec(name, t, M, (torch.float32,), dev)


def fwd_workspace(head: Head, M: int) -> int:
    n = lib().qhead_fwd_workspace(ctypes.byref(head.c()), M)
    if n == ctypes.c_size_t(-1).value:
        raise QheadError(QHEAD_EINVAL, last_error())
    return int(n)


def bwd_workspace(head: Head, M: int) -> int:
    n = lib().qhead_bwd_workspace(ctypes.byref(head.c()), M)
    if n == ctypes.c_size_t(-1).value:
        raise QheadError(QHEAD_EINVAL, last_error())
    return int(n)


def bwd_dw_workspace(head: Head, M: int) -> int:
    n = lib().qhead_bwd_dw_workspace(ctypes.byref(head.c()), M)
    if n == ctypes.c_size_t(-1).value:
        raise QheadError(QHEAD_EINVAL, last_error())
    return int(n)


def alloc_workspace(nbytes: int, device) -> torch.Tensor:
    """A 256-byte aligned device buffer of at least nbytes (torch allocations are)."""
    return torch.empty(max(nbytes, 1), dtype=torch.uint8, device=device)


def fwd(head: Head, h: torch.Tensor, targets: torch.Tensor | None = None,
        mask: torch.Tensor | None = None, *, want_logp: bool = True, want_lse: bool = True,
        want_argmax: bool = True, workspace: torch.Tensor | None = None, stream=None):
    """Returns (logp or None, lse or None, argmax or None) for every row of h."""
    M = _check_h(head, h)
    dev = h.device
    targets = _targets(targets, M, dev, required=False)
    mask = _mask(mask, M, dev)
    want_logp = want_logp and targets is not None
    logp = torch.empty(M, dtype=torch.float32, device=dev) if want_logp else None
    lse = torch.empty(M, dtype=torch.float32, device=dev) if want_lse else None
    am = torch.empty(M, dtype=torch.int32, device=dev) if want_argmax else None
    if workspace is None:
        workspace = alloc_workspace(fwd_workspace(head, M), dev)
    _check(lib().qhead_fwd(ctypes.byref(head.c()), h.data_ptr(), M, _ptr(targets), _ptr(mask),
                           _ptr(logp), _ptr(lse), _ptr(am), workspace.data_ptr(),
                           workspace.numel(), _stream(stream)))
    return logp, lse, am


def bwd(head: Head, h: torch.Tensor, targets: torch.Tensor, lse: torch.Tensor,
        dlogp: torch.Tensor, mask: torch.Tensor | None = None, *,
        workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """dh [M, H] float32 of sum_m dlogp[m] * logp[m]."""
    M = _check_h(head, h)
    dev = h.device
    targets = _targets(targets, M, dev, required=True)
    mask = _mask(mask, M, dev)
    lse, dlogp = _f32("lse", lse, M, dev), _f32("dlogp", dlogp, M, dev)
    dh = torch.empty(M, head.H, dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = alloc_workspace(bwd_workspace(head, M), dev)
    _check(lib().qhead_bwd(ctypes.byref(head.c()), h.data_ptr(), M, _ptr(targets), _ptr(mask),
                           lse.data_ptr(), dlogp.data_ptr(), dh.data_ptr(), workspace.data_ptr(),
                           workspace.numel(), _stream(stream)))
    return dh


def bwd_dw(head: Head, h: torch.Tensor, targets: torch.Tensor, lse: torch.Tensor,
           dlogp: torch.Tensor, mask: torch.Tensor | None = None, *, want_dh: bool = False,
           workspace: torch.Tensor | None = None, stream=None):
    """(dh [M, H] float32 or None, dw [V, H] float32): the gradients of
    sum_m dlogp[m] * logp[m] with respect to h and to the dequantized head."""
    M = _check_h(head, h)
    dev = h.device
    targets = _targets(targets, M, dev, required=True)
    mask = _mask(mask, M, dev)
    lse, dlogp = _f32("lse", lse, M, dev), _f32("dlogp", dlogp, M, dev)
    dh = torch.empty(M, head.H, dtype=torch.float32, device=dev) if want_dh else None
    dw = torch.empty(head.V, head.H, dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = alloc_workspace(bwd_dw_workspace(head, M), dev)
    _check(lib().qhead_bwd_dw(ctypes.byref(head.c()), h.data_ptr(), M, targets.data_ptr(),
                              _ptr(mask), lse.data_ptr(), dlogp.data_ptr(), _ptr(dh),
                              dw.data_ptr(), workspace.data_ptr(), workspace.numel(),
                              _stream(stream)))
    return dh, dw


def _ws_size(fn_name: str, head: Head, M: int) -> int:
    n = getattr(lib(), fn_name)(ctypes.byref(head.c()), M)
    if n == ctypes.c_size_t(-1).value:
        raise QheadError(QHEAD_EINVAL, last_error())
    return int(n)


def fwd_blockmax(head: Head, h: torch.Tensor, targets: torch.Tensor | None = None,
                 mask: torch.Tensor | None = None, *, workspace: torch.Tensor | None = None,
                 stream=None):
    """(logp or None, lse, argmax, block_max [M, ceil(V / 256)]): the forward
    plus each row's maximum capped logit per 256-row vocab tile."""
    M = _check_h(head, h)
    dev = h.device
    targets = _targets(targets, M, dev, required=False)
    mask = _mask(mask, M, dev)
    logp = torch.empty(M, dtype=torch.float32, device=dev) if targets is not None else None
    lse = torch.empty(M, dtype=torch.float32, device=dev)
    am = torch.empty(M, dtype=torch.int32, device=dev)
    bm = torch.full((M, (head.V + 255) // 256), float("-inf"), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = alloc_workspace(_ws_size("qhead_fwd_blockmax_workspace", head, M), dev)
    _check(lib().qhead_fwd_blockmax(ctypes.byref(head.c()), h.data_ptr(), M, _ptr(targets),
                                    _ptr(mask), _ptr(logp), lse.data_ptr(), am.data_ptr(),
                                    bm.data_ptr(), workspace.data_ptr(), workspace.numel(),
                                    _stream(stream)))
    return logp, lse, am, bm


def bwd_blockskip(head: Head, h: torch.Tensor, targets: torch.Tensor, lse: torch.Tensor,
                  dlogp: torch.Tensor, block_max: torch.Tensor, eps: float,
                  mask: torch.Tensor | None = None, *, workspace: torch.Tensor | None = None,
                  stream=None) -> torch.Tensor:
    """Approximate dh [M, H] float32: the blocks below eps (see
    qhead_bwd_blockskip) are left out of both backward phases."""
    M = _check_h(head, h)
    dev = h.device
    targets = _targets(targets, M, dev, required=True)
    mask = _mask(mask, M, dev)
    lse, dlogp = _f32("lse", lse, M, dev), _f32("dlogp", dlogp, M, dev)
    nvt = (head.V + 255) // 256
    if (not isinstance(block_max, torch.Tensor) or block_max.dtype != torch.float32
            or tuple(block_max.shape) != (M, nvt) or not block_max.is_contiguous()
            or block_max.device != dev):
        raise ValueError(f"block_max must be a contiguous float32 [{M}, {nvt}] tensor on {dev}")
    dh = torch.empty(M, head.H, dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = alloc_workspace(_ws_size("qhead_bwd_blockskip_workspace", head, M), dev)
    _check(lib().qhead_bwd_blockskip(ctypes.byref(head.c()), h.data_ptr(), M, targets.data_ptr(),
                                     _ptr(mask), lse.data_ptr(), dlogp.data_ptr(),
                                     block_max.data_ptr(), float(eps), dh.data_ptr(),
                                     workspace.data_ptr(), workspace.numel(), _stream(stream)))
    return dh


def bwd_filter(head: Head, h: torch.Tensor, targets: torch.Tensor, lse: torch.Tensor,
               dlogp: torch.Tensor, eps: float, mask: torch.Tensor | None = None, *,
               want_cold: bool = False, workspace: torch.Tensor | None = None, stream=None):
    """(dh [M, H] float32, cold or None): the approximate dh of the
    coefficient filter (see qhead_bwd_filter) and, when asked for, its block
    decisions uint8 [ceil(M / 32), ceil(V / 32)] (1 = cold)."""
    M = _check_h(head, h)
    dev = h.device
    targets = _targets(targets, M, dev, required=True)
    mask = _mask(mask, M, dev)
    lse, dlogp = _f32("lse", lse, M, dev), _f32("dlogp", dlogp, M, dev)
    dh = torch.empty(M, head.H, dtype=torch.float32, device=dev)
    cold = (torch.empty(((M + 31) // 32, (head.V + 31) // 32), dtype=torch.uint8, device=dev)
            if want_cold else None)
    if workspace is None:
        workspace = alloc_workspace(_ws_size("qhead_bwd_filter_workspace", head, M), dev)
    _check(lib().qhead_bwd_filter(ctypes.byref(head.c()), h.data_ptr(), M, targets.data_ptr(),
                                  _ptr(mask), lse.data_ptr(), dlogp.data_ptr(), float(eps),
                                  dh.data_ptr(), _ptr(cold), workspace.data_ptr(),
                                  workspace.numel(), _stream(stream)))
    return dh, cold


def verify(head: Head, h: torch.Tensor, W: int, draft: torch.Tensor | None,
           mask: torch.Tensor | None = None, *, want_lse: bool = False,
           workspace: torch.Tensor | None = None, stream=None):
    """Verify B = h.shape[0] / W windows of W = gamma + 1 rows against their
    drafts (int32 [B, W - 1]).  Returns (n_accept [B], next_token [B],
    argmax [B * W], lse [B * W] or None), all on the device."""
    M = _check_h(head, h, "[B * W, H]")
    if W < 1 or M % W:
        raise ValueError("the row count must be a multiple of W >= 1")
    B = M // W
    if draft is not None and (draft.dtype != torch.int32 or not draft.is_contiguous()
                              or draft.numel() != B * (W - 1)):
        raise ValueError("draft must be a contiguous int32 [B, W - 1] tensor")
    dev = h.device
    if draft is not None and draft.device != dev:
        raise ValueError(f"draft is on {draft.device}, h on {dev}")
    mask = _mask(mask, M, dev)
    am = torch.empty(M, dtype=torch.int32, device=dev)
    lse = torch.empty(M, dtype=torch.float32, device=dev) if want_lse else None
    n_acc = torch.empty(B, dtype=torch.int32, device=dev)
    nxt = torch.empty(B, dtype=torch.int32, device=dev)
    if workspace is None:
        workspace = alloc_workspace(fwd_workspace(head, M), dev)
    _check(lib().qhead_verify(ctypes.byref(head.c()), h.data_ptr(), B, W, _ptr(draft),
                              _ptr(mask), _ptr(lse), am.data_ptr(), n_acc.data_ptr(),
                              nxt.data_ptr(), workspace.data_ptr(), workspace.numel(),
                              _stream(stream)))
    return n_acc, nxt, am, lse
