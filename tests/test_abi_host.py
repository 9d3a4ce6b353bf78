"""Host-side checks of the C ABI: the library builds, loads and exports every
symbol include/qhead.h declares, argument errors come back as the
documented status codes before anything touches a GPU, and a plain C program
(tests/c/abi_from_c.c) compiles against the header and links the library."""
import ctypes
import os
import re
import shutil
import subprocess

import pytest

from verify_vocab_blocked_gb300 import build as qbuild
from verify_vocab_blocked_gb300 import qhead

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qhead.h")


@pytest.fixture(scope="module")
def L():
    qbuild.build()
    return qhead.lib()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(qhead_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_what_binding_lists():
    assert set(_declared_functions()) == set(qhead.EXPORTS)


def test_every_declared_symbol_is_exported(L):
    for name in _declared_functions():
        assert hasattr(L, name), name


def test_version(L):
    assert L.qhead_version().decode().startswith("qhead ")


def _head(**kw):
    # Plausible-looking, never-dereferenced device addresses: every case below
    # fails argument checks before any CUDA call.
    base = dict(wq=0x10000, scales=0x20000, biases=0x30000, V=1000, H=256, bits=4, group=64,
                sb_dtype=qhead.QHEAD_SB_F16, softcap=0.0)
    base.update(kw)
    return qhead.CHead(**base)


FWD_ARGS = dict(h=0x40000, M=4, targets=None, mask=None, logp=None, lse=0x50000, argmax=None,
                ws=0x60000, ws_bytes=1 << 20, stream=None)


def _fwd(L, head, **kw):
    a = dict(FWD_ARGS)
    a.update(kw)
    return L.qhead_fwd(ctypes.byref(head) if head is not None else None, a["h"], a["M"],
                       a["targets"], a["mask"], a["logp"], a["lse"], a["argmax"], a["ws"],
                       a["ws_bytes"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(bits=3), qhead.QHEAD_EUNSUPPORTED),
    (dict(bits=2), qhead.QHEAD_EUNSUPPORTED),
    (dict(group=32), qhead.QHEAD_EUNSUPPORTED),
    (dict(sb_dtype=7), qhead.QHEAD_EUNSUPPORTED),
    (dict(sb_dtype=3), qhead.QHEAD_EUNSUPPORTED),
    (dict(sb_dtype=-1), qhead.QHEAD_EUNSUPPORTED),
    (dict(H=192), qhead.QHEAD_EUNSUPPORTED),
    (dict(H=64), qhead.QHEAD_EUNSUPPORTED),
    (dict(H=8320), qhead.QHEAD_EUNSUPPORTED),
    (dict(V=0), qhead.QHEAD_EINVAL),
    (dict(V=1 << 31), qhead.QHEAD_EINVAL),
    (dict(wq=0x10004), qhead.QHEAD_EINVAL),
    (dict(scales=0x20001), qhead.QHEAD_EINVAL),
    (dict(scales=0x20002), qhead.QHEAD_EINVAL),
    (dict(biases=0x30008), qhead.QHEAD_EINVAL),
    (dict(wq=None), qhead.QHEAD_EINVAL),
    (dict(biases=None), qhead.QHEAD_EINVAL),
    (dict(softcap=float("nan")), qhead.QHEAD_EINVAL),
])
def test_bad_head(L, kw, code):
    assert _fwd(L, _head(**kw)) == code
    assert L.qhead_last_error().decode() != ""
    assert L.qhead_fwd_workspace(ctypes.byref(_head(**kw)), 4) == ctypes.c_size_t(-1).value


@pytest.mark.parametrize("kw", [
    dict(M=-1), dict(h=None), dict(h=0x40008), dict(logp=0x70000),
    dict(lse=None), dict(ws=None), dict(ws=0x60080),
])
def test_bad_fwd_args(L, kw):
    assert _fwd(L, _head(), **kw) == qhead.QHEAD_EINVAL
    assert L.qhead_last_error().decode() != ""


def test_null_head(L):
    assert _fwd(L, None) == qhead.QHEAD_EINVAL


def test_zero_rows_is_a_no_op(L):
    assert _fwd(L, _head(), M=0, ws=None, ws_bytes=0) == qhead.QHEAD_OK
    assert L.qhead_fwd_workspace(ctypes.byref(_head()), 0) == 0
    assert L.qhead_bwd(ctypes.byref(_head()), None, 0, None, None, None, None, None, None, 0,
                       None) == qhead.QHEAD_OK


@pytest.mark.parametrize("drop", ["h", "targets", "lse", "dlogp", "dh"])
def test_bad_bwd_args(L, drop):
    a = dict(h=0x40000, targets=0x41000, lse=0x42000, dlogp=0x43000, dh=0x44000)
    a[drop] = None
    rc = L.qhead_bwd(ctypes.byref(_head()), a["h"], 4, a["targets"], None, a["lse"],
                     a["dlogp"], a["dh"], 0x60000, 1 << 20, None)
    assert rc == qhead.QHEAD_EINVAL


def test_error_message_is_per_call(L):
    assert _fwd(L, _head(bits=3)) != 0
    assert "bits" in L.qhead_last_error().decode()
    assert _fwd(L, _head(), M=0) == 0
    assert L.qhead_last_error().decode() == ""


def _verify(L, **kw):
    a = dict(head=_head(), h=0x40000, B=2, W=5, draft=0x41000, mask=None, lse=None,
             argmax=0x42000, n_accept=0x43000, next_token=None, ws=0x60000, ws_bytes=1 << 20)
    a.update(kw)
    return L.qhead_verify(ctypes.byref(a["head"]), a["h"], a["B"], a["W"], a["draft"], a["mask"],
                          a["lse"], a["argmax"], a["n_accept"], a["next_token"], a["ws"],
                          a["ws_bytes"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(B=-1), qhead.QHEAD_EINVAL),
    (dict(W=0), qhead.QHEAD_EINVAL),
    (dict(W=(1 << 20) + 1), qhead.QHEAD_EINVAL),
    (dict(B=1 << 40), qhead.QHEAD_EINVAL),
    (dict(argmax=None), qhead.QHEAD_EINVAL),
    (dict(n_accept=None), qhead.QHEAD_EINVAL),
    (dict(draft=None), qhead.QHEAD_EINVAL),
    (dict(head=_head(bits=3)), qhead.QHEAD_EUNSUPPORTED),
])
def test_bad_verify_args(L, kw, code):
    assert _verify(L, **kw) == code
    assert L.qhead_last_error().decode() != ""


def test_verify_zero_windows_is_a_no_op(L):
    assert _verify(L, B=0, ws=None, ws_bytes=0) == qhead.QHEAD_OK


def test_bad_bwd_dw_args(L):
    a = dict(h=0x40000, targets=0x41000, lse=0x42000, dlogp=0x43000, dh=None, dw=0x44000)
    fn = L.qhead_bwd_dw
    assert fn(ctypes.byref(_head()), a["h"], 4, a["targets"], None, a["lse"], a["dlogp"], None,
              None, 0x60000, 1 << 20, None) == qhead.QHEAD_EINVAL       # no dw
    assert fn(ctypes.byref(_head()), a["h"], 4, a["targets"], None, a["lse"], a["dlogp"], None,
              0x44010, 0x60000, 1 << 20, None) == qhead.QHEAD_EINVAL    # dw not 32-byte aligned
    assert "32-byte" in L.qhead_last_error().decode()
    assert fn(ctypes.byref(_head()), None, 4, a["targets"], None, a["lse"], a["dlogp"], None,
              a["dw"], 0x60000, 1 << 20, None) == qhead.QHEAD_EINVAL    # no h
    # (workspace sizes need the device's SM count: checked in the GPU tests)


def test_bad_blockmax_and_blockskip_args(L):
    hd = ctypes.byref(_head())
    # the forward with tile maxima needs the block_max output
    assert L.qhead_fwd_blockmax(hd, 0x40000, 4, None, None, None, 0x42000, None, None,
                                0x60000, 1 << 20, None) == qhead.QHEAD_EINVAL
    assert "block_max" in L.qhead_last_error().decode()
    # the skipping backward needs block_max and an eps in [0, 1]
    args = (0x40000, 4, 0x41000, None, 0x42000, 0x43000)
    assert L.qhead_bwd_blockskip(hd, *args, None, ctypes.c_float(1e-5), 0x44000, 0x60000,
                                 1 << 20, None) == qhead.QHEAD_EINVAL
    for bad in (-1.0, 2.0, float("nan")):
        assert L.qhead_bwd_blockskip(hd, *args, 0x45000, ctypes.c_float(bad), 0x44000, 0x60000,
                                     1 << 20, None) == qhead.QHEAD_EINVAL
        assert "eps" in L.qhead_last_error().decode()
    # M = 0 is a no-op for both
    assert L.qhead_fwd_blockmax(hd, None, 0, None, None, None, None, None, None, None, 0,
                                None) == qhead.QHEAD_OK
    assert L.qhead_bwd_blockskip(hd, None, 0, None, None, None, None, None, ctypes.c_float(0.0),
                                 None, None, 0, None) == qhead.QHEAD_OK
    # (their workspace sizes, which need the device's SM count, are checked in
    # the GPU tests)


def test_bad_filter_args(L):
    hd = ctypes.byref(_head())
    args = (0x40000, 4, 0x41000, None, 0x42000, 0x43000)
    # eps must be a number >= 0 (+inf allowed: every block without a target is cold)
    for bad in (-1.0, -1e-30, float("nan")):
        assert L.qhead_bwd_filter(hd, *args, ctypes.c_float(bad), 0x44000, None, 0x60000,
                                  1 << 20, None) == qhead.QHEAD_EINVAL
        assert "eps" in L.qhead_last_error().decode()
    # dh is required; M = 0 is a no-op
    assert L.qhead_bwd_filter(hd, *args, ctypes.c_float(1e-5), None, None, 0x60000, 1 << 20,
                              None) == qhead.QHEAD_EINVAL
    assert L.qhead_bwd_filter(hd, None, 0, None, None, None, None, ctypes.c_float(1e-5), None,
                              None, None, 0, None) == qhead.QHEAD_OK
    # workspace sizes need the device's SM count: checked in the GPU tests


def test_the_abi_is_usable_from_plain_c(L, tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    libdir = os.path.dirname(qhead.LIB_PATH)
    exe = str(tmp_path / "abi_from_c")
    cmd = [cc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-I" + os.path.join(ROOT, "include"),
           os.path.join(ROOT, "tests", "c", "abi_from_c.c"), "-L" + libdir, "-lqhead",
           "-Wl,-rpath," + libdir, "-lm", "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr


@pytest.mark.parametrize("sbt", [qhead.QHEAD_SB_BF16, qhead.QHEAD_SB_F32])
def test_bf16_and_f32_scales_pass_the_head_checks(L, sbt):
    # The head is accepted; the call then fails later (no workspace here), not
    # on the element type of its scales and biases.
    rc = _fwd(L, _head(sb_dtype=sbt), ws=None)
    assert rc == qhead.QHEAD_EINVAL and "workspace" in L.qhead_last_error().decode()
