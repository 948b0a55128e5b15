"""Host-side checks of the C ABI that need no GPU.

The library must load and export every entry point include/falcon.h declares,
and argument checks must reject bad calls before touching a device (they
return an error code and launch nothing).
"""
import ctypes
import os
import re
import shutil

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "falcon.h")

pytestmark = pytest.mark.skipif(shutil.which("nvcc") is None and
                                not os.path.exists("/usr/local/cuda/bin/nvcc"),
                                reason="needs nvcc to build the library")


@pytest.fixture(scope="module")
def lib():
    from delta_rule_attention_gb300 import _build
    _build.build()
    import delta_rule_attention_gb300 as falcon
    return falcon.load_library()


def _declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\**\s*([a-z_0-9]+)\s*\(",
                       src, flags=re.M)
    return sorted(set(n for n in names if n.startswith("falcon")))


def test_header_declares_the_entry_points():
    names = _declared_functions()
    import delta_rule_attention_gb300 as falcon
    assert set(names) == set(falcon.EXPORTS), names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_version_and_strerror(lib):
    assert lib.falcon_version() == 10200
    assert lib.falcon_strerror(0) == b"ok"
    for code in range(-10, 0):
        assert lib.falcon_strerror(code) != b"unknown error code"
    assert lib.falcon_strerror(-99) == b"unknown error code"


def _shape(**kw):
    import delta_rule_attention_gb300 as falcon
    base = dict(B=1, H=2, T=64, m=16, dv=16, chunk=16, dtype=falcon.FALCON_F32,
                phi=falcon.FALCON_PHI_L2, eps=1e-6, eps_gamma=1e-6)
    base.update(kw)
    s = falcon.falcon_shape()
    for key, val in base.items():
        setattr(s, key, val)
    return s


def test_workspace_bytes(lib):
    s = _shape()
    # one map [(m + C) x (m + dv)] fp32 per (head, chunk)
    assert lib.falcon_workspace_bytes(ctypes.byref(s)) == 2 * 4 * (16 + 16) * 32 * 4
    s = _shape(T=65)  # ragged: 5 chunks
    assert lib.falcon_workspace_bytes(ctypes.byref(s)) == 2 * 5 * (16 + 16) * 32 * 4
    assert lib.falcon_workspace_bytes(ctypes.byref(_shape(m=24))) == 0
    assert lib.falcon_workspace_bytes(None) == 0


def _fake(addr=0x10000):
    return ctypes.c_void_p(addr)


@pytest.mark.parametrize("fn", ["falcon1_fwd_chunked", "falcon1a_fwd_chunked"])
@pytest.mark.parametrize("bad,code", [
    (dict(m=24), -2), (dict(dv=256), -2), (dict(chunk=48), -2), (dict(T=-1), -2),
    (dict(dtype=7), -3), (dict(phi=3), -3), (dict(eps=-1.0), -8), (dict(eps_gamma=1.0), -8),
    (dict(eps_gamma=0.0), -8), (dict(ridge=2), -8), (dict(ridge=-1), -8),
])
def test_forward_rejects_bad_shapes_without_a_device(lib, fn, bad, code):
    s = _shape(**bad)
    p = _fake()
    rc = getattr(lib, fn)(ctypes.byref(s), p, p, p, p, p, None, None, p, p, None, p,
                          ctypes.c_size_t(1 << 40), None)
    assert rc == code


@pytest.mark.parametrize("fn", ["falcon1_fwd_chunked", "falcon1a_fwd_chunked"])
def test_forward_rejects_null_misaligned_and_small_workspace(lib, fn):
    s = _shape()
    p, odd = _fake(), _fake(0x10008)
    f = getattr(lib, fn)
    big = ctypes.c_size_t(1 << 40)
    assert f(None, p, p, p, p, p, None, None, p, p, None, p, big, None) == -1
    assert f(ctypes.byref(s), None, p, p, p, p, None, None, p, p, None, p, big, None) == -1
    assert f(ctypes.byref(s), p, p, p, p, p, None, None, p, None, None, p, big, None) == -1
    assert f(ctypes.byref(s), p, odd, p, p, p, None, None, p, p, None, p, big, None) == -4
    assert f(ctypes.byref(s), p, p, p, p, p, odd, None, p, p, None, p, big, None) == -4
    assert f(ctypes.byref(s), p, p, p, p, p, None, None, p, p, None, None, big, None) == -5
    assert f(ctypes.byref(s), p, p, p, p, p, None, None, p, p, None, p,
             ctypes.c_size_t(16), None) == -5
    # B*H == 0 is a valid no-op that touches nothing
    assert f(ctypes.byref(_shape(B=0)), None, None, None, None, None, None, None, None, None,
             None, None, ctypes.c_size_t(0), None) == 0


@pytest.mark.parametrize("fn", ["falcon1_decode_step", "falcon1a_decode_step"])
def test_decode_rejects_bad_arguments_without_a_device(lib, fn):
    f = getattr(lib, fn)
    p, odd = _fake(), _fake(0x10004)
    args = lambda N=4, m=64, dv=64, dt=0, phi=1, ridge=0, eps=1e-6, eg=1e-6, q=p, S=p: f(
        N, m, dv, dt, phi, ridge, ctypes.c_float(eps), ctypes.c_float(eg), q, p, p, p, p, S, p,
        None, p, None)
    assert args(m=48) == -2
    assert args(N=-1) == -2
    assert args(dt=5) == -3
    assert args(phi=3) == -3
    assert args(ridge=2) == -8
    assert args(eg=2.0) == -8
    assert args(q=None) == -1
    assert args(S=odd) == -4
    assert args(N=0, q=None) == 0


@pytest.mark.parametrize("fn", ["falcon1_bwd_chunked", "falcon1a_bwd_chunked"])
def test_backward_rejects_bad_arguments_without_a_device(lib, fn):
    f = getattr(lib, fn)
    p, odd = _fake(), _fake(0x10008)
    big = ctypes.c_size_t(1 << 40)

    def call(s, q=p, dO=p, dq=p, dS0=None, ws=p, wsb=big):
        return f(ctypes.byref(s) if s is not None else None, q, p, p, p, p, None, None, dO, None,
                 None, dq, p, p, p, p, dS0, None, ws, wsb, None)

    for bad, code in ((dict(m=24), -2), (dict(chunk=48), -2), (dict(dtype=7), -3),
                      (dict(phi=3), -3), (dict(ridge=2), -8), (dict(eps_gamma=1.0), -8)):
        assert call(_shape(**bad)) == code, bad
    s = _shape()
    assert call(None) == -1
    assert call(s, q=None) == -1
    assert call(s, dO=None) == -1
    assert call(s, dq=None) == -1
    assert call(s, dq=odd) == -4
    assert call(s, dS0=odd) == -4
    assert call(s, ws=None) == -5
    assert call(s, wsb=ctypes.c_size_t(64)) == -5
    assert call(_shape(B=0), q=None, dO=None, dq=None, ws=None, wsb=ctypes.c_size_t(0)) == 0


def test_backward_workspace_bytes(lib):
    s = _shape()  # B1 H2 T64 m16 dv16 C16: 4 chunks per head
    BH, nch, m, dv, C, T = 2, 4, 16, 16, 16, 64
    floats = [BH * nch * (m + C) * (m + dv), BH * nch * m * dv, BH * nch * m * dv, BH * T * m]
    want = sum((n + 63) // 64 * 64 for n in floats) * 4
    assert lib.falcon_bwd_workspace_bytes(ctypes.byref(s)) == want
    assert lib.falcon_bwd_workspace_bytes(ctypes.byref(_shape(m=24))) == 0
