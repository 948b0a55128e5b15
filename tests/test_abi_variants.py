"""Host-side argument checks of the Falcon-2, Falcon-2A and Falcon-3A entry
points, of the fixed-scratch Falcon-1 forward and of Falcon-1A with the
normalised read (no GPU needed).

Every call here is invalid in exactly one argument, so each must come back
with that argument's error code before any device is touched; a valid call
would launch kernels on the fake addresses used here, so none is made.  The
fixed-scratch entry point must give the codes of falcon1_fwd_chunked (its
scratch array is looked up only after every argument check), which is what
these tests see on a machine without a GPU.
"""
import ctypes
import os
import shutil

import pytest

pytestmark = pytest.mark.skipif(shutil.which("nvcc") is None and
                                not os.path.exists("/usr/local/cuda/bin/nvcc"),
                                reason="needs nvcc to build the library")

NULL_PTR, BAD_SHAPE, BAD_DTYPE, MISALIGNED, WORKSPACE, BAD_ARG = -1, -2, -3, -4, -5, -8

# One argument out of range at a time, with the code it must produce (the
# shape checks shared by every forward entry point).
BAD_SHAPES = [
    (dict(m=24), BAD_SHAPE), (dict(dv=256), BAD_SHAPE), (dict(chunk=48), BAD_SHAPE),
    (dict(T=-1), BAD_SHAPE), (dict(B=-1), BAD_SHAPE), (dict(B=70000, H=1), BAD_SHAPE),
    (dict(dtype=7), BAD_DTYPE), (dict(phi=3), BAD_DTYPE), (dict(eps=-1.0), BAD_ARG),
    (dict(eps=float("nan")), BAD_ARG), (dict(eps_gamma=1.0), BAD_ARG),
    (dict(eps_gamma=0.0), BAD_ARG), (dict(ridge=2), BAD_ARG),
]


@pytest.fixture(scope="module")
def lib():
    from delta_rule_attention_gb300 import _build
    _build.build()
    import delta_rule_attention_gb300 as falcon
    return falcon.load_library()


def _shape(**kw):
    import delta_rule_attention_gb300 as falcon
    base = dict(B=1, H=2, T=64, m=16, dv=16, chunk=16, dtype=falcon.FALCON_F32,
                phi=falcon.FALCON_PHI_L2, eps=1e-6, eps_gamma=1e-6)
    base.update(kw)
    s = falcon.falcon_shape()
    for key, val in base.items():
        setattr(s, key, val)
    return s


def _tc_shape(**kw):
    """A shape the tensor-core Falcon-2A / Falcon-3A paths take (they need a
    workspace)."""
    import delta_rule_attention_gb300 as falcon
    return _shape(B=1, H=2, T=256, m=64, dv=64, chunk=64, dtype=falcon.FALCON_BF16, **kw)


P, ODD = ctypes.c_void_p(0x10000), ctypes.c_void_p(0x10008)
BIG = ctypes.c_size_t(1 << 40)


def _call(lib, name, s, q=P, S0=None, x_prev=None, S_out=P, ws=P, wsb=BIG, window=4,
          z0=None, z_out=None, eps_attn=1e-6):
    """Call `name` with the argument order of its declaration; pointers not
    given are valid-looking fake addresses."""
    f = getattr(lib, name)
    sp = ctypes.byref(s) if s is not None else None
    if name == "falcon1a_fwd_chunked_normalized":
        return f(sp, q, P, P, P, P, S0, z0, x_prev, ctypes.c_float(eps_attn), P, S_out, z_out,
                 None, ws, wsb, None)
    if name in ("falcon2_fwd_recurrent", "falcon2a_fwd_recurrent", "falcon2_fwd_chunked"):
        return f(sp, q, P, P, P, P, S0, x_prev, P, S_out, None, None)
    if name == "falcon2a_fwd_chunked":
        return f(sp, q, P, P, P, P, S0, x_prev, P, S_out, None, ws, wsb, None)
    if name == "falcon3a_fwd_recurrent":
        return f(sp, window, q, P, P, P, P, S0, P, S_out, None, None)
    if name == "falcon3a_fwd_chunked":
        return f(sp, window, q, P, P, P, P, S0, P, S_out, None, ws, wsb, None)
    if name == "falcon1_fwd_chunked_fixed_scratch":
        return f(sp, q, P, P, P, P, S0, x_prev, P, S_out, None, None)
    raise ValueError(name)


VARIANTS = ["falcon2_fwd_recurrent", "falcon2a_fwd_recurrent", "falcon2a_fwd_chunked",
            "falcon2_fwd_chunked",
            "falcon3a_fwd_recurrent", "falcon3a_fwd_chunked", "falcon1_fwd_chunked_fixed_scratch",
            "falcon1a_fwd_chunked_normalized"]


@pytest.mark.parametrize("name", VARIANTS)
@pytest.mark.parametrize("bad,code", BAD_SHAPES)
def test_variants_reject_bad_shapes(lib, name, bad, code):
    assert _call(lib, name, _shape(**bad)) == code


@pytest.mark.parametrize("name", VARIANTS)
def test_variants_reject_null_and_misaligned_pointers(lib, name):
    s = _shape()
    assert _call(lib, name, None) == NULL_PTR
    assert _call(lib, name, s, q=None) == NULL_PTR
    assert _call(lib, name, s, S_out=None) == NULL_PTR
    assert _call(lib, name, s, q=ODD) == MISALIGNED
    assert _call(lib, name, s, S0=ODD) == MISALIGNED


@pytest.mark.parametrize("name", VARIANTS)
def test_variants_with_no_heads_touch_nothing(lib, name):
    # B*H == 0 is a valid no-op: every pointer may be NULL and no device is
    # needed (so the call succeeds on a machine without a GPU).
    assert _call(lib, name, _shape(B=0), q=None, S_out=None, ws=None,
                 wsb=ctypes.c_size_t(0)) == 0


@pytest.mark.parametrize("name", ["falcon2_fwd_recurrent", "falcon2a_fwd_recurrent",
                                  "falcon2a_fwd_chunked", "falcon2_fwd_chunked",
                                  "falcon1_fwd_chunked_fixed_scratch",
                                  "falcon1a_fwd_chunked_normalized"])
def test_misaligned_x_prev_is_rejected(lib, name):
    assert _call(lib, name, _shape(), x_prev=ODD) == MISALIGNED


@pytest.mark.parametrize("name", ["falcon3a_fwd_recurrent", "falcon3a_fwd_chunked"])
@pytest.mark.parametrize("window", [0, -1, 33, 1 << 20])
def test_falcon3a_rejects_windows_outside_1_to_32(lib, name, window):
    assert _call(lib, name, _shape(), window=window) == BAD_ARG
    assert _call(lib, name, _tc_shape(), window=window) == BAD_ARG


@pytest.mark.parametrize("name", ["falcon2a_fwd_chunked", "falcon3a_fwd_chunked"])
def test_tensor_core_chunk_forms_need_an_aligned_workspace(lib, name):
    s = _tc_shape()
    need = lib.falcon_workspace_bytes(ctypes.byref(s))
    assert need > 0
    assert _call(lib, name, s, ws=None) == WORKSPACE
    assert _call(lib, name, s, wsb=ctypes.c_size_t(need - 1)) == WORKSPACE
    # 16-byte aligned is not enough: the workspace must sit on 256 bytes
    assert _call(lib, name, s, ws=ctypes.c_void_p(0x10010)) == MISALIGNED


def test_falcon2_chunk_form_needs_no_workspace(lib):
    """The tensor-core Falcon-2 chunk form runs one CTA per head from its
    inputs alone: with no workspace the arguments pass and the call stops only
    at the device check (no GPU here)."""
    import delta_rule_attention_gb300 as falcon
    rc = _call(lib, "falcon2_fwd_chunked", _tc_shape(), ws=None, wsb=ctypes.c_size_t(0))
    assert rc in (-9, -6), rc  # FALCON_ERR_DEVICE, FALCON_ERR_CUDA


def test_codes_are_the_headers():
    import re
    header = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                          "include", "falcon.h")
    defs = dict((k, int(v)) for k, v in
                re.findall(r"#define FALCON_ERR_([A-Z_]+) \((-?[0-9]+)\)", open(header).read()))
    assert (defs["NULL_PTR"], defs["BAD_SHAPE"], defs["BAD_DTYPE"], defs["MISALIGNED"],
            defs["WORKSPACE"], defs["BAD_ARG"]) == (NULL_PTR, BAD_SHAPE, BAD_DTYPE, MISALIGNED,
                                                    WORKSPACE, BAD_ARG)


def test_fixed_scratch_codes_match_the_workspace_entry_point(lib):
    """Each invalid call gets the same code from the fixed-scratch entry point
    as from falcon1_fwd_chunked with an ample workspace."""
    def regular(s, q=P, S0=None, x_prev=None, S_out=P):
        return lib.falcon1_fwd_chunked(ctypes.byref(s) if s is not None else None, q, P, P, P,
                                       P, S0, x_prev, P, S_out, None, P, BIG, None)

    cases = [dict(s=None), dict(s=_shape(), q=None), dict(s=_shape(), S_out=None),
             dict(s=_shape(), q=ODD), dict(s=_shape(), S0=ODD), dict(s=_shape(), x_prev=ODD)]
    cases += [dict(s=_shape(**bad)) for bad, _ in BAD_SHAPES]
    for c in cases:
        want = regular(**c)
        assert want < 0, c
        assert _call(lib, "falcon1_fwd_chunked_fixed_scratch", **c) == want, c


@pytest.mark.parametrize("eps_attn", [-1e-3, float("nan"), float("inf")])
def test_normalized_read_rejects_bad_eps_attn(lib, eps_attn):
    assert _call(lib, "falcon1a_fwd_chunked_normalized", _shape(), eps_attn=eps_attn) == BAD_ARG


def test_normalized_read_checks_its_state_and_workspace(lib):
    name = "falcon1a_fwd_chunked_normalized"
    assert _call(lib, name, _shape(), z0=ODD) == MISALIGNED
    assert _call(lib, name, _shape(), z_out=ODD) == MISALIGNED
    s = _shape()
    need = lib.falcon_normalized_workspace_bytes(ctypes.byref(s))
    # room for the denominator beyond the forward's own workspace
    assert need > lib.falcon_workspace_bytes(ctypes.byref(s)) > 0
    assert _call(lib, name, s, wsb=ctypes.c_size_t(need - 1)) == WORKSPACE
    assert _call(lib, name, s, ws=None) == WORKSPACE
    assert lib.falcon_normalized_workspace_bytes(ctypes.byref(_shape(m=24))) == 0
