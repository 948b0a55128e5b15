"""fp64 CPU oracle for the Falcon-1 / Falcon-1A, Falcon-2 / Falcon-2A and Falcon-3A recurrences,
and the backward pass of Falcon-1 / Falcon-1A.

TEST INFRASTRUCTURE ONLY.  Nothing in the library path imports this package:
only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline legs of
``bench.py`` do.  The arithmetic lives in ``falcon_oracle.c`` (plain C, fp64,
token by token); this module compiles it with gcc and wraps it with ctypes.
It shares no code with the CUDA library and never calls it.

Every function here is pinned by ``tests/test_oracle_pins.py`` against
closed forms, an autograd gradient step, the masked-parallel forms and
brute-force sums (see the docstrings there for the passage each pin follows).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "falcon_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

FALCON1 = 1  # regression rule (Section 3.1, Eq. (3.3))
FALCON1A = 2  # inner-product rule (Section 4.3, Eq. (4.6))
FALCON2 = 3  # per-column regression rule (Section 3.1, Section 4.2)
FALCON2A = 4  # per-column inner-product rule (Section 4.3)
_RULES = {"falcon1": FALCON1, "falcon1a": FALCON1A, FALCON1: FALCON1, FALCON1A: FALCON1A}
_RULES2 = {"falcon2": FALCON2, "falcon2a": FALCON2A, FALCON2: FALCON2, FALCON2A: FALCON2A}
_PHIS = {"identity": 0, "l2": 1, "rms": 2}
_RIDGES = {"given": 0, "scaled": 1}


def build(force: bool = False) -> str:
    """Compile ``falcon_oracle.c`` into ``liboracle.so`` next to it (gcc, -O2)."""
    stale = (not os.path.exists(_LIB_PATH)) or (
        os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-o", tmp,
                        _SRC, "-lm", "-lpthread"], check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            d = ctypes.POINTER(ctypes.c_double)
            i64 = ctypes.c_int64
            lib.falcon_oracle_forward.restype = ctypes.c_int
            lib.falcon_oracle_forward.argtypes = [
                ctypes.c_int, i64, i64, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_double, ctypes.c_double, d, d, d, d, d, d, d, d, d, d, d,
                ctypes.c_int]
            lib.falcon2_oracle_forward.restype = ctypes.c_int
            lib.falcon2_oracle_forward.argtypes = [
                ctypes.c_int, i64, i64, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_double, ctypes.c_double, d, d, d, d, d, d, d, d, d, d,
                ctypes.c_int]
            lib.falcon3a_oracle_forward.restype = ctypes.c_int
            lib.falcon3a_oracle_forward.argtypes = [
                i64, i64, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_double, ctypes.c_double, d, d, d, d, d, d, d, d, d, ctypes.c_int]
            lib.falcon_oracle_backward.restype = ctypes.c_int
            lib.falcon_oracle_backward.argtypes = [
                ctypes.c_int, i64, i64, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_double, ctypes.c_double] + [d] * 17 + [ctypes.c_int]
            lib.falcon1a_oracle_forward_normalized.restype = ctypes.c_int
            lib.falcon1a_oracle_forward_normalized.argtypes = [
                i64, i64, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_double, ctypes.c_double, ctypes.c_double] + [d] * 12 + [ctypes.c_int]
            lib.falcon_oracle_decode_step.restype = ctypes.c_int
            lib.falcon_oracle_decode_step.argtypes = [
                ctypes.c_int, i64, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_double, ctypes.c_double, d, d, d, d, d, d, d,
                ctypes.POINTER(ctypes.c_ubyte), d]
            _lib = lib
    return _lib


def _f64(a):
    """Widen to a C-contiguous float64 numpy array (exact for bf16/fp32)."""
    if a is None:
        return None
    if hasattr(a, "detach"):  # torch tensor
        a = a.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def forward(rule, q, k, v, beta, lam, S0=None, x_prev=None, phi="l2",
            eps=1e-6, eps_gamma=1e-6, trajectory=False, threads=None, ridge="given"):
    """Run the recurrence over whole sequences.

    Shapes: q, k [..., T, m]; v [..., T, dv]; beta, lam [..., T];
    S0 [..., m, dv] or None (zeros); x_prev [..., m] or None (sentinel).
    The leading dims (B, H, ...) are flattened into independent heads.
    Returns a dict with o [..., T, dv], S [..., m, dv], x_last [..., m] and,
    if ``trajectory``, S_traj [..., T, m, dv] (the state after each token).
    phi: "identity", "l2" or "rms"; ridge: "given" (lam is lambda_t) or
    "scaled" (lam is the base ridge, lambda_t = lam_t * ||x_t||^2).
    """
    lib = _load()
    q, k, v, beta, lam = (_f64(t) for t in (q, k, v, beta, lam))
    S0, x_prev = _f64(S0), _f64(x_prev)
    lead = q.shape[:-2]
    T, m = q.shape[-2], q.shape[-1]
    dv = v.shape[-1]
    BH = int(np.prod(lead)) if lead else 1
    assert k.shape == q.shape and v.shape == lead + (T, dv)
    assert beta.shape == lead + (T,) and lam.shape == lead + (T,)
    if S0 is not None:
        assert S0.shape == lead + (m, dv)
    if x_prev is not None:
        assert x_prev.shape == lead + (m,)
    o = np.zeros(lead + (T, dv))
    S = np.zeros(lead + (m, dv))
    x_last = np.zeros(lead + (m,))
    traj = np.zeros(lead + (T, m, dv)) if trajectory else None
    nthreads = threads or os.cpu_count() or 1
    rc = lib.falcon_oracle_forward(
        _RULES[rule], BH, T, m, dv, _PHIS[phi], _RIDGES[ridge], eps, eps_gamma, _ptr(q), _ptr(k),
        _ptr(v), _ptr(beta), _ptr(lam), _ptr(S0), _ptr(x_prev), _ptr(o), _ptr(S),
        _ptr(x_last), _ptr(traj), int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (rc={rc})")
    out = {"o": o, "S": S, "x_last": x_last}
    if trajectory:
        out["S_traj"] = traj
    return out


def backward(rule, q, k, v, beta, lam, dO, S0=None, x_prev=None, dS_T=None, dx_last=None,
             phi="l2", eps=1e-6, eps_gamma=1e-6, threads=None, ridge="given"):
    """Gradients of L = <dO, o> + <dS_T, S_T> + <dx_last, x_last> through the
    Falcon-1 / Falcon-1A recurrence (reverse mode, token by token, fp64).

    Shapes as ``forward``; dO [..., T, dv]; dS_T [..., m, dv] and dx_last
    [..., m] may be None (zero cotangents).  Returns a dict with dq, dk
    [..., T, m], dv [..., T, dv], dbeta, dlambda [..., T] (dlambda is the
    gradient for the lam input: the base ridge when ridge="scaled"), dS0
    [..., m, dv] and dx_prev [..., m] (zeros for a fresh sequence).
    """
    lib = _load()
    q, k, v, beta, lam, dO = (_f64(t) for t in (q, k, v, beta, lam, dO))
    S0, x_prev, dS_T, dx_last = (_f64(t) for t in (S0, x_prev, dS_T, dx_last))
    lead = q.shape[:-2]
    T, m = q.shape[-2], q.shape[-1]
    dv = v.shape[-1]
    BH = int(np.prod(lead)) if lead else 1
    assert k.shape == q.shape and v.shape == lead + (T, dv) and dO.shape == v.shape
    assert beta.shape == lead + (T,) and lam.shape == lead + (T,)
    for t, shp in ((S0, (m, dv)), (dS_T, (m, dv)), (x_prev, (m,)), (dx_last, (m,))):
        if t is not None:
            assert t.shape == lead + shp
    out = {"dq": np.zeros(q.shape), "dk": np.zeros(q.shape), "dv": np.zeros(v.shape),
           "dbeta": np.zeros(beta.shape), "dlambda": np.zeros(beta.shape),
           "dS0": np.zeros(lead + (m, dv)), "dx_prev": np.zeros(lead + (m,))}
    nthreads = threads or os.cpu_count() or 1
    rc = lib.falcon_oracle_backward(
        _RULES[rule], BH, T, m, dv, _PHIS[phi], _RIDGES[ridge], eps, eps_gamma, _ptr(q), _ptr(k),
        _ptr(v), _ptr(beta), _ptr(lam), _ptr(S0), _ptr(x_prev), _ptr(dO), _ptr(dS_T),
        _ptr(dx_last), _ptr(out["dq"]), _ptr(out["dk"]), _ptr(out["dv"]), _ptr(out["dbeta"]),
        _ptr(out["dlambda"]), _ptr(out["dS0"]), _ptr(out["dx_prev"]), int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (rc={rc})")
    return out


def forward2(rule, q, k, v, beta, lam, S0=None, x_prev=None, phi="l2",
             eps=1e-6, eps_gamma=1e-6, threads=None, ridge="given"):
    """Falcon-2 / Falcon-2A over whole sequences: as ``forward`` except that
    ``beta`` has one gain per value column, shape [..., T, dv], and ``rule`` is
    "falcon2" or "falcon2a".  Returns a dict with o, S and x_last."""
    lib = _load()
    q, k, v, beta, lam = (_f64(t) for t in (q, k, v, beta, lam))
    S0, x_prev = _f64(S0), _f64(x_prev)
    lead = q.shape[:-2]
    T, m = q.shape[-2], q.shape[-1]
    dv = v.shape[-1]
    BH = int(np.prod(lead)) if lead else 1
    assert k.shape == q.shape and v.shape == lead + (T, dv)
    assert beta.shape == lead + (T, dv) and lam.shape == lead + (T,)
    if S0 is not None:
        assert S0.shape == lead + (m, dv)
    if x_prev is not None:
        assert x_prev.shape == lead + (m,)
    o = np.zeros(lead + (T, dv))
    S = np.zeros(lead + (m, dv))
    x_last = np.zeros(lead + (m,))
    nthreads = threads or os.cpu_count() or 1
    rc = lib.falcon2_oracle_forward(
        _RULES2[rule], BH, T, m, dv, _PHIS[phi], _RIDGES[ridge], eps, eps_gamma, _ptr(q), _ptr(k),
        _ptr(v), _ptr(beta), _ptr(lam), _ptr(S0), _ptr(x_prev), _ptr(o), _ptr(S),
        _ptr(x_last), int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (rc={rc})")
    return {"o": o, "S": S, "x_last": x_last}


def forward3a(q, k, v, beta, lam, window, S0=None, phi="l2", eps=1e-6, eps_gamma=1e-6,
              threads=None, ridge="given"):
    """Falcon-3A (sliding window of ``window`` write pairs) over whole fresh
    sequences; shapes as ``forward`` (no x_prev: the window does not reach
    into a previous segment).  Returns a dict with o, S and x_last."""
    lib = _load()
    q, k, v, beta, lam = (_f64(t) for t in (q, k, v, beta, lam))
    S0 = _f64(S0)
    lead = q.shape[:-2]
    T, m = q.shape[-2], q.shape[-1]
    dv = v.shape[-1]
    BH = int(np.prod(lead)) if lead else 1
    assert k.shape == q.shape and v.shape == lead + (T, dv)
    assert beta.shape == lead + (T,) and lam.shape == lead + (T,)
    if S0 is not None:
        assert S0.shape == lead + (m, dv)
    o = np.zeros(lead + (T, dv))
    S = np.zeros(lead + (m, dv))
    x_last = np.zeros(lead + (m,))
    nthreads = threads or os.cpu_count() or 1
    rc = lib.falcon3a_oracle_forward(
        BH, T, m, dv, _PHIS[phi], _RIDGES[ridge], int(window), eps, eps_gamma, _ptr(q), _ptr(k),
        _ptr(v), _ptr(beta), _ptr(lam), _ptr(S0), _ptr(o), _ptr(S), _ptr(x_last), int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (rc={rc})")
    return {"o": o, "S": S, "x_last": x_last}


def forward_normalized(q, k, v, beta, lam, S0=None, z0=None, x_prev=None, phi="l2",
                       eps=1e-6, eps_gamma=1e-6, eps_attn=1e-6, threads=None, ridge="given"):
    """Falcon-1A with the normalised read o_t = S_t^T phi(q_t) / (z_t^T phi(q_t)
    + eps_attn), z_t = gamma_t z_{t-1} + eta_t x_t (Section 2.2, Eq. (2.1)-(2.3),
    with the Falcon-1A gain and decay on the normaliser).  Shapes as in
    ``forward``; z0 [..., m] or None (zeros).  Returns o, S, z and x_last."""
    lib = _load()
    q, k, v, beta, lam = (_f64(t) for t in (q, k, v, beta, lam))
    S0, z0, x_prev = _f64(S0), _f64(z0), _f64(x_prev)
    lead = q.shape[:-2]
    T, m = q.shape[-2], q.shape[-1]
    dv = v.shape[-1]
    BH = int(np.prod(lead)) if lead else 1
    assert k.shape == q.shape and v.shape == lead + (T, dv)
    assert beta.shape == lead + (T,) and lam.shape == lead + (T,)
    for name, t, shp in (("S0", S0, lead + (m, dv)), ("z0", z0, lead + (m,)),
                         ("x_prev", x_prev, lead + (m,))):
        assert t is None or t.shape == shp, name
    o = np.zeros(lead + (T, dv))
    S = np.zeros(lead + (m, dv))
    z = np.zeros(lead + (m,))
    x_last = np.zeros(lead + (m,))
    rc = lib.falcon1a_oracle_forward_normalized(
        BH, T, m, dv, _PHIS[phi], _RIDGES[ridge], eps, eps_gamma, eps_attn, _ptr(q), _ptr(k),
        _ptr(v), _ptr(beta), _ptr(lam), _ptr(S0), _ptr(z0), _ptr(x_prev), _ptr(o), _ptr(S),
        _ptr(z), _ptr(x_last), int(threads or os.cpu_count() or 1))
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (rc={rc})")
    return {"o": o, "S": S, "z": z, "x_last": x_last}


def decode_step(rule, q, k, v, beta, lam, S, x_prev, fresh=None, phi="l2",
                eps=1e-6, eps_gamma=1e-6, ridge="given"):
    """One token for N independent states.  ``S`` [N, m, dv] and ``x_prev``
    [N, m] must be float64 numpy arrays; they are updated in place.  ``fresh``
    ([N] bool or None) marks states whose sequence starts at this token.
    Returns o [N, dv]."""
    lib = _load()
    q, k, v, beta, lam = (_f64(t) for t in (q, k, v, beta, lam))
    assert isinstance(S, np.ndarray) and S.dtype == np.float64 and S.flags.c_contiguous
    assert isinstance(x_prev, np.ndarray) and x_prev.dtype == np.float64
    assert x_prev.flags.c_contiguous
    N, m = q.shape
    dv = v.shape[-1]
    o = np.zeros((N, dv))
    fr = None
    if fresh is not None:
        fr = np.ascontiguousarray(np.asarray(fresh, dtype=np.uint8))
        fr = fr.ctypes.data_as(ctypes.POINTER(ctypes.c_ubyte))
    rc = lib.falcon_oracle_decode_step(
        _RULES[rule], N, m, dv, _PHIS[phi], _RIDGES[ridge], eps, eps_gamma, _ptr(q), _ptr(k),
        _ptr(v),
        _ptr(beta), _ptr(lam), _ptr(S), _ptr(x_prev), fr, _ptr(o))
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (rc={rc})")
    return o
