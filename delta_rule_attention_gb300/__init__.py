"""Python binding of the Falcon GB300 C library (include/falcon.h).

Argument marshalling only: every step of the computation runs in the CUDA
kernels of ``libfalcon_gb300.so``.  The functions carry the C names, take
torch CUDA tensors, pass their device pointers and the current CUDA stream,
and raise ``FalconError`` on a nonzero return code.  There is no fallback:
if the library is missing, importing a function that needs it raises.

    import delta_rule_attention_gb300 as falcon
    o, S, x_last = falcon.falcon1_fwd_chunked(q, k, v, beta, lam, chunk=64)
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfalcon_gb300.so")

FALCON_BF16 = 0
FALCON_F32 = 1
FALCON_PHI_IDENTITY = 0
FALCON_PHI_L2 = 1
FALCON_PHI_RMS = 2
_PHI = {"identity": FALCON_PHI_IDENTITY, "l2": FALCON_PHI_L2, "rms": FALCON_PHI_RMS}
FALCON_RIDGE_GIVEN = 0
FALCON_RIDGE_SCALED = 1
_RIDGE = {"given": FALCON_RIDGE_GIVEN, "scaled": FALCON_RIDGE_SCALED}
_DTYPE = {torch.bfloat16: FALCON_BF16, torch.float32: FALCON_F32}

# Entry points declared in include/falcon.h.
EXPORTS = (
    "falcon_workspace_bytes", "falcon1_fwd_chunked", "falcon1a_fwd_chunked",
    "falcon1_decode_step", "falcon1a_decode_step", "falcon_sync_check",
    "falcon_strerror", "falcon_version", "falcon1_fwd_chunked_fixed_scratch",
    "falcon_selftest_wait_timeout", "falcon2_fwd_recurrent", "falcon2a_fwd_recurrent",
    "falcon3a_fwd_recurrent", "falcon_bwd_workspace_bytes", "falcon1_bwd_chunked",
    "falcon1a_bwd_chunked", "falcon3a_fwd_chunked", "falcon2a_fwd_chunked",
    "falcon_normalized_workspace_bytes", "falcon1a_fwd_chunked_normalized",
    "falcon2_fwd_chunked",
)
FALCON_ERR_SCRATCH_LIMIT = -10
FALCON_FIXED_SCRATCH_BYTES = 16 * 1024 * 1024


class FalconError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what} failed with code {code}: {strerror(code)}")
        self.code = code


class falcon_shape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int64), ("H", ctypes.c_int64), ("T", ctypes.c_int64),
                ("m", ctypes.c_int32), ("dv", ctypes.c_int32), ("chunk", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("phi", ctypes.c_int32),
                ("eps", ctypes.c_float), ("eps_gamma", ctypes.c_float), ("ridge", ctypes.c_int32)]


_lib = None
_lock = threading.Lock()


def load_library(path: str | None = None):
    """Load the shared library (built by ``__graft_entry__.build()``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(
                f"{p} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'`"
                " (the CUDA library has no CPU fallback)")
        lib = ctypes.CDLL(p)
        vp, f32p, i64, i32, sz = (ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                                  ctypes.c_int32, ctypes.c_size_t)
        shp = ctypes.POINTER(falcon_shape)
        lib.falcon_workspace_bytes.restype = sz
        lib.falcon_workspace_bytes.argtypes = [shp]
        for name in ("falcon1_fwd_chunked", "falcon1a_fwd_chunked"):
            fn = getattr(lib, name)
            fn.restype = ctypes.c_int
            fn.argtypes = [shp, vp, vp, vp, f32p, f32p, f32p, f32p, vp, f32p, f32p, vp, sz, vp]
        lib.falcon_normalized_workspace_bytes.restype = sz
        lib.falcon_normalized_workspace_bytes.argtypes = [shp]
        lib.falcon1a_fwd_chunked_normalized.restype = ctypes.c_int
        lib.falcon1a_fwd_chunked_normalized.argtypes = [
            shp, vp, vp, vp, f32p, f32p, f32p, f32p, f32p, ctypes.c_float, vp, f32p, f32p, f32p,
            vp, sz, vp]
        lib.falcon_bwd_workspace_bytes.restype = sz
        lib.falcon_bwd_workspace_bytes.argtypes = [shp]
        for name in ("falcon1_bwd_chunked", "falcon1a_bwd_chunked"):
            fn = getattr(lib, name)
            fn.restype = ctypes.c_int
            fn.argtypes = [shp, vp, vp, vp, f32p, f32p, f32p, f32p, vp, f32p, f32p, vp, vp, vp,
                           f32p, f32p, f32p, f32p, vp, sz, vp]
        for name in ("falcon1_decode_step", "falcon1a_decode_step"):
            fn = getattr(lib, name)
            fn.restype = ctypes.c_int
            fn.argtypes = [i64, i32, i32, i32, i32, i32, ctypes.c_float, ctypes.c_float,
                           vp, vp, vp, f32p, f32p, f32p, f32p, vp, vp, vp]
        for name in ("falcon2_fwd_recurrent", "falcon2a_fwd_recurrent", "falcon2_fwd_chunked"):
            fn = getattr(lib, name)
            fn.restype = ctypes.c_int
            fn.argtypes = [shp, vp, vp, vp, f32p, f32p, f32p, f32p, vp, f32p, f32p, vp]
        lib.falcon2a_fwd_chunked.restype = ctypes.c_int
        lib.falcon2a_fwd_chunked.argtypes = [shp, vp, vp, vp, f32p, f32p, f32p, f32p, vp, f32p,
                                             f32p, vp, sz, vp]
        lib.falcon3a_fwd_chunked.restype = ctypes.c_int
        lib.falcon3a_fwd_chunked.argtypes = [shp, i32, vp, vp, vp, f32p, f32p, f32p, vp, f32p,
                                             f32p, vp, sz, vp]
        lib.falcon3a_fwd_recurrent.restype = ctypes.c_int
        lib.falcon3a_fwd_recurrent.argtypes = [shp, i32, vp, vp, vp, f32p, f32p, f32p, vp, f32p,
                                               f32p, vp]
        lib.falcon1_fwd_chunked_fixed_scratch.restype = ctypes.c_int
        lib.falcon1_fwd_chunked_fixed_scratch.argtypes = [shp, vp, vp, vp, f32p, f32p, f32p,
                                                          f32p, vp, f32p, f32p, vp]
        lib.falcon_selftest_wait_timeout.restype = ctypes.c_int
        lib.falcon_selftest_wait_timeout.argtypes = [ctypes.c_uint32, vp]
        lib.falcon_sync_check.restype = ctypes.c_int
        lib.falcon_sync_check.argtypes = [vp]
        lib.falcon_strerror.restype = ctypes.c_char_p
        lib.falcon_strerror.argtypes = [ctypes.c_int]
        lib.falcon_version.restype = ctypes.c_int
        lib.falcon_version.argtypes = []
        _lib = lib
        return lib


def strerror(code: int) -> str:
    try:
        return load_library().falcon_strerror(int(code)).decode()
    except RuntimeError:
        return f"code {code}"


def _ptr(t):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(rc, what):
    if rc != 0:
        raise FalconError(rc, what)


def _need(t, name, dtype=None, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return t


def make_shape(B, H, T, m, dv, chunk, dtype, phi="l2", eps=1e-6, eps_gamma=1e-6,
               ridge="given"):
    """phi: "identity", "l2" or "rms"; ridge: "given" (lambda is lambda_t) or
    "scaled" (lambda is the base ridge, lambda_t = lambda * ||x_t||^2)."""
    return falcon_shape(int(B), int(H), int(T), int(m), int(dv), int(chunk),
                        _DTYPE[dtype] if isinstance(dtype, torch.dtype) else int(dtype),
                        _PHI[phi] if isinstance(phi, str) else int(phi), float(eps),
                        float(eps_gamma), _RIDGE[ridge] if isinstance(ridge, str) else int(ridge))


def falcon_workspace_bytes(shape: falcon_shape) -> int:
    return int(load_library().falcon_workspace_bytes(ctypes.byref(shape)))


def _fwd(name, q, k, v, beta, lam, S0=None, x_prev=None, chunk=64, phi="l2", eps=1e-6,
         eps_gamma=1e-6, o=None, S_out=None, x_last=None, workspace=None, stream=None,
         want_x_last=True, ridge="given"):
    lib = load_library()
    _need(q, "q")
    B, H, T, m = q.shape
    dv = v.shape[-1]
    dt = q.dtype
    if dt not in _DTYPE:
        raise TypeError("q, k, v must be bfloat16 or float32")
    _need(k, "k", dt, (B, H, T, m))
    _need(v, "v", dt, (B, H, T, dv))
    _need(beta, "beta", torch.float32, (B, H, T))
    _need(lam, "lambda", torch.float32, (B, H, T))
    if S0 is not None:
        _need(S0, "S0", torch.float32, (B, H, m, dv))
    if x_prev is not None:
        _need(x_prev, "x_prev", torch.float32, (B, H, m))
    dev = q.device
    if o is None:
        o = torch.empty((B, H, T, dv), dtype=dt, device=dev)
    if S_out is None:
        S_out = torch.empty((B, H, m, dv), dtype=torch.float32, device=dev)
    if x_last is None and want_x_last:
        x_last = torch.empty((B, H, m), dtype=torch.float32, device=dev)
    shape = make_shape(B, H, T, m, dv, chunk, dt, phi, eps, eps_gamma, ridge)
    need = int(lib.falcon_workspace_bytes(ctypes.byref(shape)))
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = getattr(lib, name)(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(beta),
                            _ptr(lam), _ptr(S0), _ptr(x_prev), _ptr(o), _ptr(S_out),
                            _ptr(x_last), _ptr(workspace), ws_bytes, _stream(stream))
    _check(rc, name)
    return o, S_out, x_last


def falcon1_fwd_chunked(q, k, v, beta, lam, S0=None, x_prev=None, chunk=64, phi="l2",
                        eps=1e-6, eps_gamma=1e-6, **kw):
    """Falcon-1 chunk-parallel forward.  q, k [B,H,T,m], v [B,H,T,dv] (bf16 or
    fp32), beta, lam [B,H,T] fp32; S0 [B,H,m,dv] fp32 or None; x_prev [B,H,m]
    fp32 or None (fresh sequence).  Returns (o, S_T, x_last)."""
    return _fwd("falcon1_fwd_chunked", q, k, v, beta, lam, S0, x_prev, chunk, phi, eps,
                eps_gamma, **kw)


def falcon1_fwd_chunked_fixed_scratch(q, k, v, beta, lam, S0=None, x_prev=None, chunk=64,
                                      phi="l2", eps=1e-6, eps_gamma=1e-6, o=None, S_out=None,
                                      x_last=None, stream=None, ridge="given"):
    """Falcon-1 chunked forward that needs no workspace: for callers that
    cannot allocate device memory, the library uses a fixed scratch array of
    FALCON_FIXED_SCRATCH_BYTES built into it.  Pass preallocated o, S_out,
    x_last to keep the whole call free of allocation (otherwise this wrapper
    allocates the outputs with torch, as the caller's own buffers).  Calls whose
    GPU work overlaps share that array and race; the first call on a device
    resolves its address and should precede any stream capture.  Returns
    (o, S_T, x_last)."""
    lib = load_library()
    _need(q, "q")
    B, H, T, m = q.shape
    dv = v.shape[-1]
    dt = q.dtype
    if dt not in _DTYPE:
        raise TypeError("q, k, v must be bfloat16 or float32")
    dev = q.device
    if o is None:
        o = torch.empty((B, H, T, dv), dtype=dt, device=dev)
    if S_out is None:
        S_out = torch.empty((B, H, m, dv), dtype=torch.float32, device=dev)
    if x_last is None:
        x_last = torch.empty((B, H, m), dtype=torch.float32, device=dev)
    for t, name in ((k, "k"), (v, "v"), (beta, "beta"), (lam, "lambda"), (o, "o"),
                    (S_out, "S_out"), (x_last, "x_last"), (S0, "S0"), (x_prev, "x_prev")):
        if t is not None:
            _need(t, name)
    shape = make_shape(B, H, T, m, dv, chunk, dt, phi, eps, eps_gamma, ridge)
    rc = lib.falcon1_fwd_chunked_fixed_scratch(
        ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(lam), _ptr(S0),
        _ptr(x_prev), _ptr(o), _ptr(S_out), _ptr(x_last), _stream(stream))
    _check(rc, "falcon1_fwd_chunked_fixed_scratch")
    return o, S_out, x_last


def falcon1a_fwd_chunked(q, k, v, beta, lam, S0=None, x_prev=None, chunk=64, phi="l2",
                         eps=1e-6, eps_gamma=1e-6, **kw):
    """Falcon-1A chunk-parallel forward; arguments as falcon1_fwd_chunked."""
    return _fwd("falcon1a_fwd_chunked", q, k, v, beta, lam, S0, x_prev, chunk, phi, eps,
                eps_gamma, **kw)


def falcon_normalized_workspace_bytes(shape: falcon_shape) -> int:
    return int(load_library().falcon_normalized_workspace_bytes(ctypes.byref(shape)))


def falcon1a_fwd_chunked_normalized(q, k, v, beta, lam, S0=None, z0=None, x_prev=None,
                                    eps_attn=1e-6, chunk=64, phi="l2", eps=1e-6, eps_gamma=1e-6,
                                    o=None, S_out=None, z_out=None, x_last=None, workspace=None,
                                    stream=None, ridge="given"):
    """Falcon-1A forward with the normalised read o_t = S_t^T phi(q_t) /
    (z_t^T phi(q_t) + eps_attn), z_t = gamma_t z_{t-1} + eta_t x_t.  Arguments
    as falcon1a_fwd_chunked, plus z0 [B,H,m] fp32 or None.  Returns
    (o, S_T, z_T, x_last)."""
    lib = load_library()
    _need(q, "q")
    B, H, T, m = q.shape
    dv = v.shape[-1]
    dt = q.dtype
    if dt not in _DTYPE:
        raise TypeError("q, k, v must be bfloat16 or float32")
    _need(k, "k", dt, (B, H, T, m))
    _need(v, "v", dt, (B, H, T, dv))
    _need(beta, "beta", torch.float32, (B, H, T))
    _need(lam, "lambda", torch.float32, (B, H, T))
    for t, name, shp in ((S0, "S0", (B, H, m, dv)), (z0, "z0", (B, H, m)),
                         (x_prev, "x_prev", (B, H, m))):
        if t is not None:
            _need(t, name, torch.float32, shp)
    dev = q.device
    if o is None:
        o = torch.empty((B, H, T, dv), dtype=dt, device=dev)
    if S_out is None:
        S_out = torch.empty((B, H, m, dv), dtype=torch.float32, device=dev)
    if z_out is None:
        z_out = torch.empty((B, H, m), dtype=torch.float32, device=dev)
    if x_last is None:
        x_last = torch.empty((B, H, m), dtype=torch.float32, device=dev)
    shape = make_shape(B, H, T, m, dv, chunk, dt, phi, eps, eps_gamma, ridge)
    need = int(lib.falcon_normalized_workspace_bytes(ctypes.byref(shape)))
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = lib.falcon1a_fwd_chunked_normalized(
        ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(lam), _ptr(S0),
        _ptr(z0), _ptr(x_prev), float(eps_attn), _ptr(o), _ptr(S_out), _ptr(z_out),
        _ptr(x_last), _ptr(workspace), ws_bytes, _stream(stream))
    _check(rc, "falcon1a_fwd_chunked_normalized")
    return o, S_out, z_out, x_last


def falcon_bwd_workspace_bytes(shape: falcon_shape) -> int:
    return int(load_library().falcon_bwd_workspace_bytes(ctypes.byref(shape)))


def _bwd(name, q, k, v, beta, lam, dO, S0=None, x_prev=None, dS_T=None, dx_last=None, chunk=64,
         phi="l2", eps=1e-6, eps_gamma=1e-6, ridge="given", workspace=None, stream=None,
         grads=None):
    lib = load_library()
    _need(q, "q")
    B, H, T, m = q.shape
    dv = v.shape[-1]
    dt = q.dtype
    if dt not in _DTYPE:
        raise TypeError("q, k, v must be bfloat16 or float32")
    _need(k, "k", dt, (B, H, T, m))
    _need(v, "v", dt, (B, H, T, dv))
    _need(dO, "dO", dt, (B, H, T, dv))
    _need(beta, "beta", torch.float32, (B, H, T))
    _need(lam, "lambda", torch.float32, (B, H, T))
    for t, nm, shp in ((S0, "S0", (B, H, m, dv)), (dS_T, "dS_T", (B, H, m, dv)),
                       (x_prev, "x_prev", (B, H, m)), (dx_last, "dx_last", (B, H, m))):
        if t is not None:
            _need(t, nm, torch.float32, shp)
    dev = q.device
    g = grads if grads is not None else {}
    g.setdefault("dq", torch.empty_like(q))
    g.setdefault("dk", torch.empty_like(k))
    g.setdefault("dv", torch.empty_like(v))
    g.setdefault("dbeta", torch.empty_like(beta))
    g.setdefault("dlambda", torch.empty_like(lam))
    g.setdefault("dS0", torch.empty((B, H, m, dv), dtype=torch.float32, device=dev))
    g.setdefault("dx_prev", torch.empty((B, H, m), dtype=torch.float32, device=dev))
    shape = make_shape(B, H, T, m, dv, chunk, dt, phi, eps, eps_gamma, ridge)
    need = int(lib.falcon_bwd_workspace_bytes(ctypes.byref(shape)))
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = getattr(lib, name)(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(beta),
                            _ptr(lam), _ptr(S0), _ptr(x_prev), _ptr(dO), _ptr(dS_T),
                            _ptr(dx_last), _ptr(g["dq"]), _ptr(g["dk"]), _ptr(g["dv"]),
                            _ptr(g["dbeta"]), _ptr(g["dlambda"]), _ptr(g["dS0"]),
                            _ptr(g["dx_prev"]), _ptr(workspace), ws_bytes, _stream(stream))
    _check(rc, name)
    return g


def falcon1_bwd_chunked(q, k, v, beta, lam, dO, S0=None, x_prev=None, dS_T=None, dx_last=None,
                        chunk=64, phi="l2", eps=1e-6, eps_gamma=1e-6, **kw):
    """Backward of falcon1_fwd_chunked: gradients of <dO, o> + <dS_T, S_T> +
    <dx_last, x_last>.  dO has the dtype of q; dS_T [B,H,m,dv] and dx_last
    [B,H,m] fp32 or None.  Returns a dict with dq, dk, dv (dtype of q), dbeta,
    dlambda, dS0, dx_prev (fp32).  ``grads`` may pass preallocated outputs."""
    return _bwd("falcon1_bwd_chunked", q, k, v, beta, lam, dO, S0, x_prev, dS_T, dx_last,
                chunk, phi, eps, eps_gamma, **kw)


def falcon1a_bwd_chunked(q, k, v, beta, lam, dO, S0=None, x_prev=None, dS_T=None, dx_last=None,
                         chunk=64, phi="l2", eps=1e-6, eps_gamma=1e-6, **kw):
    """Backward of falcon1a_fwd_chunked; arguments as falcon1_bwd_chunked."""
    return _bwd("falcon1a_bwd_chunked", q, k, v, beta, lam, dO, S0, x_prev, dS_T, dx_last,
                chunk, phi, eps, eps_gamma, **kw)


def _fwd2(name, q, k, v, beta, lam, S0=None, x_prev=None, phi="l2", eps=1e-6,
          eps_gamma=1e-6, o=None, S_out=None, x_last=None, stream=None, want_x_last=True,
          ridge="given", workspace=None, chunked=False):
    lib = load_library()
    _need(q, "q")
    B, H, T, m = q.shape
    dv = v.shape[-1]
    dt = q.dtype
    if dt not in _DTYPE:
        raise TypeError("q, k, v must be bfloat16 or float32")
    _need(k, "k", dt, (B, H, T, m))
    _need(v, "v", dt, (B, H, T, dv))
    _need(beta, "beta", torch.float32, (B, H, T, dv))
    _need(lam, "lambda", torch.float32, (B, H, T))
    if S0 is not None:
        _need(S0, "S0", torch.float32, (B, H, m, dv))
    if x_prev is not None:
        _need(x_prev, "x_prev", torch.float32, (B, H, m))
    dev = q.device
    if o is None:
        o = torch.empty((B, H, T, dv), dtype=dt, device=dev)
    if S_out is None:
        S_out = torch.empty((B, H, m, dv), dtype=torch.float32, device=dev)
    if x_last is None and want_x_last:
        x_last = torch.empty((B, H, m), dtype=torch.float32, device=dev)
    shape = make_shape(B, H, T, m, dv, 64, dt, phi, eps, eps_gamma, ridge)
    if chunked:
        need = int(lib.falcon_workspace_bytes(ctypes.byref(shape)))
        if workspace is None and need > 0:
            workspace = torch.empty(need, dtype=torch.uint8, device=dev)
        ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
        rc = getattr(lib, name)(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(beta),
                                _ptr(lam), _ptr(S0), _ptr(x_prev), _ptr(o), _ptr(S_out),
                                _ptr(x_last), _ptr(workspace), ws_bytes, _stream(stream))
    else:
        rc = getattr(lib, name)(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(beta),
                                _ptr(lam), _ptr(S0), _ptr(x_prev), _ptr(o), _ptr(S_out),
                                _ptr(x_last), _stream(stream))
    _check(rc, name)
    return o, S_out, x_last


def falcon2a_fwd_chunked(q, k, v, beta, lam, S0=None, x_prev=None, phi="l2", eps=1e-6,
                         eps_gamma=1e-6, **kw):
    """Falcon-2A forward in chunk form (tensor cores for bf16 with m = dv = 64,
    the token-recurrent kernel otherwise); arguments as falcon2a_fwd_recurrent,
    plus an optional workspace of falcon_workspace_bytes(shape) bytes."""
    return _fwd2("falcon2a_fwd_chunked", q, k, v, beta, lam, S0, x_prev, phi, eps, eps_gamma,
                 chunked=True, **kw)


def falcon2_fwd_chunked(q, k, v, beta, lam, S0=None, x_prev=None, phi="l2", eps=1e-6,
                        eps_gamma=1e-6, **kw):
    """Falcon-2 forward in chunk form (tensor cores for bf16 with m = dv = 64,
    one CTA per head; the token-recurrent kernel otherwise); arguments and
    results as falcon2_fwd_recurrent, no workspace."""
    return _fwd2("falcon2_fwd_chunked", q, k, v, beta, lam, S0, x_prev, phi, eps, eps_gamma,
                 **kw)


def falcon2_fwd_recurrent(q, k, v, beta, lam, S0=None, x_prev=None, phi="l2", eps=1e-6,
                          eps_gamma=1e-6, **kw):
    """Falcon-2 forward (per-column step sizes), token-recurrent.  As
    falcon1_fwd_chunked except beta [B,H,T,dv] fp32 (one gain per value column)
    and no chunk or workspace.  Returns (o, S_T, x_last)."""
    return _fwd2("falcon2_fwd_recurrent", q, k, v, beta, lam, S0, x_prev, phi, eps, eps_gamma,
                 **kw)


def falcon2a_fwd_recurrent(q, k, v, beta, lam, S0=None, x_prev=None, phi="l2", eps=1e-6,
                           eps_gamma=1e-6, **kw):
    """Falcon-2A forward (per-column inner-product rule); arguments as
    falcon2_fwd_recurrent."""
    return _fwd2("falcon2a_fwd_recurrent", q, k, v, beta, lam, S0, x_prev, phi, eps, eps_gamma,
                 **kw)


def falcon3a_fwd_recurrent(q, k, v, beta, lam, window, S0=None, phi="l2", eps=1e-6,
                           eps_gamma=1e-6, o=None, S_out=None, x_last=None, stream=None,
                           want_x_last=True, ridge="given"):
    """Falcon-3A forward (sliding window of ``window`` write pairs, 1..32) over
    fresh sequences.  q, k [B,H,T,m], v [B,H,T,dv] (bf16 or fp32), beta, lam
    [B,H,T] fp32; S0 [B,H,m,dv] fp32 or None.  Returns (o, S_T, x_last)."""
    lib = load_library()
    _need(q, "q")
    B, H, T, m = q.shape
    dv = v.shape[-1]
    dt = q.dtype
    if dt not in _DTYPE:
        raise TypeError("q, k, v must be bfloat16 or float32")
    _need(k, "k", dt, (B, H, T, m))
    _need(v, "v", dt, (B, H, T, dv))
    _need(beta, "beta", torch.float32, (B, H, T))
    _need(lam, "lambda", torch.float32, (B, H, T))
    if S0 is not None:
        _need(S0, "S0", torch.float32, (B, H, m, dv))
    dev = q.device
    if o is None:
        o = torch.empty((B, H, T, dv), dtype=dt, device=dev)
    if S_out is None:
        S_out = torch.empty((B, H, m, dv), dtype=torch.float32, device=dev)
    if x_last is None and want_x_last:
        x_last = torch.empty((B, H, m), dtype=torch.float32, device=dev)
    shape = make_shape(B, H, T, m, dv, 64, dt, phi, eps, eps_gamma, ridge)
    rc = lib.falcon3a_fwd_recurrent(ctypes.byref(shape), int(window), _ptr(q), _ptr(k), _ptr(v),
                                    _ptr(beta), _ptr(lam), _ptr(S0), _ptr(o), _ptr(S_out),
                                    _ptr(x_last), _stream(stream))
    _check(rc, "falcon3a_fwd_recurrent")
    return o, S_out, x_last


def falcon3a_fwd_chunked(q, k, v, beta, lam, window, S0=None, phi="l2", eps=1e-6,
                         eps_gamma=1e-6, o=None, S_out=None, x_last=None, workspace=None,
                         stream=None, want_x_last=True, ridge="given"):
    """Falcon-3A forward in chunk form (the masked-attention form; tensor cores
    for bf16 with m = dv = 64, the token-recurrent kernel otherwise).
    Arguments as falcon3a_fwd_recurrent, plus an optional workspace of
    falcon_workspace_bytes(shape) bytes.  Returns (o, S_T, x_last)."""
    lib = load_library()
    _need(q, "q")
    B, H, T, m = q.shape
    dv = v.shape[-1]
    dt = q.dtype
    if dt not in _DTYPE:
        raise TypeError("q, k, v must be bfloat16 or float32")
    _need(k, "k", dt, (B, H, T, m))
    _need(v, "v", dt, (B, H, T, dv))
    _need(beta, "beta", torch.float32, (B, H, T))
    _need(lam, "lambda", torch.float32, (B, H, T))
    if S0 is not None:
        _need(S0, "S0", torch.float32, (B, H, m, dv))
    dev = q.device
    if o is None:
        o = torch.empty((B, H, T, dv), dtype=dt, device=dev)
    if S_out is None:
        S_out = torch.empty((B, H, m, dv), dtype=torch.float32, device=dev)
    if x_last is None and want_x_last:
        x_last = torch.empty((B, H, m), dtype=torch.float32, device=dev)
    shape = make_shape(B, H, T, m, dv, 64, dt, phi, eps, eps_gamma, ridge)
    need = int(lib.falcon_workspace_bytes(ctypes.byref(shape)))
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = lib.falcon3a_fwd_chunked(ctypes.byref(shape), int(window), _ptr(q), _ptr(k), _ptr(v),
                                  _ptr(beta), _ptr(lam), _ptr(S0), _ptr(o), _ptr(S_out),
                                  _ptr(x_last), _ptr(workspace), ws_bytes, _stream(stream))
    _check(rc, "falcon3a_fwd_chunked")
    return o, S_out, x_last


def _decode(name, q, k, v, beta, lam, S, x_prev, fresh=None, phi="l2", eps=1e-6,
            eps_gamma=1e-6, o=None, stream=None, ridge="given"):
    lib = load_library()
    _need(q, "q")
    N, m = q.shape
    dv = v.shape[-1]
    dt = q.dtype
    _need(k, "k", dt, (N, m))
    _need(v, "v", dt, (N, dv))
    _need(beta, "beta", torch.float32, (N,))
    _need(lam, "lambda", torch.float32, (N,))
    _need(S, "S", torch.float32, (N, m, dv))
    _need(x_prev, "x_prev", torch.float32, (N, m))
    if fresh is not None:
        _need(fresh, "fresh", torch.uint8, (N,))
    if o is None:
        o = torch.empty((N, dv), dtype=dt, device=q.device)
    rc = getattr(lib, name)(N, m, dv, _DTYPE[dt], _PHI[phi], _RIDGE[ridge], float(eps),
                            float(eps_gamma),
                            _ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(lam), _ptr(S),
                            _ptr(x_prev), _ptr(fresh), _ptr(o), _stream(stream))
    _check(rc, name)
    return o


def falcon1_decode_step(q, k, v, beta, lam, S, x_prev, fresh=None, phi="l2", eps=1e-6,
                        eps_gamma=1e-6, o=None, stream=None, ridge="given"):
    """One Falcon-1 token for N states: S [N,m,dv] and x_prev [N,m] are updated
    in place; fresh [N] uint8 marks sequences starting at this token.  Returns o."""
    return _decode("falcon1_decode_step", q, k, v, beta, lam, S, x_prev, fresh, phi, eps,
                   eps_gamma, o, stream, ridge)


def falcon1a_decode_step(q, k, v, beta, lam, S, x_prev, fresh=None, phi="l2", eps=1e-6,
                         eps_gamma=1e-6, o=None, stream=None, ridge="given"):
    """One Falcon-1A token for N states (see falcon1_decode_step)."""
    return _decode("falcon1a_decode_step", q, k, v, beta, lam, S, x_prev, fresh, phi, eps,
                   eps_gamma, o, stream, ridge)


def falcon_sync_check(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device error status."""
    return int(load_library().falcon_sync_check(_stream(stream)))


def falcon_selftest_wait_timeout(limit_us: int = 20000, stream=None) -> None:
    """Run the failure-path diagnostic: a kernel whose wait can never complete
    gives up after limit_us and records the expiry in the device error word
    (read it with falcon_sync_check, which then returns FALCON_ERR_TIMEOUT)."""
    _check(load_library().falcon_selftest_wait_timeout(int(limit_us), _stream(stream)),
           "falcon_selftest_wait_timeout")


def falcon_version() -> int:
    return int(load_library().falcon_version())
