"""fp64 check of the chunk decomposition the CUDA kernels implement.

This is neither the oracle nor the CUDA path: it restates, in numpy, the
per-chunk algebra derived from the Falcon-1 update (p1 = page
hyper.ai/fr/papers/2608.27763, Section 3.1 Eq. (3.3); positive-decay
renormalisation, Section 4.4 Eq. (4.15)-(4.16) and Section 4.3 'Decay
positivity') and checks it against the oracle.  It fixes the derivation
before any kernel is written: chunk sizes 1..T, ragged tails, carried state
and clamp-active draws.

Within a chunk with entering state S, local tokens i = 1..C, write features
x_i, step sizes eta_i, log-decays l_i = log(gamma_i), inclusive prefixes
g_i = l_1 + ... + l_i (g_0 = 0):

  Falcon-1:  A_ij = eta_i e^{g_{i-1} - g_j} <x_i, x_j>  (j < i),  T = (I + A)^{-1}
             W = T Diag(eta_i e^{g_{i-1}}) X,   U~ = T Diag(eta) V
  Falcon-1A: W = 0,                              U~ = Diag(eta) V
  P_ij = e^{g_i - g_j} <q_i, x_j>  (j <= i)
  Xt   = Diag(e^{g_C - g_j}) X
  S'   = (e^{g_C} I - Xt^T W) S + Xt^T U~
  O    = (Diag(e^{g}) Q - P W) S + P U~

Every exponential has a non-positive argument, so nothing overflows when the
decay product of a chunk underflows.
"""
import numpy as np
import pytest

import oracle


def _phi(u, phi):
    if phi == "identity":
        return u
    return u / np.maximum(np.linalg.norm(u, axis=-1, keepdims=True), 1e-12)


def chunked_forward(rule, q, k, v, beta, lam, C, S0=None, x_prev=None, phi="l2",
                    eps=1e-6, eps_gamma=1e-6):
    BH, T, m = q.shape
    dv = v.shape[-1]
    Q, K = _phi(q, phi), _phi(k, phi)
    o = np.zeros((BH, T, dv))
    S_out = np.zeros((BH, m, dv))
    for b in range(BH):
        S = np.zeros((m, dv)) if S0 is None else S0[b].copy()
        xp = None if x_prev is None else x_prev[b]
        for c0 in range(0, T, C):
            n = min(C, T - c0)
            X = np.zeros((n, m))
            for i in range(n):
                t = c0 + i
                if t > 0:
                    X[i] = K[b, t - 1]
                elif xp is not None:
                    X[i] = xp
            den = (X * X).sum(1) + lam[b, c0:c0 + n] + eps
            eta = np.where(den > 0, beta[b, c0:c0 + n] / np.where(den > 0, den, 1), 0.0)
            if c0 == 0 and xp is None:
                eta[0] = 0.0
            alpha = np.minimum(eta * lam[b, c0:c0 + n], 1 - eps_gamma)
            lg = np.log1p(-alpha)
            g = np.cumsum(lg)
            gx = g - lg  # g_{i-1}
            Qc, Vc = Q[b, c0:c0 + n], v[b, c0:c0 + n]
            ii, jj = np.meshgrid(np.arange(n), np.arange(n), indexing="ij")
            if rule == "falcon1":
                A = np.where(jj < ii, eta[:, None] * np.exp(np.minimum(gx[:, None] - g[None, :], 0))
                             * (X @ X.T), 0.0)
                Tm = np.linalg.inv(np.eye(n) + A)
                W = Tm @ ((eta * np.exp(gx))[:, None] * X)
                Ut = Tm @ (eta[:, None] * Vc)
            else:
                W = np.zeros((n, m))
                Ut = eta[:, None] * Vc
            P = np.where(jj <= ii, np.exp(np.minimum(g[:, None] - g[None, :], 0)) * (Qc @ X.T), 0.0)
            Xt = np.exp(g[-1] - g)[:, None] * X
            o[b, c0:c0 + n] = (np.exp(g)[:, None] * Qc - P @ W) @ S + P @ Ut
            S = (np.exp(g[-1]) * np.eye(m) - Xt.T @ W) @ S + Xt.T @ Ut
        S_out[b] = S
    return o, S_out


def _case(seed, BH=2, T=70, m=6, dv=4, lam_shift=-2.0):
    g = np.random.default_rng(seed)
    q = g.standard_normal((BH, T, m))
    k = g.standard_normal((BH, T, m))
    v = g.standard_normal((BH, T, dv))
    beta = 2 / (1 + np.exp(-g.standard_normal((BH, T))))
    lam = np.log1p(np.exp(g.standard_normal((BH, T)) + lam_shift))
    return q, k, v, beta, lam


@pytest.mark.parametrize("rule", ["falcon1", "falcon1a"])
@pytest.mark.parametrize("C", [1, 7, 16, 64, 70, 128])
@pytest.mark.parametrize("lam_shift", [-2.0, 1.0])
def test_chunk_form_matches_oracle(rule, C, lam_shift):
    q, k, v, beta, lam = _case(31, lam_shift=lam_shift)
    S0 = np.random.default_rng(32).standard_normal((2, 6, 4))
    xp = np.random.default_rng(33).standard_normal((2, 6))
    for carried in (False, True):
        ref = oracle.forward(rule, q, k, v, beta, lam, S0=S0 if carried else None,
                             x_prev=_phi(xp, "l2") if carried else None)
        o, S = chunked_forward(rule, q, k, v, beta, lam, C, S0=S0 if carried else None,
                               x_prev=_phi(xp, "l2") if carried else None)
        np.testing.assert_allclose(o, ref["o"], rtol=1e-9, atol=1e-9)
        np.testing.assert_allclose(S, ref["S"], rtol=1e-9, atol=1e-9)


def test_chunk_form_survives_underflowing_decay():
    """Large lambda with beta near 2: the clamp fires and a chunk's decay
    product exp(g_C) is far below the smallest normal double; the
    chunk form must stay finite and equal the recurrence."""
    q, k, v, beta, lam = _case(41, T=256, lam_shift=4.0)
    beta[:] = 1.99
    o, S = chunked_forward("falcon1", q, k, v, beta, lam, 64, eps_gamma=1e-6)
    ref = oracle.forward("falcon1", q, k, v, beta, lam, eps_gamma=1e-6)
    assert np.isfinite(o).all() and np.isfinite(S).all()
    np.testing.assert_allclose(o, ref["o"], rtol=1e-9, atol=1e-9)
