"""fp64 check of the chunk form the normalised read's GPU path implements
(neither the oracle nor the CUDA path: a numpy restatement, checked against
the oracle's token loop).

The normaliser of page hyper.ai/fr/papers/2608.27763, Section 2.2, Eq. (2.3),
with the Falcon-1A gain and clamped decay, z_t = gamma_t z_{t-1} + eta_t x_t, is
the state column that a constant unit target would write.  Inside a chunk
entered with z_c (g the chunk-local inclusive log prefix of gamma):

    z_t^T phi(q_t) = e^{g_t} <phi(q_t), z_c> + r_t,   r_t = sum_{j <= t} P_tj eta_j,
    P_tj = e^{g_t - g_j} <phi(q_t), x_j>,
    z_{c+1} = e^{g_C} z_c + y_C,                      y_C = sum_j eta_j e^{g_C - g_j} x_j,

so r_t is the Gram rows P (the same decayed rows the numerator's in-chunk term
P Diag(eta) V uses) times the step sizes, and y_C the decayed features times
the step sizes.  The read divides the Falcon-1A numerator by
z_t^T phi(q_t) + eps_attn.
"""
import numpy as np
import pytest

import oracle


def _l2(u):
    return u / np.maximum(np.linalg.norm(u, axis=-1, keepdims=True), 1e-12)


def normalized_chunked(q, k, v, beta, lam, C, S0=None, z0=None, x_prev=None, eps=1e-6,
                       eps_gamma=1e-6, eps_attn=1e-6):
    """The normalised read from the per-chunk terms (r_t, y_C, e^{g_t}, e^{g_C})
    chained across chunks; the numerator is the oracle's Falcon-1A forward."""
    BH, T, m = q.shape
    num = oracle.forward("falcon1a", q, k, v, beta, lam, S0=S0, x_prev=x_prev, phi="l2",
                         eps=eps, eps_gamma=eps_gamma, threads=1)
    den = np.zeros((BH, T))
    z_out = np.zeros((BH, m))
    for b in range(BH):
        qf = _l2(q[b])
        x = np.zeros((T, m))                  # x_t: write feature of token t
        x[1:] = _l2(k[b, :-1])
        if x_prev is not None:
            x[0] = x_prev[b]
        E = (x * x).sum(-1)
        eta = np.zeros(T)
        lg = np.zeros(T)
        for t in range(T):
            if t == 0 and x_prev is None:     # the sentinel: no write
                continue
            d = E[t] + lam[b, t] + eps
            eta[t] = beta[b, t] / d if d > 0 else 0.0
            a = min(eta[t] * lam[b, t], 1 - eps_gamma)
            lg[t] = np.log(eps_gamma) if a >= 1 - eps_gamma else np.log1p(-a)
        z = z0[b].copy() if z0 is not None else np.zeros(m)
        for t0 in range(0, T, C):
            sl = slice(t0, min(T, t0 + C))
            g = np.cumsum(lg[sl])
            Q, X, et = qf[sl], x[sl], eta[sl]
            D = np.tril(np.exp(np.minimum(g[:, None] - g[None, :], 0.0)))
            P = D * (Q @ X.T)
            r = P @ et                                   # the in-chunk read
            yC = X.T @ (et * np.exp(g[-1] - g))          # the chunk's increment
            den[b, sl] = np.exp(g) * (Q @ z) + r
            z = np.exp(g[-1]) * z + yC
        z_out[b] = z
    o = num["o"] / (den[..., None] + eps_attn)
    return o, z_out


def _case(seed, BH=2, T=150, m=6, dv=5, lam_shift=-1.5):
    g = np.random.default_rng(seed)
    # positive features: the setting in which the pages call the read attention-like
    q = np.abs(g.standard_normal((BH, T, m))) + 0.05
    k = np.abs(g.standard_normal((BH, T, m))) + 0.05
    v = g.standard_normal((BH, T, dv))
    beta = 2 / (1 + np.exp(-g.standard_normal((BH, T))))
    lam = np.log1p(np.exp(g.standard_normal((BH, T)) + lam_shift))
    S0 = g.standard_normal((BH, m, dv)) * 0.5
    z0 = g.random((BH, m)) + 0.1
    xp = _l2(np.abs(g.standard_normal((BH, m))))
    return q, k, v, beta, lam, S0, z0, xp


@pytest.mark.parametrize("C", [16, 64])
@pytest.mark.parametrize("carried", [False, True])
@pytest.mark.parametrize("lam_shift", [-1.5, 2.5])
def test_normalizer_chunk_terms(C, carried, lam_shift):
    q, k, v, beta, lam, S0, z0, xp = _case(31 + C, lam_shift=lam_shift)
    kw = dict(S0=S0, z0=z0, x_prev=xp) if carried else {}
    o, z = normalized_chunked(q, k, v, beta, lam, C, **kw)
    ref = oracle.forward_normalized(q, k, v, beta, lam, phi="l2", threads=1, **kw)
    np.testing.assert_allclose(z, ref["z"], rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(o, ref["o"], rtol=1e-9, atol=1e-12)


def test_normalizer_chunk_terms_catch_a_dropped_decay():
    """The check is sharp: the increment without its decay e^{g_C - g_j} (a
    plausible slip) leaves z_T off by far more than the tolerance."""
    q, k, v, beta, lam, S0, z0, xp = _case(5, lam_shift=1.0)
    ref = oracle.forward_normalized(q, k, v, beta, lam, S0=S0, z0=z0, x_prev=xp, phi="l2",
                                    threads=1)
    BH, T, m = q.shape
    x = np.zeros((BH, T, m))
    x[:, 1:] = _l2(k[:, :-1])
    x[:, 0] = xp
    E = (x * x).sum(-1)
    eta = beta / (E + lam + 1e-6)
    a = np.minimum(eta * lam, 1 - 1e-6)
    lg = np.log1p(-a)
    z = z0.copy()
    for t0 in range(0, T, 16):
        sl = slice(t0, min(T, t0 + 16))
        g = np.cumsum(lg[:, sl], axis=1)
        z = np.exp(g[:, -1:]) * z + np.einsum("btm,bt->bm", x[:, sl], eta[:, sl])  # no decay
    assert np.abs(z - ref["z"]).max() > 1e-3 * np.abs(ref["z"]).max()
