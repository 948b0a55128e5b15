"""fp64 check of the chunk forms the Falcon-3A and Falcon-2A tensor-core
kernels implement (neither the oracle nor the CUDA path: numpy restatements,
checked against the oracle's token loops).

Falcon-3A (page hyper.ai/fr/papers/2608.27763, Section 4.5 and the
masked-attention form of Section 4.6): within a chunk entered with state S,
S_t = e^{g_t} S + sum_j x_j v_j^T w_{t,j} over the chunk's pairs and the 64
before it, where w follows w_{t,j} = gamma_t w_{t-1,j} + [j in I_t] eta_t / B_t
down each column; o_t = S_t^T phi(q_t).

Falcon-2A (Section 4.3 with the per-column step sizes of Section 4.2): per
column j, G_{j,.} the chunk-local log prefix of that column,
o_{t,j} = e^{G_{j,t}} (Q S)_{t,j} + e^{G_{j,t} - r_j} (A U~)_{t,j},
U~_{s,j} = e^{r_j - G_{j,s}} eta_{j,s} v_{s,j} (A the causal part of Q X^T,
r_j = G_{j,C}/2), and S'_{:,j} = e^{G_{j,C}} S_{:,j} + X^T V'_{:,j},
V'_{s,j} = e^{G_{j,C} - G_{j,s}} eta_{j,s} v_{s,j}.
"""
import numpy as np
import pytest

import oracle


def _l2(u):
    return u / np.maximum(np.linalg.norm(u, axis=-1, keepdims=True), 1e-12)


def falcon3a_chunked(q, k, v, beta, lam, window, C, S0=None, eps=1e-6, eps_gamma=1e-6):
    BH, T, m = q.shape
    dv = v.shape[-1]
    o = np.zeros((BH, T, dv))
    S_out = np.zeros((BH, m, dv))
    for b in range(BH):
        qf, kf = _l2(q[b]), _l2(k[b])
        x = np.zeros((T + 1, m))          # x_j = phi(k_{j-1}), x_0 = 0
        x[1:] = kf
        E = (x * x).sum(-1)
        S = S0[b].copy() if S0 is not None else np.zeros((m, dv))
        for t0 in range(0, T, C):
            n = min(C, T - t0)
            coef = np.zeros(C)
            gam = np.ones(C)
            for i in range(n):
                t = t0 + i
                if t < 1:
                    continue
                j0 = max(t - window + 1, 1)
                Bt = t - j0 + 1
                Eb = E[j0:t + 1].mean()
                den = Eb + lam[b, t] + eps
                eta = beta[b, t] / den if den > 0 else 0.0
                a = min(eta * lam[b, t], 1 - eps_gamma)
                gam[i] = 1 - a
                coef[i] = eta / Bt
            g = np.cumsum(np.log(gam))
            # the chunk's pairs and the 64 before it
            js = np.arange(t0 - 64, t0 + C)
            W = np.zeros((C, len(js)))
            w = np.zeros(len(js))
            for i in range(C):
                t = t0 + i
                inn = (js >= 1) & (js <= t) & (t <= js + window - 1)
                w = gam[i] * w + np.where(inn, coef[i], 0.0)
                W[i] = w
            X = np.array([x[j] if 0 <= j <= T else np.zeros(m) for j in js])
            Vt = np.array([v[b, j] if 0 <= j < T else np.zeros(dv) for j in js])
            Q = np.zeros((C, m))
            Q[:n] = qf[t0:t0 + n]
            O = np.exp(g)[:, None] * (Q @ S) + ((Q @ X.T) * W) @ Vt
            S = np.exp(g[-1]) * S + X.T @ (W[-1][:, None] * Vt)
            o[b, t0:t0 + n] = O[:n]
        S_out[b] = S
    return o, S_out


def falcon2a_chunked(q, k, v, beta, lam, C, S0=None, x_prev=None, eps=1e-6, eps_gamma=1e-6):
    BH, T, m = q.shape
    dv = v.shape[-1]
    o = np.zeros((BH, T, dv))
    S_out = np.zeros((BH, m, dv))
    for b in range(BH):
        qf, kf = _l2(q[b]), _l2(k[b])
        x = np.zeros((T, m))
        x[1:] = kf[:-1]
        if x_prev is not None:
            x[0] = x_prev[b]
        E = (x * x).sum(-1)
        S = S0[b].copy() if S0 is not None else np.zeros((m, dv))
        for t0 in range(0, T, C):
            n = min(C, T - t0)
            eta = np.zeros((C, dv))
            lg = np.zeros((C, dv))
            for i in range(n):
                t = t0 + i
                if t == 0 and x_prev is None:
                    continue
                den = E[t] + lam[b, t] + eps
                et = np.where(den > 0, beta[b, t] / den, 0.0)
                a = np.minimum(et * lam[b, t], 1 - eps_gamma)
                eta[i] = et
                lg[i] = np.log(1 - a)
            G = np.cumsum(lg, axis=0)          # per column
            r = 0.5 * G[-1]
            X = np.zeros((C, m))
            X[:n] = x[t0:t0 + n]
            Q = np.zeros((C, m))
            Q[:n] = qf[t0:t0 + n]
            V = np.zeros((C, dv))
            V[:n] = v[b, t0:t0 + n]
            A = np.tril(Q @ X.T)
            Ut = np.exp(r[None, :] - G) * eta * V
            O = np.exp(G) * (Q @ S) + np.exp(G - r[None, :]) * (A @ Ut)
            Vp = np.exp(G[-1][None, :] - G) * eta * V
            S = np.exp(G[-1])[None, :] * S + X.T @ Vp
            o[b, t0:t0 + n] = O[:n]
        S_out[b] = S
    return o, S_out


def _case(seed, BH=2, T=150, m=6, dv=5, lam_shift=-1.5, per_column=False):
    g = np.random.default_rng(seed)
    q = g.standard_normal((BH, T, m))
    k = g.standard_normal((BH, T, m))
    v = g.standard_normal((BH, T, dv))
    beta = 2 / (1 + np.exp(-g.standard_normal((BH, T, dv) if per_column else (BH, T))))
    lam = np.log1p(np.exp(g.standard_normal((BH, T)) + lam_shift))
    S0 = g.standard_normal((BH, m, dv)) * 0.5
    xp = _l2(g.standard_normal((BH, m)))
    return q, k, v, beta, lam, S0, xp


@pytest.mark.parametrize("window", [1, 3, 32])
@pytest.mark.parametrize("C", [16, 64])
@pytest.mark.parametrize("lam_shift", [-1.5, 2.5])
def test_falcon3a_chunk_form(window, C, lam_shift):
    q, k, v, beta, lam, S0, _ = _case(7 + window, lam_shift=lam_shift)
    o, S = falcon3a_chunked(q, k, v, beta, lam, window, C, S0=S0)
    ref = oracle.forward3a(q, k, v, beta, lam, window, S0=S0, phi="l2", threads=1)
    np.testing.assert_allclose(o, ref["o"], rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(S, ref["S"], rtol=1e-10, atol=1e-10)


@pytest.mark.parametrize("C", [16, 64])
@pytest.mark.parametrize("carried", [False, True])
def test_falcon2a_chunk_form(C, carried):
    q, k, v, beta, lam, S0, xp = _case(21, per_column=True)
    kw = dict(S0=S0, x_prev=xp) if carried else {}
    o, S = falcon2a_chunked(q, k, v, beta, lam, C, **kw)
    ref = oracle.forward2("falcon2a", q, k, v, beta, lam, phi="l2", threads=1, **kw)
    np.testing.assert_allclose(o, ref["o"], rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(S, ref["S"], rtol=1e-10, atol=1e-10)
