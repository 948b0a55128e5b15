"""fp64 check of the chunk-form backward the CUDA kernels implement.

Neither the oracle nor the CUDA path: a numpy restatement of the per-chunk
algebra of the backward kernels, checked against the oracle's token-by-token
reverse mode (itself pinned by finite differences).  It fixes the derivation
before any kernel is written.

Forward of one chunk (entering state S, local tokens i = 1..C; notation of
test_chunk_algebra.py; p1 = page hyper.ai/fr/papers/2608.27763, Section 3.1
Eq. (3.3), Section 4.4 Eq. (4.15)-(4.16)):

  R = Diag(eta) V - Diag(eta e^{g_-}) X S        (Falcon-1A: R = Diag(eta) V)
  U = (I + A)^{-1} R                              (Falcon-1A: A = 0)
  O = Diag(e^g) Q S + P U,   S' = e^{g_C} S + X^T Diag(e^{g_C - g}) U

Backward of the chunk, given dO and the cotangent dS' of the state leaving it
(the cotangent of the entering state is Mc^T [dS'; dO], the transposed chunk
map, computed by a reverse scan over chunks):

  dU = P^T dO + Diag(e^{g_C - g}) X dS'
  dR = (I + A)^{-T} dU                            (one back substitution)
  dA = -(dR U^T) on j < i,   dP = (dO U^T) on j <= i,   dV = Diag(eta) dR
  dQ = Diag(e^g) dO S^T + (dP o E) X
  dX = -Diag(eta e^{g_-}) dR S^T + (dP o E)^T Q + Diag(e^{g_C - g}) U dS'^T
       + (dK + dK^T) X + 2 Diag(dE) X,   dK_ij = dA_ij eta_i e^{g_{i-1} - g_j}
  with E_ij = e^{g_i - g_j}; the log-prefix cotangent dg collects every
  e^{...} factor, the per-token d log(gamma_r) is its suffix sum, and the
  chain through the clamp, eta = beta / (E + lambda + eps) and the ridge
  follows as in the oracle.
"""
import numpy as np
import pytest

import oracle


def _phi(u, phi):
    if phi == "identity":
        return u
    if phi == "rms":
        return u / np.sqrt((u * u).sum(-1, keepdims=True) / u.shape[-1] + 1e-6)
    return u / np.maximum(np.linalg.norm(u, axis=-1, keepdims=True), 1e-12)


def _phi_vjp(u, g, phi):
    if phi == "identity":
        return g
    if phi == "rms":
        m = u.shape[-1]
        s = 1.0 / np.sqrt((u * u).sum(-1, keepdims=True) / m + 1e-6)
        return s * g - s ** 3 * u * (u * g).sum(-1, keepdims=True) / m
    n = np.maximum(np.linalg.norm(u, axis=-1, keepdims=True), 1e-12)
    f = u / n
    return (g - f * (f * g).sum(-1, keepdims=True)) / n


def chunked_backward(rule, q, k, v, beta, lam, dO, C, S0=None, x_prev=None, dS_T=None,
                     dx_last=None, phi="l2", ridge="given", eps=1e-6, eps_gamma=1e-6):
    f1 = rule == "falcon1"
    BH, T, m = q.shape
    dv = v.shape[-1]
    out = {n: np.zeros(s) for n, s in (("dq", q.shape), ("dk", q.shape), ("dv", v.shape),
                                       ("dbeta", beta.shape), ("dlambda", beta.shape),
                                       ("dS0", (BH, m, dv)), ("dx_prev", (BH, m)))}
    nch = -(-T // C)
    for b in range(BH):
        qf, kf = _phi(q[b], phi), _phi(k[b], phi)
        x = np.zeros((T, m))
        if T:
            x[1:] = kf[:-1]
        if x_prev is not None and T:
            x[0] = x_prev[b]
        E = (x * x).sum(-1)
        lam_e = lam[b] * E if ridge == "scaled" else lam[b].copy()
        den = E + lam_e + eps
        eta = np.where(den > 0, beta[b] / np.where(den > 0, den, 1.0), 0.0)
        if x_prev is None and T:
            eta[0] = 0.0
        a_raw = eta * lam_e
        clamped = a_raw >= 1 - eps_gamma
        gam = np.where(clamped, eps_gamma, 1 - a_raw)
        lg = np.log(gam)
        live = (den > 0) & ~((np.arange(T) == 0) & (x_prev is None))

        def pad(a, n, t0):
            z = np.zeros((C,) + a.shape[1:])
            z[:n] = a[t0:t0 + n]
            return z

        S = S0[b].copy() if S0 is not None else np.zeros((m, dv))
        chunks = []
        for c in range(nch):
            t0 = c * C
            n = min(C, T - t0)
            X, Q, V, et, l, dOc = (pad(a, n, t0) for a in (x, qf, v[b], eta, lg, dO[b]))
            g = np.cumsum(l)
            gx = g - l
            gC = g[-1]
            K = X @ X.T
            i, j = np.indices((C, C))
            A = np.where(j < i, et[:, None] * np.exp(np.minimum(gx[:, None] - g[None, :], 0))
                         * K, 0.0) if f1 else np.zeros((C, C))
            EP = np.where(j <= i, np.exp(np.minimum(g[:, None] - g[None, :], 0)), 0.0)
            P = EP * (Q @ X.T)
            R = et[:, None] * V
            if f1:
                R = R - (et * np.exp(gx))[:, None] * (X @ S)
            IA = np.eye(C) + A
            U = np.linalg.solve(IA, R)
            chunks.append(dict(t0=t0, n=n, X=X, Q=Q, V=V, et=et, g=g, gx=gx, gC=gC, K=K, A=A,
                               EP=EP, P=P, U=U, IA=IA, S=S.copy(), dO=dOc))
            # chunk map, as the forward applies it
            O = np.exp(g)[:, None] * (Q @ S) + P @ U
            S = np.exp(gC) * S + X.T @ (np.exp(gC - g)[:, None] * U)
            del O
        # reverse scan: cotangent of each chunk's leaving state
        dS = dS_T[b].copy() if dS_T is not None else np.zeros((m, dv))
        dX = np.zeros((T, m))
        dQ = np.zeros((T, m))
        for c in reversed(range(nch)):
            ch = chunks[c]
            X, Q, V, et, g, gx, gC = (ch[n] for n in ("X", "Q", "V", "et", "g", "gx", "gC"))
            A, EP, P, U, IA, Sc, dOc, K = (ch[n] for n in ("A", "EP", "P", "U", "IA", "S", "dO",
                                                        "K"))
            t0, n = ch["t0"], ch["n"]
            dSp = dS
            dU = P.T @ dOc + np.exp(gC - g)[:, None] * (X @ dSp)
            dR = np.linalg.solve(IA.T, dU)
            i, j = np.indices((C, C))
            dA = np.where(j < i, -(dR @ U.T), 0.0) if f1 else np.zeros((C, C))
            dP = np.where(j <= i, dOc @ U.T, 0.0)
            dV = et[:, None] * dR
            Y, Z, W2 = dR @ Sc.T, dOc @ Sc.T, U @ dSp.T
            deta = (dR * V).sum(-1)
            if f1:
                deta += -np.exp(gx) * (X * Y).sum(-1)
                deta += (dA * np.exp(np.minimum(gx[:, None] - g[None, :], 0)) * K).sum(-1)
            dg = np.exp(g) * (Q * Z).sum(-1)
            if f1:
                tb = -et * np.exp(gx) * (X * Y).sum(-1)
                dg[:-1] += tb[1:]
                dAA = dA * A
                dg[:-1] += dAA.sum(1)[1:]
                dg -= dAA.sum(0)
            dPP = dP * P
            dg += dPP.sum(1) - dPP.sum(0)
            cj = np.exp(gC - g) * (X * W2).sum(-1)
            dg[-1] += np.exp(gC) * (dSp * Sc).sum() + cj.sum()
            dg -= cj
            dlg = np.cumsum(dg[::-1])[::-1]
            dE = np.zeros(C)
            for r in range(n):
                t = t0 + r
                if not live[t]:
                    continue
                de, dl = deta[r], 0.0
                if not clamped[t]:
                    dal = -dlg[r] / gam[t]
                    de += lam_e[t] * dal
                    dl += eta[t] * dal
                out["dbeta"][b, t] = de / den[t]
                dden = -de * eta[t] / den[t]
                dE[r] = dden
                dl += dden
                if ridge == "scaled":
                    out["dlambda"][b, t] = dl * E[t]
                    dE[r] += dl * lam[b, t]
                else:
                    out["dlambda"][b, t] = dl
            dK = dA * et[:, None] * np.exp(np.minimum(gx[:, None] - g[None, :], 0))
            dXc = ((dP * EP).T @ Q + np.exp(gC - g)[:, None] * W2 + (dK + dK.T) @ X
                   + 2 * dE[:, None] * X)
            if f1:
                dXc -= (et * np.exp(gx))[:, None] * Y
            dQc = np.exp(g)[:, None] * Z + (dP * EP) @ X
            dX[t0:t0 + n] = dXc[:n]
            dQ[t0:t0 + n] = dQc[:n]
            out["dv"][b, t0:t0 + n] = dV[:n]
            # cotangent of the entering state: the transposed chunk map
            Mc_top = np.exp(gC) * np.eye(m)
            Mc_bot = np.exp(g)[:, None] * Q
            if f1:
                W = np.linalg.solve(IA, (et * np.exp(gx))[:, None] * X)
                Mc_top = Mc_top - X.T @ (np.exp(gC - g)[:, None] * W)
                Mc_bot = Mc_bot - P @ W
            dS = Mc_top.T @ dSp + Mc_bot.T @ dOc
        out["dS0"][b] = dS
        out["dq"][b] = _phi_vjp(q[b], dQ, phi)
        gk = np.zeros((T, m))
        if T:
            gk[:-1] = dX[1:]
            if dx_last is not None:
                gk[-1] = dx_last[b]
        out["dk"][b] = _phi_vjp(k[b], gk, phi)
        if x_prev is not None:
            out["dx_prev"][b] = dX[0] if T else dx_last[b]
    return out


def _case(seed, BH=2, T=37, m=6, dv=4, lam_shift=-1.5):
    g = np.random.default_rng(seed)
    return dict(
        q=g.standard_normal((BH, T, m)), k=g.standard_normal((BH, T, m)),
        v=g.standard_normal((BH, T, dv)),
        beta=2.0 / (1 + np.exp(-g.standard_normal((BH, T)))),
        lam=np.log1p(np.exp(g.standard_normal((BH, T)) + lam_shift)),
        dO=g.standard_normal((BH, T, dv)), S0=g.standard_normal((BH, m, dv)) * 0.5,
        x_prev=_phi(g.standard_normal((BH, m)), "l2"), dS_T=g.standard_normal((BH, m, dv)),
        dx_last=g.standard_normal((BH, m)))


def _compare(got, want, tol=1e-9):
    for name in want:
        scale = max(np.abs(want[name]).max(), 1e-12)
        err = np.abs(got[name] - want[name]).max() / scale
        assert err < tol, (name, err)


@pytest.mark.parametrize("rule", ["falcon1", "falcon1a"])
@pytest.mark.parametrize("C", [1, 4, 8, 16, 37, 64])
@pytest.mark.parametrize("carried", [False, True])
def test_chunk_backward_matches_oracle(rule, C, carried):
    c = _case(3 + C)
    kw = dict(S0=c["S0"], x_prev=c["x_prev"], dS_T=c["dS_T"], dx_last=c["dx_last"]) \
        if carried else {}
    want = oracle.backward(rule, c["q"], c["k"], c["v"], c["beta"], c["lam"], c["dO"], phi="l2",
                           threads=1, **kw)
    got = chunked_backward(rule, c["q"], c["k"], c["v"], c["beta"], c["lam"], c["dO"], C,
                           phi="l2", **kw)
    _compare(got, want)


@pytest.mark.parametrize("rule", ["falcon1", "falcon1a"])
@pytest.mark.parametrize("phi,ridge", [("identity", "given"), ("rms", "scaled"),
                                       ("l2", "scaled")])
def test_chunk_backward_variants_and_clamp(rule, phi, ridge):
    """Feature maps, the scale-coupled ridge, and a ridge large enough that
    many tokens take the clamped decay."""
    c = _case(9, T=29, lam_shift=2.0)
    kw = dict(S0=c["S0"], x_prev=c["x_prev"], dS_T=c["dS_T"], dx_last=c["dx_last"])
    want = oracle.backward(rule, c["q"], c["k"], c["v"], c["beta"], c["lam"], c["dO"], phi=phi,
                           ridge=ridge, threads=1, **kw)
    got = chunked_backward(rule, c["q"], c["k"], c["v"], c["beta"], c["lam"], c["dO"], 8,
                           phi=phi, ridge=ridge, **kw)
    _compare(got, want)
