"""fp64 check of the Falcon-2 chunk forms (the blocked decayed-accumulator
form, and the factored form the CUDA kernel implements).

This is neither the oracle nor the CUDA path: it restates, in numpy, the
chunk algebra derived from the per-column Falcon-2 update (page
hyper.ai/fr/papers/2608.27763, the regression-family display of Section 3.1
with the per-column NLMS step sizes of Section 4.2: every value column j runs
its own scalar-step delta rule, sharing the write features x_t) and checks it
against the oracle before any kernel relies on it.

Per column j, inside a chunk entered with state S (local tokens i), the
written residual u_{ij} = eta_{ij} r_{ij} solves a unit-lower system whose
off-diagonal part is the shared Gram K_{il} = <x_i, x_l> scaled by the
column's decay products.  No exponential is taken: every decay enters as a
product of the gammas themselves (each in (0, 1]), so nothing overflows when
decays are strong or clamped.  With the accumulator
    acc^{(i)}_t = e^{G_i} (X S)_t + sum_{l<=i} e^{G_i - G_l} K_{tl} u_l,
(e^{G_i} the product of gamma over the chunk's tokens up to i) the row-t
residual is v_t - acc^{(t-1)}_t, and acc^{(i)} = gamma_i acc^{(i-1)} +
K_{.,i} u_i.  The chunk is cut into blocks of `blk` rows: inside a block the
accumulators run token by token; across blocks the contribution of earlier
blocks is a shared-matrix product K_{b,b'} U~^{[b']}, with U~^{[b']}_l the
u_l decayed to the end of block b', combined in Horner order with the block
decays.  The output and the state leaving the chunk follow the same way:
    o_{tj}   = e^{G_t} (Q S)_{tj} + sum_{l<=t} e^{G_t - G_l} <q_t, x_l> u_{lj}
    S'_{:,j} = e^{G_C} S_{:,j} + sum_l x_l e^{G_C - G_l} u_{lj}.
"""
import numpy as np
import pytest

import oracle


def _phi(u, phi):
    if phi == "identity":
        return u
    return u / np.maximum(np.linalg.norm(u, axis=-1, keepdims=True), 1e-12)


def chunked_forward2(q, k, v, beta, lam, C=64, blk=16, S0=None, x_prev=None, phi="l2",
                     eps=1e-6, eps_gamma=1e-6):
    BH, T, m = q.shape
    dv = v.shape[-1]
    Q, Kf = _phi(q, phi), _phi(k, phi)
    o = np.zeros((BH, T, dv))
    S_out = np.zeros((BH, m, dv))
    for h in range(BH):
        S = np.zeros((m, dv)) if S0 is None else S0[h].copy()
        xp = None if x_prev is None else x_prev[h]
        for c0 in range(0, T, C):
            n = min(C, T - c0)
            # Chunk rows padded to C: tokens past T write nothing (eta = 0,
            # gamma = 1) and read nothing (q = 0).
            X = np.zeros((C, m))
            Qc = np.zeros((C, m))
            V = np.zeros((C, dv))
            eta = np.zeros((C, dv))
            gam = np.ones((C, dv))
            for i in range(n):
                t = c0 + i
                if t > 0:
                    X[i] = Kf[h, t - 1]
                elif xp is not None:
                    X[i] = xp
                Qc[i] = Q[h, t]
                V[i] = v[h, t]
                sentinel = t == 0 and xp is None
                den = X[i] @ X[i] + lam[h, t] + eps
                e = np.zeros(dv) if (sentinel or den <= 0) else beta[h, t] / den
                a = e * lam[h, t]
                eta[i] = e
                gam[i] = np.where(a >= 1 - eps_gamma, eps_gamma, 1 - a)
            Kg = X @ X.T
            P0 = Qc @ X.T
            XS, QS = X @ S, Qc @ S
            nb = C // blk
            U = np.zeros((C, dv))
            Ut = []          # U~^{[b]}: u decayed to the end of block b
            Dblk = []        # product of gamma over block b (per column)
            Pc = np.ones(dv)  # product of gamma over the blocks before b
            for b in range(nb):
                s = b * blk
                rows = slice(s, s + blk)
                # Horner over the earlier blocks (K and P0 share the operands)
                RK = np.zeros((blk, dv))
                RP = np.zeros((blk, dv))
                for bp in range(b):
                    src = slice(bp * blk, bp * blk + blk)
                    RK = Dblk[bp] * RK + Kg[rows, src] @ Ut[bp]
                    RP = Dblk[bp] * RP + P0[rows, src] @ Ut[bp]
                acc = Pc * XS[rows] + RK
                ao = Pc * QS[rows] + RP
                for i in range(blk):
                    U[s + i] = eta[s + i] * (V[s + i] - acc[i])
                    acc[i + 1:] = gam[s + i] * acc[i + 1:] + np.outer(Kg[s + i + 1:s + blk, s + i],
                                                                     U[s + i])
                    ao[i:] = gam[s + i] * ao[i:] + np.outer(P0[s + i:s + blk, s + i], U[s + i])
                    if c0 + s + i < T:
                        o[h, c0 + s + i] = ao[i]
                d = np.ones(dv)
                ut = np.zeros((blk, dv))
                for i in reversed(range(blk)):
                    ut[i] = d * U[s + i]
                    d = d * gam[s + i]
                Ut.append(ut)
                Dblk.append(d)
                Pc = Pc * d
            dec = np.ones(dv)
            inc = np.zeros((C, dv))
            for i in reversed(range(C)):
                inc[i] = dec * U[i]
                dec = dec * gam[i]
            S = dec * S + X.T @ inc
        S_out[h] = S
    return o, S_out


def factored_forward2(q, k, v, beta, lam, C=64, blk=16, S0=None, x_prev=None, phi="l2",
                      eps=1e-6, eps_gamma=1e-6, min_decay=np.exp(-60.0)):
    """The form the tensor-core kernel runs.  With E_t the product of a
    column's gammas over the chunk up to token t (E_{-1} = 1) and w = u / E:
      u_t = eta_t v_t - eta_t E_{t-1} ((X S)_t + sum_{l<t} K_{tl} w_l)
      o_t = E_t ((Q S)_t + sum_{l<=t} <q_t, x_l> w_l),   S' = E_C (S + X^T W)
    (e^{G_t - G_l} = E_t / E_l).  Inside a block of `blk` rows the u run token
    by token; the rows before the block enter as one product K_{b,<b} W_{<b}.
    A chunk whose decay product falls below `min_decay` in some column runs
    the tokens one by one (the factors 1 / E would leave the fp32 range)."""
    BH, T, m = q.shape
    dv = v.shape[-1]
    Q, Kf = _phi(q, phi), _phi(k, phi)
    o = np.zeros((BH, T, dv))
    S_out = np.zeros((BH, m, dv))
    n_tokenwise = 0
    for h in range(BH):
        S = np.zeros((m, dv)) if S0 is None else S0[h].copy()
        xp = None if x_prev is None else x_prev[h]
        for c0 in range(0, T, C):
            n = min(C, T - c0)
            X = np.zeros((C, m))
            Qc = np.zeros((C, m))
            V = np.zeros((C, dv))
            eta = np.zeros((C, dv))
            gam = np.ones((C, dv))
            for i in range(n):
                t = c0 + i
                if t > 0:
                    X[i] = Kf[h, t - 1]
                elif xp is not None:
                    X[i] = xp
                Qc[i] = Q[h, t]
                V[i] = v[h, t]
                sentinel = t == 0 and xp is None
                den = X[i] @ X[i] + lam[h, t] + eps
                e = np.zeros(dv) if (sentinel or den <= 0) else beta[h, t] / den
                a = e * lam[h, t]
                eta[i] = e
                gam[i] = np.where(a >= 1 - eps_gamma, eps_gamma, 1 - a)
            E = np.cumprod(gam, axis=0)
            if (E[-1] < min_decay).any():
                n_tokenwise += 1
                for i in range(n):
                    u = eta[i] * (V[i] - X[i] @ S)
                    S = gam[i] * S + np.outer(X[i], u)
                    o[h, c0 + i] = Qc[i] @ S
                continue
            Eprev = np.vstack([np.ones((1, dv)), E[:-1]])
            Kg = X @ X.T
            P0 = np.tril(Qc @ X.T)
            XS, QS = X @ S, Qc @ S
            W = np.zeros((C, dv))
            for b in range(C // blk):
                s = b * blk
                acc = XS[s:s + blk] + Kg[s:s + blk, :s] @ W[:s]
                for i in range(blk):
                    u = eta[s + i] * V[s + i] - eta[s + i] * Eprev[s + i] * acc[i]
                    W[s + i] = u / E[s + i]
                    acc[i + 1:] += np.outer(Kg[s + i + 1:s + blk, s + i], W[s + i])
            O = E * (QS + P0 @ W)
            o[h, c0:c0 + n] = O[:n]
            S = E[-1] * (S + X.T @ W)
        S_out[h] = S
    return o, S_out, n_tokenwise


def _case(seed, BH, T, m, dv, lam_shift=-2.0, carried=False, x_prev=False):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((BH, T, m))
    k = rng.standard_normal((BH, T, m))
    v = rng.standard_normal((BH, T, dv))
    beta = 2.0 / (1.0 + np.exp(-rng.standard_normal((BH, T, dv))))
    lam = np.log1p(np.exp(rng.standard_normal((BH, T)) + lam_shift))
    S0 = 0.5 * rng.standard_normal((BH, m, dv)) if carried else None
    xp = None
    if x_prev:
        xp = rng.standard_normal((BH, m))
        xp /= np.linalg.norm(xp, axis=-1, keepdims=True)
    return q, k, v, beta, lam, S0, xp


@pytest.mark.parametrize("C,blk", [(64, 16), (64, 8), (32, 16), (16, 4), (64, 64)])
@pytest.mark.parametrize("T", [1, 37, 64, 150])
@pytest.mark.parametrize("carried", [False, True])
def test_blocked_chunk_form_matches_oracle(C, blk, T, carried):
    q, k, v, beta, lam, S0, xp = _case(7 + T + C, 2, T, 16, 12, carried=carried, x_prev=carried)
    o, S = chunked_forward2(q, k, v, beta, lam, C=C, blk=blk, S0=S0, x_prev=xp)
    ref = oracle.forward2("falcon2", q, k, v, beta, lam, S0=S0, x_prev=xp)
    np.testing.assert_allclose(o, ref["o"], rtol=1e-9, atol=1e-10)
    np.testing.assert_allclose(S, ref["S"], rtol=1e-9, atol=1e-10)


@pytest.mark.parametrize("phi", ["identity", "l2"])
def test_blocked_chunk_form_clamped_and_strong_decay(phi):
    """lambda = softplus(n + 3): the clamp fires on some (token, column) pairs
    (gamma = eps_gamma), so decay products inside a chunk underflow; the form
    uses products of gammas only, so it stays finite and exact."""
    q, k, v, beta, lam, S0, _ = _case(3, 2, 200, 16, 8, lam_shift=3.0, carried=True)
    o, S = chunked_forward2(q, k, v, beta, lam, C=64, blk=16, S0=S0, phi=phi)
    ref = oracle.forward2("falcon2", q, k, v, beta, lam, S0=S0, phi=phi)
    eta_lam = beta * (lam[..., None] / (1.0 + lam[..., None]))
    assert (eta_lam >= 1 - 1e-6).any() or phi == "identity"
    assert np.isfinite(o).all() and np.isfinite(S).all()
    np.testing.assert_allclose(o, ref["o"], rtol=1e-8, atol=1e-10)
    np.testing.assert_allclose(S, ref["S"], rtol=1e-8, atol=1e-10)


def test_blocked_chunk_form_tied_gains_is_falcon1():
    """One gain for every column: the form reduces to Falcon-1 (Section 4.2)."""
    q, k, v, beta, lam, S0, xp = _case(11, 2, 100, 16, 16, carried=True, x_prev=True)
    beta1 = beta[..., 0]
    tied = np.repeat(beta1[..., None], 16, axis=-1)
    o, S = chunked_forward2(q, k, v, tied, lam, S0=S0, x_prev=xp)
    ref = oracle.forward("falcon1", q, k, v, beta1, lam, S0=S0, x_prev=xp)
    np.testing.assert_allclose(o, ref["o"], rtol=1e-9, atol=1e-10)
    np.testing.assert_allclose(S, ref["S"], rtol=1e-9, atol=1e-10)


@pytest.mark.parametrize("T", [1, 37, 64, 150])
@pytest.mark.parametrize("carried", [False, True])
def test_factored_chunk_form_matches_oracle(T, carried):
    q, k, v, beta, lam, S0, xp = _case(23 + T, 2, T, 16, 12, carried=carried, x_prev=carried)
    o, S, nt = factored_forward2(q, k, v, beta, lam, S0=S0, x_prev=xp)
    assert nt == 0
    ref = oracle.forward2("falcon2", q, k, v, beta, lam, S0=S0, x_prev=xp)
    np.testing.assert_allclose(o, ref["o"], rtol=1e-9, atol=1e-10)
    np.testing.assert_allclose(S, ref["S"], rtol=1e-9, atol=1e-10)


def test_factored_chunk_form_strong_decay_runs_token_by_token():
    """lambda = softplus(n + 3): clamped gammas push some chunks' decay
    products below e^{-60}; those chunks take the token loop, the others the
    factored form, and the result is the oracle's."""
    q, k, v, beta, lam, S0, _ = _case(5, 2, 300, 16, 8, lam_shift=3.0, carried=True)
    o, S, nt = factored_forward2(q, k, v, beta, lam, S0=S0)
    assert nt > 0
    ref = oracle.forward2("falcon2", q, k, v, beta, lam, S0=S0)
    assert np.isfinite(o).all() and np.isfinite(S).all()
    np.testing.assert_allclose(o, ref["o"], rtol=1e-8, atol=1e-10)
    np.testing.assert_allclose(S, ref["S"], rtol=1e-8, atol=1e-10)
