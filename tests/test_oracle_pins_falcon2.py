"""Pins of the Falcon-2 / Falcon-2A oracle (per-column step sizes).

Passages (p1 = hyper.ai/fr/papers/2608.27763): the regression-family display
of Section 3.1 (Falcon-2: S_t = S_{t-1}(I - lambda_t Diag(eta_t)) +
x_t (eta_t o r_t)^T, eta_{j,t} = beta_{j,t} / (||x_t||^2 + lambda_t + eps)),
the "Per-column NLMS step sizes" paragraph of Section 4.2 (tied gains reduce
to the scalar rule; the loss separates over the columns of S, so Falcon-2 is
d_v independent scalar-step updates), Section 4.3 "Falcon-2A: per-column
inner-product write" and the Falcon-1A/Falcon-2A step sizes (E_t = ||x_t||^2;
the clamp acts per column).  None of the tests re-types the oracle's token
loop: they use the Falcon-1 oracle on single columns, the gradient of the
printed per-column loss by autograd, closed-form interpolation, and the
masked-parallel (attention) form of the inner-product rule summed by brute
force.
"""
import numpy as np
import pytest
import torch

import oracle

from test_oracle_pins import _eta_gamma, _phi, _write_features


def _case2(seed, BH=2, T=20, m=5, dv=4, lam_shift=-2.0):
    g = np.random.default_rng(seed)
    q = g.standard_normal((BH, T, m))
    k = g.standard_normal((BH, T, m))
    v = g.standard_normal((BH, T, dv))
    beta = 2.0 / (1 + np.exp(-g.standard_normal((BH, T, dv))))  # one gain per column
    lam = np.log1p(np.exp(g.standard_normal((BH, T)) + lam_shift))
    return q, k, v, beta, lam


@pytest.mark.parametrize("rule2,rule1", [("falcon2", "falcon1"), ("falcon2a", "falcon1a")])
def test_tied_gains_reduce_to_scalar_rule(rule2, rule1):
    """p1 Section 4.2: with beta_{j,t} = beta_t for every column the per-column
    step size is the scalar NLMS step, so Falcon-2(A) is Falcon-1(A)."""
    q, k, v, beta, lam = _case2(1)
    b1 = beta[..., 0]
    tied = np.repeat(b1[..., None], v.shape[-1], axis=-1)
    S0 = np.random.default_rng(2).standard_normal((2, 5, 4)) * 0.3
    a = oracle.forward2(rule2, q, k, v, tied, lam, S0=S0, phi="l2")
    b = oracle.forward(rule1, q, k, v, b1, lam, S0=S0, phi="l2")
    for key in ("o", "S", "x_last"):
        np.testing.assert_allclose(a[key], b[key], rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("rule2,rule1", [("falcon2", "falcon1"), ("falcon2a", "falcon1a")])
@pytest.mark.parametrize("lam_shift", [-2.0, 1.5])
def test_columns_are_independent_scalar_updates(rule2, rule1, lam_shift):
    """p1 Section 4.2: Falcon-2 is a collection of d_v independent scalar-step
    updates sharing x_t and lambda_t: column j equals the scalar rule run on
    value channel j alone with gain beta_{j,t} (lam_shift 1.5 clamps some
    columns and not others)."""
    q, k, v, beta, lam = _case2(3, lam_shift=lam_shift)
    S0 = np.random.default_rng(4).standard_normal((2, 5, 4)) * 0.3
    xp = _phi(np.random.default_rng(5).standard_normal((2, 5)), "l2")
    full = oracle.forward2(rule2, q, k, v, beta, lam, S0=S0, x_prev=xp, phi="l2")
    for j in range(v.shape[-1]):
        col = oracle.forward(rule1, q, k, v[..., j:j + 1], beta[..., j], lam,
                             S0=S0[..., j:j + 1], x_prev=xp, phi="l2")
        np.testing.assert_allclose(full["o"][..., j:j + 1], col["o"], rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(full["S"][..., j:j + 1], col["S"], rtol=1e-11, atol=1e-12)


def test_falcon2_step_is_columnwise_gradient_step():
    """p1 Section 3.1 / 4.2: each column takes a gradient step of the ridge
    loss l(S) = 1/2 ||y - S^T x||^2 + lambda/2 ||S||^2 with its own step eta_j,
    i.e. S_t = S_{t-1} - grad l(S_{t-1}) Diag(eta_t) (unclamped case)."""
    g = np.random.default_rng(7)
    m, dv = 6, 5
    for trial in range(5):
        S = g.standard_normal((m, dv))
        x = _phi(g.standard_normal(m), "l2")
        y = g.standard_normal(dv)
        beta = g.uniform(0.1, 1.9, dv)
        lam = float(g.uniform(0.0, 0.5))
        eps = 1e-6
        eta = beta / (x @ x + lam + eps)  # the printed per-column step size
        St = torch.tensor(S, requires_grad=True)
        xt, yt = torch.tensor(x), torch.tensor(y)
        loss = 0.5 * ((yt - St.T @ xt) ** 2).sum() + 0.5 * lam * (St ** 2).sum()
        loss.backward()
        want = S - St.grad.numpy() * eta[None, :]
        # one token through the oracle: x_1 = x (carried), y_1 = y
        out = oracle.forward2("falcon2", np.zeros((1, 1, m)), np.zeros((1, 1, m)), y[None, None],
                              beta[None, None], np.array([[lam]]), S0=S[None], x_prev=x[None],
                              phi="identity", eps=eps)
        np.testing.assert_allclose(out["S"][0], want, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("phi", ["identity", "l2"])
def test_falcon2_nlms_interpolation(phi):
    """p1 Section 3.1: with lambda = 0, eps = 0 and unit gains the NLMS step
    interpolates: S_t^T x_t = v_t for every t >= 2, in every column."""
    q, k, v, beta, lam = _case2(11, T=12)
    out_S = []
    xs = _write_features(k, phi)
    ones = np.ones_like(beta)
    S = None
    for t in range(1, 12):
        r = oracle.forward2("falcon2", q[:, :t + 1], k[:, :t + 1], v[:, :t + 1], ones[:, :t + 1],
                            np.zeros((2, t + 1)), phi=phi, eps=0.0)
        pred = np.einsum("bmd,bm->bd", r["S"], xs[:, t])
        np.testing.assert_allclose(pred, v[:, t], rtol=1e-9, atol=1e-9)


@pytest.mark.parametrize("phi", ["identity", "l2"])
@pytest.mark.parametrize("lam_shift", [-30.0, -1.0, 2.0])
def test_falcon2a_masked_parallel_form(phi, lam_shift):
    """p1 Section 4.3 (Falcon-2A) unrolled: S_t[:, j] = sum_{s<=t}
    (prod_{r=s+1..t} gamma_{j,r}) eta_{j,s} x_s v_{s,j}, read o_t = S_t^T phi(q_t):
    a per-column decayed linear attention, summed here by brute force with
    gamma_{j,r} = 1 - min(eta_{j,r} lambda_r, 1 - eps_gamma).  lam_shift -30
    is the additive (lambda ~ 0) case; 2.0 clamps some columns."""
    q, k, v, beta, lam = _case2(21, T=16, lam_shift=lam_shift)
    eps, eg = 1e-6, 1e-6
    x = _write_features(k, phi)
    qf = _phi(q, phi)
    BH, T, dv = v.shape
    # per-column step sizes and decays (E_t = ||x_t||^2, sentinel at t = 1)
    den = (x * x).sum(-1) + lam + eps
    eta = beta / den[..., None]
    eta[:, 0, :] = 0.0
    gam = 1.0 - np.minimum(eta * lam[..., None], 1.0 - eg)
    want = np.zeros((BH, T, dv))
    for b in range(BH):
        for t in range(T):
            for j in range(dv):
                acc = 0.0
                for s in range(t + 1):
                    dec = np.prod(gam[b, s + 1:t + 1, j])
                    acc += dec * eta[b, s, j] * (qf[b, t] @ x[b, s]) * v[b, s, j]
                want[b, t, j] = acc
    got = oracle.forward2("falcon2a", q, k, v, beta, lam, phi=phi, eps=eps, eps_gamma=eg)
    np.testing.assert_allclose(got["o"], want, rtol=1e-10, atol=1e-12)


def test_falcon2_first_token_does_not_write():
    """p1 Section 3 boundary: eta_{j,1} = 0 for all j, so with S0 = 0 the first
    output is zero whatever beta and lambda are."""
    q, k, v, beta, lam = _case2(31, T=3)
    beta[:, 0, :] = 1.9
    lam[:, 0] = 5.0
    for rule in ("falcon2", "falcon2a"):
        out = oracle.forward2(rule, q, k, v, beta, lam, phi="l2")
        np.testing.assert_array_equal(out["o"][:, 0], 0.0)
