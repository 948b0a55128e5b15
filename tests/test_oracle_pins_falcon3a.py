"""Pins of the Falcon-3A oracle (sliding-window inner-product rule; page
hyper.ai/fr/papers/2608.27763, Section 4.5, and its parallel (attention) form
of Section 4.6):

  - with a window of one pair the rule is Falcon-1A (Section 4.5: "for B = 1
    and t >= 2 ... reduces to the scalar non-sliding inner-product update");
  - the masked-attention form O = Diag(delta) Q S0 + (Q X^T o M) V with
    M_{t,j} = sum_{s=j}^{min(t, j+B-1)} (eta_s / B_s) prod_{r=s+1}^t gamma_r and
    delta_t = prod_{r<=t} gamma_r (Section 4.6), summed by brute force with the
    step sizes computed here from the window energies (the clamped decays
    enter the same products);
  - the scale-coupled ridge lambda_t = lambda_bar_t * E_bar_t (Section 4.5).
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


def _case(seed, BH=2, T=20, m=5, dv=3, lam_shift=-1.0):
    g = np.random.default_rng(seed)
    q = g.standard_normal((BH, T, m))
    k = g.standard_normal((BH, T, m))
    v = g.standard_normal((BH, T, dv))
    beta = 2.0 / (1 + np.exp(-g.standard_normal((BH, T))))
    lam = np.log1p(np.exp(g.standard_normal((BH, T)) + lam_shift))
    S0 = g.standard_normal((BH, m, dv)) * 0.3
    return q, k, v, beta, lam, S0


@pytest.mark.parametrize("phi", ["l2", "rms"])
def test_window_one_is_falcon1a(phi):
    q, k, v, beta, lam, S0 = _case(1)
    a = oracle.forward3a(q, k, v, beta, lam, 1, S0=S0, phi=phi)
    b = oracle.forward("falcon1a", q, k, v, beta, lam, S0=S0, phi=phi)
    for key in ("o", "S", "x_last"):
        np.testing.assert_allclose(a[key], b[key], rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("B", [2, 3, 7, 40])
@pytest.mark.parametrize("lam_shift", [-30.0, -1.0, 2.5])
@pytest.mark.parametrize("phi", ["identity", "l2"])
def test_masked_attention_form(B, lam_shift, phi):
    q, k, v, beta, lam, S0 = _case(7 + B, lam_shift=lam_shift)
    eps, eg = 1e-6, 1e-6
    BH, T, dv = v.shape
    kf, qf = _phi(k, phi), _phi(q, phi)
    x = np.zeros_like(kf)
    x[:, 1:] = kf[:, :-1]  # x_1 = 0, x_t = phi(k_{t-1})
    # per step s (0-based; s = 0 is the boundary): window, B_s, E_bar, eta, gamma
    eta = np.zeros((BH, T))
    gam = np.ones((BH, T))
    Bs = np.ones(T)
    for s in range(1, T):
        j0 = max(1, s - B + 1)
        Bs[s] = s - j0 + 1
        Ebar = (x[:, j0:s + 1] ** 2).sum((-1, -2)) / Bs[s]
        den = Ebar + lam[:, s] + eps
        eta[:, s] = beta[:, s] / den
        gam[:, s] = 1.0 - np.minimum(eta[:, s] * lam[:, s], 1.0 - eg)
    want = np.zeros((BH, T, dv))
    for b in range(BH):
        for t in range(T):
            delta = np.prod(gam[b, :t + 1])
            acc = delta * (qf[b, t] @ S0[b])
            for j in range(1, t + 1):
                M = 0.0
                for s in range(j, min(t, j + B - 1) + 1):
                    M += eta[b, s] / Bs[s] * np.prod(gam[b, s + 1:t + 1])
                acc = acc + M * (qf[b, t] @ x[b, j]) * v[b, j]
            want[b, t] = acc
    # The final state in the same form: S_T = delta_T S0 + sum_j M_{T,j} x_j v_j^T,
    # the mask row of the last token (the read o_T = S_T^T phi(q_T) pins it only
    # along phi(q_T)).
    want_S = np.zeros((BH,) + S0.shape[1:])
    for b in range(BH):
        t = T - 1
        acc = np.prod(gam[b, :t + 1]) * S0[b]
        for j in range(1, t + 1):
            M = 0.0
            for s in range(j, min(t, j + B - 1) + 1):
                M += eta[b, s] / Bs[s] * np.prod(gam[b, s + 1:t + 1])
            acc = acc + M * np.outer(x[b, j], v[b, j])
        want_S[b] = acc
    got = oracle.forward3a(q, k, v, beta, lam, B, S0=S0, phi=phi, eps=eps, eps_gamma=eg)
    np.testing.assert_allclose(got["o"], want, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(got["S"], want_S, rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("B", [1, 4])
def test_scale_coupled_ridge_uses_window_energy(B):
    q, k, v, beta, lbar, S0 = _case(21, lam_shift=0.5)
    T = q.shape[1]
    x = np.zeros_like(k)
    x[:, 1:] = _phi(k, "l2")[:, :-1]
    lam_eff = np.zeros_like(lbar)
    for s in range(1, T):
        j0 = max(1, s - B + 1)
        lam_eff[:, s] = lbar[:, s] * (x[:, j0:s + 1] ** 2).sum((-1, -2)) / (s - j0 + 1)
    a = oracle.forward3a(q, k, v, beta, lbar, B, S0=S0, phi="l2", ridge="scaled")
    b = oracle.forward3a(q, k, v, beta, lam_eff, B, S0=S0, phi="l2", ridge="given")
    for key in ("o", "S"):
        np.testing.assert_allclose(a[key], b[key], rtol=1e-12, atol=1e-12)
