"""Pins of the oracle's normalised read (Falcon-1A with a normaliser z).

Page hyper.ai/fr/papers/2608.27763, Section 2.2: Eq. (2.1) is normalised
linear attention, Eq. (2.2) its recurrent form with the normaliser z_t, and
Eq. (2.3) the same on the shifted write stream x_1 = 0, x_t = phi(k_{t-1}):

    o_t = S_t^T phi(q_t) / (z_t^T phi(q_t) + eps_attn),
    S_t = S_{t-1} + x_t v_t^T,   z_t = z_{t-1} + x_t.

The Falcon-1A version is deferred to an appendix the pages do not include;
the reading taken gives z the numerator's gain and clamped decay,
z_t = gamma_t z_{t-1} + eta_t x_t, which at lambda = 0 and unit gain is
Eq. (2.3) exactly.  The pins:
  * Eq. (2.3) summed by brute force over all pairs (fresh and carried state);
  * with decay and the clamp active: the numerator is the Falcon-1A read and
    the denominator is the Falcon-1A read of a constant unit target (z is the
    state column such a target writes), both from the separately pinned
    Falcon-1A oracle;
  * split-run continuation with (S, z, x_prev) carried.
"""
import numpy as np
import pytest

import oracle


def _positive_case(seed, BH=3, T=40, m=8, dv=5, lam_shift=None):
    rng = np.random.default_rng(seed)
    # positive features keep the denominators away from zero (the pages note the
    # normalised read is attention-like only for a nonnegative normaliser)
    q = np.abs(rng.standard_normal((BH, T, m))) + 0.05
    k = np.abs(rng.standard_normal((BH, T, m))) + 0.05
    v = rng.standard_normal((BH, T, dv))
    if lam_shift is None:
        lam = np.zeros((BH, T))
        beta = np.full((BH, T), 1.0 + 1e-6)  # eta = 1 for unit-norm features, eps = 1e-6
    else:
        beta = 2.0 / (1.0 + np.exp(-rng.standard_normal((BH, T))))
        lam = np.log1p(np.exp(rng.standard_normal((BH, T)) + lam_shift))
    return q, k, v, beta, lam


def _unit(u):
    return u / np.linalg.norm(u, axis=-1, keepdims=True)


@pytest.mark.parametrize("carried", [False, True])
@pytest.mark.parametrize("eps_attn", [0.0, 1e-3])
def test_shifted_normalised_linear_attention_brute_force(carried, eps_attn):
    """lambda = 0, eta = 1 (l2 features, beta = 1 + eps): Eq. (2.3) by O(T^2) sums."""
    q, k, v, beta, lam = _positive_case(3 + int(carried))
    BH, T, m = q.shape
    dv = v.shape[-1]
    rng = np.random.default_rng(99)
    S0 = np.abs(rng.standard_normal((BH, m, dv))) if carried else None
    z0 = np.abs(rng.standard_normal((BH, m))) + 0.1 if carried else None
    x_prev = _unit(np.abs(rng.standard_normal((BH, m))) + 0.05) if carried else None
    qf, kf = _unit(q), _unit(k)
    want = np.zeros((BH, T, dv))
    for b in range(BH):
        xs = np.zeros((T, m))  # the shifted write stream
        xs[1:] = kf[b, :-1]
        if carried:
            xs[0] = x_prev[b]
        for t in range(T):
            num = np.zeros(dv) if S0 is None else S0[b].T @ qf[b, t]
            den = 0.0 if z0 is None else z0[b] @ qf[b, t]
            for j in range(t + 1):
                w = qf[b, t] @ xs[j]
                num = num + w * v[b, j]
                den += w
            want[b, t] = num / (den + eps_attn) if (den + eps_attn) != 0 else 0.0
    got = oracle.forward_normalized(q, k, v, beta, lam, S0=S0, z0=z0, x_prev=x_prev, phi="l2",
                                    eps=1e-6, eps_gamma=1e-6, eps_attn=eps_attn)
    if not carried:
        # token 1: x_1 = 0 and z_1 = 0, so o_1 = 0 / eps_attn (0 when eps_attn = 0
        # gives 0/0: only compare t >= 2 there)
        t0 = 0 if eps_attn > 0 else 1
        np.testing.assert_allclose(got["o"][:, t0:], want[:, t0:], rtol=1e-10, atol=1e-12)
    else:
        np.testing.assert_allclose(got["o"], want, rtol=1e-10, atol=1e-12)
    # the normaliser is the sum of the written features (plus z0)
    z_want = (np.zeros((BH, m)) if z0 is None else z0) + kf[:, :-1].sum(1)
    if carried:
        z_want = z_want + x_prev
    np.testing.assert_allclose(got["z"], z_want, rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("phi", ["l2", "rms", "identity"])
@pytest.mark.parametrize("lam_shift", [-2.0, 1.5])
def test_decayed_read_is_ratio_of_falcon1a_reads(phi, lam_shift):
    """With decay (lambda_shift 1.5 makes the clamp fire), the numerator is the
    Falcon-1A read and the denominator the Falcon-1A read of a unit target."""
    q, k, v, beta, lam = _positive_case(11, lam_shift=lam_shift)
    BH, T, m = q.shape
    rng = np.random.default_rng(5)
    S0 = rng.standard_normal((BH, m, v.shape[-1]))
    z0 = np.abs(rng.standard_normal((BH, m)))
    x_prev = _unit(np.abs(rng.standard_normal((BH, m))))
    eps_attn = 1e-4
    got = oracle.forward_normalized(q, k, v, beta, lam, S0=S0, z0=z0, x_prev=x_prev, phi=phi,
                                    eps_attn=eps_attn)
    num = oracle.forward("falcon1a", q, k, v, beta, lam, S0=S0, x_prev=x_prev, phi=phi)
    ones = np.ones((BH, T, 1))
    den = oracle.forward("falcon1a", q, k, ones, beta, lam, S0=z0[..., None], x_prev=x_prev,
                         phi=phi)
    np.testing.assert_allclose(got["o"], num["o"] / (den["o"] + eps_attn), rtol=1e-11,
                               atol=1e-13)
    np.testing.assert_allclose(got["S"], num["S"], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(got["z"], den["S"][..., 0], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(got["x_last"], num["x_last"], rtol=0, atol=0)
    if lam_shift > 0:  # the clamp really fires in this draw
        kf = _unit(k)
        xs = np.concatenate([x_prev[:, None], kf[:, :-1]], 1)
        eta = beta / ((xs ** 2).sum(-1) + lam + 1e-6)
        assert (eta * lam >= 1 - 1e-6).any()


def test_split_run_continuation():
    """Carrying (S, z, x_prev) across two calls equals one call."""
    q, k, v, beta, lam = _positive_case(21, T=50, lam_shift=-1.0)
    full = oracle.forward_normalized(q, k, v, beta, lam, phi="l2", eps_attn=1e-3)
    for T1 in (1, 17, 49):
        a = oracle.forward_normalized(q[:, :T1], k[:, :T1], v[:, :T1], beta[:, :T1],
                                      lam[:, :T1], phi="l2", eps_attn=1e-3)
        b = oracle.forward_normalized(q[:, T1:], k[:, T1:], v[:, T1:], beta[:, T1:],
                                      lam[:, T1:], S0=a["S"], z0=a["z"], x_prev=a["x_last"],
                                      phi="l2", eps_attn=1e-3)
        np.testing.assert_allclose(np.concatenate([a["o"], b["o"]], 1), full["o"], rtol=1e-12,
                                   atol=1e-13)
        np.testing.assert_allclose(b["S"], full["S"], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(b["z"], full["z"], rtol=1e-12, atol=1e-13)
