"""Pins of the fp64 oracle against what the pages and the mathematics fix.

Each test states the passage it follows.  None of them re-types the oracle's
token loop: they use closed forms worked by hand (tests/golden/), the gradient
of the printed loss taken by autograd, the masked-parallel (attention) forms
solved with a library linear solve, brute-force O(T^2) sums, and invariants
(linearity, scale invariance of the l2 feature map, continuation).

Page names: p1 = hyper.ai/fr/papers/2608.27763, p3 = juhoplayground.github.io
(Korean blog post), p4 = rcap.io/posts/fast-weight-attention-... .
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng_seed = 1234


def _rand_case(seed, BH=3, T=24, m=5, dv=3, lam_shift=-2.0, beta_scale=2.0):
    g = np.random.default_rng(seed)
    q = g.standard_normal((BH, T, m))
    k = g.standard_normal((BH, T, m))
    v = g.standard_normal((BH, T, dv))
    beta = beta_scale / (1 + np.exp(-g.standard_normal((BH, T))))
    lam = np.log1p(np.exp(g.standard_normal((BH, T)) + lam_shift))
    return q, k, v, beta, lam


def _phi(u, phi):
    if phi == "identity":
        return u
    return u / np.maximum(np.linalg.norm(u, axis=-1, keepdims=True), 1e-12)


def _write_features(k, phi, x_prev=None):
    """x_1 = 0 (or x_prev), x_t = phi(k_{t-1})  -- p1 Section 2.2 Eq. (2.3)."""
    kf = _phi(k, phi)
    x = np.zeros_like(kf)
    x[..., 1:, :] = kf[..., :-1, :]
    if x_prev is not None:
        x[..., 0, :] = x_prev
    return x


def _eta_gamma(x, beta, lam, eps, eps_gamma, sentinel=True):
    """eta from p1 Eq. (3.4) (0 at the sentinel t = 1 and when the denominator
    vanishes) and gamma = 1 - min(eta*lambda, 1 - eps_gamma) (p1 Section 4.3,
    'Decay positivity')."""
    den = (x * x).sum(-1) + lam + eps
    eta = np.where(den > 0, beta / np.where(den > 0, den, 1.0), 0.0)
    if sentinel:
        eta[..., 0] = 0.0
    alpha = np.minimum(eta * lam, 1.0 - eps_gamma)
    return eta, 1.0 - alpha


# --------------------------------------------------------------------------
# Golden fixtures worked by hand.
# --------------------------------------------------------------------------

def test_golden_constant_pair():
    """Hand-derived constant-pair sequence (tests/golden/constant_pair.json):
    sentinel at t = 1, geometric approach of Falcon-1 to the ridge solution
    x v^T / (||x||^2 + lambda), geometric accumulation for Falcon-1A."""
    fx = json.load(open(os.path.join(GOLDEN, "constant_pair.json")))
    inp = fx["inputs"]
    arr = {n: np.array(inp[n], dtype=np.float64)[None] for n in ("q", "k", "v", "beta", "lambda")}
    for rule in ("falcon1", "falcon1a"):
        out = oracle.forward(rule, arr["q"], arr["k"], arr["v"], arr["beta"], arr["lambda"],
                             phi=inp["phi"], eps=inp["eps"], eps_gamma=inp["eps_gamma"])
        exp = fx[rule]
        np.testing.assert_array_equal(out["o"][0], np.array(exp["o"]))
        np.testing.assert_array_equal(out["S"][0], np.array(exp["S"]))
        np.testing.assert_array_equal(out["x_last"][0], np.array(exp["x_last"]))


def test_golden_clamp_and_sign_flip():
    """Hand-derived carried steps (tests/golden/clamp_and_sign_flip.json):
    the positive-decay clamp (p1 Section 4.3), the eigenvalue 1 - beta along x
    (p3, transition eigen-structure) and a carried Falcon-1A step."""
    fx = json.load(open(os.path.join(GOLDEN, "clamp_and_sign_flip.json")))
    for case in fx["cases"]:
        inp = case["inputs"]
        a = {n: np.array(inp[n], dtype=np.float64)[None]
             for n in ("q", "k", "v", "beta", "lambda", "x_prev", "S0")}
        out = oracle.forward(case["rule"], a["q"], a["k"], a["v"], a["beta"], a["lambda"],
                             S0=a["S0"], x_prev=a["x_prev"], phi=inp["phi"],
                             eps=inp["eps"], eps_gamma=inp["eps_gamma"])
        np.testing.assert_allclose(out["o"][0], np.array(case["o"]), rtol=0, atol=1e-15,
                                   err_msg=case["name"])
        np.testing.assert_allclose(out["S"][0], np.array(case["S"]), rtol=0, atol=1e-15,
                                   err_msg=case["name"])
        np.testing.assert_array_equal(out["x_last"][0], np.array(case["x_last"]))


# --------------------------------------------------------------------------
# Check (a): NLMS interpolation.
# --------------------------------------------------------------------------

@pytest.mark.parametrize("phi", ["identity", "l2"])
def test_nlms_interpolation(phi):
    """p1 Section 3.1: with lambda = 0 and eps = 0 the step is classical NLMS;
    with beta = 1 the post-update state reproduces the target exactly,
    S_t^T x_t = v_t for every t >= 2.  At t = 1 the sentinel leaves S0 as is.
    m != dv so a transposed state fails."""
    q, k, v, beta, lam = _rand_case(1, m=6, dv=4)
    beta[:] = 1.0
    lam[:] = 0.0
    S0 = np.random.default_rng(2).standard_normal((q.shape[0], 6, 4))
    out = oracle.forward("falcon1", q, k, v, beta, lam, S0=S0, phi=phi, eps=0.0,
                         trajectory=True)
    x = _write_features(k, phi)
    St = out["S_traj"]
    pred = np.einsum("btij,bti->btj", St, x)
    err = np.abs(pred[:, 1:] - v[:, 1:]).max() / np.abs(v).max()
    assert err < 1e-12
    np.testing.assert_array_equal(St[:, 0], S0)


# --------------------------------------------------------------------------
# Check (b): one gradient step on the printed ridge loss; per-step descent.
# --------------------------------------------------------------------------

@pytest.mark.parametrize("lam_shift", [-2.0, 1.5])
def test_update_is_gradient_step_and_descends(lam_shift):
    """p1 Eq. (3.1)-(3.3): S_t = S_{t-1} - eta_t grad l_t(S_{t-1}) for the
    instantaneous ridge loss l_t(S) = 1/2||S^T x_t - v_t||^2 + lambda/2 ||S||_F^2,
    with the gradient taken by autograd (not by the printed formula) and with
    the effective ridge lambda~ = alpha/eta where the clamp is active (p1
    Section 4.3).  Lemma 3.1 (p1 Section 3.2): l_t(S_t) <= l_t(S_{t-1}) -
    eta(2 - eta L)/2 ||grad||^2 with L = ||x_t||^2 + lambda~."""
    eps, eps_gamma = 1e-3, 1e-6
    q, k, v, beta, lam = _rand_case(3, T=32, lam_shift=lam_shift)
    S0 = np.random.default_rng(4).standard_normal((q.shape[0], 5, 3))
    out = oracle.forward("falcon1", q, k, v, beta, lam, S0=S0, phi="l2", eps=eps,
                         eps_gamma=eps_gamma, trajectory=True)
    x = _write_features(k, "l2")
    eta, gamma = _eta_gamma(x, beta, lam, eps, eps_gamma)
    St = out["S_traj"]
    n_clamped = 0
    for b in range(q.shape[0]):
        prev = S0[b]
        for t in range(q.shape[1]):
            lam_eff = (1.0 - gamma[b, t]) / eta[b, t] if eta[b, t] > 0 else 0.0
            n_clamped += int(eta[b, t] * lam[b, t] > 1 - eps_gamma)
            S = torch.tensor(prev, requires_grad=True)
            xt = torch.tensor(x[b, t])
            vt = torch.tensor(v[b, t])
            loss = 0.5 * ((S.T @ xt - vt) ** 2).sum() + 0.5 * lam_eff * (S ** 2).sum()
            (grad,) = torch.autograd.grad(loss, S)
            grad = grad.numpy()
            expect = prev - eta[b, t] * grad
            np.testing.assert_allclose(St[b, t], expect, rtol=1e-12, atol=1e-12)

            def ell(M):
                return 0.5 * ((M.T @ x[b, t] - v[b, t]) ** 2).sum() + 0.5 * lam_eff * (M ** 2).sum()
            L = (x[b, t] ** 2).sum() + lam_eff
            bound = ell(prev) - eta[b, t] * (2 - eta[b, t] * L) / 2 * (grad ** 2).sum()
            assert ell(St[b, t]) <= bound + 1e-12 * max(1.0, abs(ell(prev)))
            assert ell(St[b, t]) <= ell(prev) + 1e-12 * max(1.0, abs(ell(prev)))
            prev = St[b, t]
    if lam_shift > 0:
        assert n_clamped > 0  # the large-lambda draw exercises the clamp


# --------------------------------------------------------------------------
# Check (c): Falcon-1A at lambda = 0 is shifted unnormalised linear attention.
# --------------------------------------------------------------------------

@pytest.mark.parametrize("phi", ["identity", "l2"])
def test_falcon1a_is_shifted_linear_attention(phi):
    """p1 Section 2.2 Eq. (2.3)-(2.4) with lambda = 0: the denominator-free
    read gives o_t = S0^T phi(q_t) + sum_{j=2..t} eta_j <phi(q_t), phi(k_{j-1})> v_j.
    Computed here as an O(T^2) double loop."""
    eps = 1e-6
    q, k, v, beta, lam = _rand_case(5, T=20)
    lam[:] = 0.0
    S0 = np.random.default_rng(6).standard_normal((q.shape[0], 5, 3))
    out = oracle.forward("falcon1a", q, k, v, beta, lam, S0=S0, phi=phi, eps=eps)
    qf, kf = _phi(q, phi), _phi(k, phi)
    BH, T = q.shape[:2]
    ref = np.zeros_like(out["o"])
    for b in range(BH):
        for t in range(T):
            acc = S0[b].T @ qf[b, t]
            for j in range(1, t + 1):
                xj = kf[b, j - 1]
                eta_j = beta[b, j] / ((xj ** 2).sum() + eps)
                acc = acc + eta_j * (qf[b, t] @ xj) * v[b, j]
            ref[b, t] = acc
    np.testing.assert_allclose(out["o"], ref, rtol=1e-11, atol=1e-11)


# --------------------------------------------------------------------------
# Check (d): recurrent form == masked-parallel (attention) form.
# --------------------------------------------------------------------------

def _decay_products(gamma):
    """prod_{r=j+1}^{t} gamma_r as a [T, T] lower-triangular matrix (j <= t)."""
    T = gamma.shape[0]
    P = np.zeros((T, T))
    for t in range(T):
        for j in range(t + 1):
            P[t, j] = np.prod(gamma[j + 1:t + 1])
    return P


@pytest.mark.parametrize("lam_shift", [-2.0, 1.0])
@pytest.mark.parametrize("phi", ["identity", "l2"])
def test_masked_parallel_falcon1a(phi, lam_shift):
    """p1 Section 4.6 Eq. (4.20)-(4.23) at window B = 1 (which is Falcon-1A,
    p1 Section 4.5 last paragraph):  O = Diag(delta) Q S0 + (Q X^T . M) V with
    M_{t,j} = eta_j prod_{r=j+1}^{t} gamma_r and delta_t = prod_{r<=t} gamma_r.
    Includes clamp-active draws (lam_shift = 1)."""
    eps, eps_gamma = 1e-6, 1e-6
    q, k, v, beta, lam = _rand_case(7, T=48, lam_shift=lam_shift)
    S0 = np.random.default_rng(8).standard_normal((q.shape[0], 5, 3))
    out = oracle.forward("falcon1a", q, k, v, beta, lam, S0=S0, phi=phi, eps=eps,
                         eps_gamma=eps_gamma)
    x = _write_features(k, phi)
    Q = _phi(q, phi)
    eta, gamma = _eta_gamma(x, beta, lam, eps, eps_gamma)
    for b in range(q.shape[0]):
        D = _decay_products(gamma[b])
        M = D * eta[b][None, :]
        delta = np.cumprod(gamma[b])
        O = delta[:, None] * (Q[b] @ S0[b]) + ((Q[b] @ x[b].T) * M) @ v[b]
        np.testing.assert_allclose(out["o"][b], O, rtol=1e-10, atol=1e-10)
        S_T = delta[-1] * S0[b] + x[b].T @ (M[-1][:, None] * v[b])
        np.testing.assert_allclose(out["S"][b], S_T, rtol=1e-10, atol=1e-10)


@pytest.mark.parametrize("lam_shift", [-2.0, 1.0])
@pytest.mark.parametrize("phi", ["identity", "l2"])
def test_masked_parallel_falcon1(phi, lam_shift):
    """The whole-sequence WY/UT form of Falcon-1 (the masked-parallel form the
    pages name but do not print for Falcon-1; read as one chunk spanning the
    sequence, p3 complexity table and WY remark).  With u_t := r_t the
    residual, S_t = delta_t S0 + sum_{j<=t} D_{t,j} eta_j x_j u_j^T, hence
    (I + A) (eta u) = Diag(eta) (V - Diag(delta_{t-1}) X S0) with
    A_{t,j} = eta_t D_{t-1,j} <x_t, x_j> for j < t, solved with a library
    solve; then O = Diag(delta) Q S0 + (Q X^T . D)(eta u)."""
    eps, eps_gamma = 1e-6, 1e-6
    q, k, v, beta, lam = _rand_case(9, T=64, lam_shift=lam_shift)
    S0 = np.random.default_rng(10).standard_normal((q.shape[0], 5, 3))
    out = oracle.forward("falcon1", q, k, v, beta, lam, S0=S0, phi=phi, eps=eps,
                         eps_gamma=eps_gamma)
    x = _write_features(k, phi)
    Q = _phi(q, phi)
    eta, gamma = _eta_gamma(x, beta, lam, eps, eps_gamma)
    T = q.shape[1]
    for b in range(q.shape[0]):
        D = _decay_products(gamma[b])
        delta = np.cumprod(gamma[b])
        delta_prev = np.concatenate([[1.0], delta[:-1]])
        G = x[b] @ x[b].T
        A = np.zeros((T, T))
        for t in range(T):
            for j in range(t):
                A[t, j] = eta[b, t] * D[t - 1, j] * G[t, j]
        rhs = eta[b][:, None] * (v[b] - delta_prev[:, None] * (x[b] @ S0[b]))
        W = np.linalg.solve(np.eye(T) + A, rhs)
        O = delta[:, None] * (Q[b] @ S0[b]) + ((Q[b] @ x[b].T) * D) @ W
        np.testing.assert_allclose(out["o"][b], O, rtol=1e-9, atol=1e-9)
        S_T = delta[-1] * S0[b] + x[b].T @ (D[-1][:, None] * W)
        np.testing.assert_allclose(out["S"][b], S_T, rtol=1e-9, atol=1e-9)


# --------------------------------------------------------------------------
# Invariants.
# --------------------------------------------------------------------------

@pytest.mark.parametrize("rule", ["falcon1", "falcon1a"])
def test_linear_in_values_and_initial_state(rule):
    """The transition gamma I - eta x x^T (or gamma I) depends only on k, beta,
    lambda (p1 Section 3.3, 'Decay & Targeted Forget'); the recurrence is
    therefore linear in (V, S0) jointly."""
    q, k, v, beta, lam = _rand_case(11)
    g = np.random.default_rng(12)
    v2 = g.standard_normal(v.shape)
    Sa = g.standard_normal((q.shape[0], 5, 3))
    Sb = g.standard_normal((q.shape[0], 5, 3))
    o1 = oracle.forward(rule, q, k, v, beta, lam, S0=Sa)
    o2 = oracle.forward(rule, q, k, v2, beta, lam, S0=Sb)
    o12 = oracle.forward(rule, q, k, v + 2.5 * v2, beta, lam, S0=Sa + 2.5 * Sb)
    np.testing.assert_allclose(o12["o"], o1["o"] + 2.5 * o2["o"], rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(o12["S"], o1["S"] + 2.5 * o2["S"], rtol=1e-10, atol=1e-10)


@pytest.mark.parametrize("rule", ["falcon1", "falcon1a"])
def test_l2_feature_map_scale_invariance(rule):
    """With phi(u) = u/||u|| (the QK-l2 variant of the experiments), positive
    per-token rescaling of q and k changes nothing; negating q_t negates o_t
    (the read is linear in phi(q_t), p1 Section 4 summary)."""
    q, k, v, beta, lam = _rand_case(13)
    g = np.random.default_rng(14)
    sq = np.exp(g.standard_normal(q.shape[:-1] + (1,)))
    sk = np.exp(g.standard_normal(k.shape[:-1] + (1,)))
    a = oracle.forward(rule, q, k, v, beta, lam, phi="l2")
    b = oracle.forward(rule, q * sq, k * sk, v, beta, lam, phi="l2")
    np.testing.assert_allclose(b["o"], a["o"], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(b["S"], a["S"], rtol=1e-11, atol=1e-12)
    sign = np.where(g.standard_normal(q.shape[:-1] + (1,)) > 0, 1.0, -1.0)
    c = oracle.forward(rule, q * sign, k, v, beta, lam, phi="l2")
    np.testing.assert_allclose(c["o"], a["o"] * sign, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("rule", ["falcon1", "falcon1a"])
def test_continuation_split_equals_full(rule):
    """Exact continuation needs the state and the last write feature
    phi(k_T) (the B = 1 case of the tail in p1 Section 4.4): running T1 tokens
    and then T - T1 tokens with (S, x_prev) carried equals one run."""
    q, k, v, beta, lam = _rand_case(15, T=30)
    full = oracle.forward(rule, q, k, v, beta, lam)
    for T1 in (1, 13, 29):
        a = oracle.forward(rule, q[:, :T1], k[:, :T1], v[:, :T1], beta[:, :T1], lam[:, :T1])
        b = oracle.forward(rule, q[:, T1:], k[:, T1:], v[:, T1:], beta[:, T1:], lam[:, T1:],
                           S0=a["S"], x_prev=a["x_last"])
        np.testing.assert_allclose(np.concatenate([a["o"], b["o"]], 1), full["o"],
                                   rtol=1e-13, atol=1e-13)
        np.testing.assert_allclose(b["S"], full["S"], rtol=1e-13, atol=1e-13)
        np.testing.assert_array_equal(b["x_last"], full["x_last"])


@pytest.mark.parametrize("rule", ["falcon1", "falcon1a"])
def test_decode_steps_equal_forward(rule):
    """The recurrent decode form (p3 complexity table: O(1) state per token)
    run token by token, fresh at the first token, equals the sequence form."""
    q, k, v, beta, lam = _rand_case(17, T=12)
    S0 = np.random.default_rng(18).standard_normal((q.shape[0], 5, 3))
    full = oracle.forward(rule, q, k, v, beta, lam, S0=S0)
    S = S0.copy()
    xp = np.full((q.shape[0], 5), np.nan)  # must be ignored at the sentinel
    outs = []
    for t in range(q.shape[1]):
        fresh = np.full(q.shape[0], t == 0)
        outs.append(oracle.decode_step(rule, q[:, t], k[:, t], v[:, t], beta[:, t], lam[:, t],
                                       S, xp, fresh=fresh))
    np.testing.assert_allclose(np.stack(outs, 1), full["o"], rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(S, full["S"], rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(xp, full["x_last"], rtol=0, atol=0)


def test_sentinel_ignores_lambda_at_first_token():
    """p1 Section 3: eta_1 := 0 so that lambda_1 > 0 does not decay a carried
    state when no pair is written: a fresh call with S0 != 0 and one token
    returns S0 unchanged and o_1 = S0^T phi(q_1)."""
    q, k, v, beta, lam = _rand_case(19, T=1)
    lam[:] = 5.0
    S0 = np.random.default_rng(20).standard_normal((q.shape[0], 5, 3))
    for rule in ("falcon1", "falcon1a"):
        out = oracle.forward(rule, q, k, v, beta, lam, S0=S0, phi="identity")
        np.testing.assert_array_equal(out["S"], S0)
        np.testing.assert_allclose(out["o"][:, 0], np.einsum("bij,bi->bj", S0, q[:, 0]),
                                   rtol=1e-14, atol=1e-14)


def test_zero_length_and_zero_denominator():
    """T = 0 returns S0 and x_prev untouched.  A zero write feature with
    lambda = eps = 0 makes the denominator vanish: eta := 0 (p1 Eq. (3.4)),
    so the step is a no-op."""
    q, k, v, beta, lam = _rand_case(21, T=0)
    S0 = np.ones((q.shape[0], 5, 3))
    xp = np.ones((q.shape[0], 5))
    out = oracle.forward("falcon1", q, k, v, beta, lam, S0=S0, x_prev=xp)
    np.testing.assert_array_equal(out["S"], S0)
    np.testing.assert_array_equal(out["x_last"], xp)
    q, k, v, beta, lam = _rand_case(22, T=2)
    lam[:] = 0.0
    k[:, 0] = 0.0
    out = oracle.forward("falcon1", q, k, v, beta, lam, S0=S0, phi="identity", eps=0.0)
    np.testing.assert_array_equal(out["S"], S0)
