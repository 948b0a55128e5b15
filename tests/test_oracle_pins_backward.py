"""Pins of the oracle's backward pass (Falcon-1 / Falcon-1A).

Page hyper.ai/fr/papers/2608.27763 (p1) says training differentiates through
the update (Section 3, "Implicit fast-memory objective") and that the
backward pass goes through the log-decay renormalisation and the normalised
step size (Section 4.6, "Backward pass"); the appendix with its formulas is
not on the pages.  So the backward is pinned to what defines a gradient,
with no reference to how the oracle computes it:

  - central finite differences of the oracle's forward (itself pinned by
    test_oracle_pins*.py) for every input, every rule, feature map and ridge
    form, with and without carried state and end cotangents, including
    tokens on the clamped branch of the decay;
  - exact affine identities: S0 -> (o, S_T) and v -> (o, S_T) are affine for
    Falcon-1 and Falcon-1A, and q enters only the read, so
    L(z + D) - L(z) = <dL/dz, D> for any finite D, with no step-size error;
  - a closed form: Falcon-1A at lambda = 0 is shifted linear attention
    o_t = sum_{j<=t} eta_j <phi(q_t), x_j> v_j (p1 Eq. (4.6) with gamma = 1),
    so dv_j = eta_j sum_{t>=j} <phi(q_t), x_j> dO_t.
"""
import zlib

import numpy as np
import pytest

import oracle


def _case(seed, BH=2, T=6, m=4, dv=3, lam_shift=-1.0, beta_scale=1.0):
    g = np.random.default_rng(seed)
    c = {
        "q": g.standard_normal((BH, T, m)) * 1.3,
        "k": g.standard_normal((BH, T, m)) * 0.9,
        "v": g.standard_normal((BH, T, dv)),
        "beta": beta_scale * 2.0 / (1 + np.exp(-g.standard_normal((BH, T)))),
        "lam": np.log1p(np.exp(g.standard_normal((BH, T)) + lam_shift)),
        "S0": g.standard_normal((BH, m, dv)) * 0.5,
        "x_prev": g.standard_normal((BH, m)) * 0.4,
    }
    cot = {
        "dO": g.standard_normal((BH, T, dv)),
        "dS_T": g.standard_normal((BH, m, dv)),
        "dx_last": g.standard_normal((BH, m)),
    }
    return c, cot


def _loss(rule, c, cot, phi, ridge, carried, ends):
    out = oracle.forward(rule, c["q"], c["k"], c["v"], c["beta"], c["lam"],
                         S0=c["S0"] if carried else None,
                         x_prev=c["x_prev"] if carried else None, phi=phi, ridge=ridge,
                         threads=1)
    L = float((cot["dO"] * out["o"]).sum())
    if ends:
        L += float((cot["dS_T"] * out["S"]).sum()) + float((cot["dx_last"] * out["x_last"]).sum())
    return L


def _grads(rule, c, cot, phi, ridge, carried, ends):
    return oracle.backward(rule, c["q"], c["k"], c["v"], c["beta"], c["lam"], cot["dO"],
                           S0=c["S0"] if carried else None,
                           x_prev=c["x_prev"] if carried else None,
                           dS_T=cot["dS_T"] if ends else None,
                           dx_last=cot["dx_last"] if ends else None,
                           phi=phi, ridge=ridge, threads=1)


_NAMES = {"q": "dq", "k": "dk", "v": "dv", "beta": "dbeta", "lam": "dlambda", "S0": "dS0",
          "x_prev": "dx_prev"}


def _fd_check(rule, c, cot, phi, ridge, carried, ends, h=1e-6, rtol=2e-6):
    g = _grads(rule, c, cot, phi, ridge, carried, ends)
    names = ["q", "k", "v", "beta", "lam"] + (["S0", "x_prev"] if carried else [])
    for name in names:
        arr = c[name]
        fd = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            old = arr[idx]
            step = h * max(1.0, abs(old))
            arr[idx] = old + step
            lp = _loss(rule, c, cot, phi, ridge, carried, ends)
            arr[idx] = old - step
            lm = _loss(rule, c, cot, phi, ridge, carried, ends)
            arr[idx] = old
            fd[idx] = (lp - lm) / (2 * step)
        got = g[_NAMES[name]]
        scale = max(np.abs(fd).max(), 1e-3)
        err = np.abs(got - fd).max() / scale
        assert err < rtol, (name, err)
    if not carried:
        assert np.all(g["dx_prev"] == 0)


@pytest.mark.parametrize("rule", ["falcon1", "falcon1a"])
@pytest.mark.parametrize("phi", ["identity", "l2", "rms"])
@pytest.mark.parametrize("ridge", ["given", "scaled"])
@pytest.mark.parametrize("carried,ends", [(False, False), (True, True)])
def test_backward_matches_finite_differences(rule, phi, ridge, carried, ends):
    """Every gradient against central differences of the forward."""
    seed = zlib.crc32(f"{rule}/{phi}/{ridge}/{carried}".encode()) % 1000
    c, cot = _case(seed)
    _fd_check(rule, c, cot, phi, ridge, carried, ends)


@pytest.mark.parametrize("rule", ["falcon1", "falcon1a"])
def test_backward_on_clamped_tokens(rule):
    """Large ridge: eta_t lambda_t > 1 - eps_gamma on many tokens, where the
    decay is the constant eps_gamma (p1 Section 4.3, "Decay positivity");
    the finite differences stay on one branch."""
    c, cot = _case(11, T=8, lam_shift=3.0, beta_scale=1.0)
    c["beta"][:] = np.where(np.arange(8) % 2 == 0, 1.6, 0.7)
    out = oracle.forward(rule, c["q"], c["k"], c["v"], c["beta"], c["lam"], S0=c["S0"],
                         x_prev=c["x_prev"], phi="l2", threads=1)
    # eta lambda with E = ||x||^2: 1 for l2 features, ||x_prev||^2 at token 1
    E = np.ones_like(c["lam"])
    E[:, 0] = (c["x_prev"] ** 2).sum(-1)
    eta = c["beta"] / (E + c["lam"] + 1e-6)
    margin = eta * c["lam"] - (1 - 1e-6)
    assert (margin > 1e-3).sum() >= 4 and np.all(np.abs(margin) > 1e-4)
    assert np.isfinite(out["o"]).all()
    _fd_check(rule, c, cot, "l2", "given", True, True)


@pytest.mark.parametrize("rule", ["falcon1", "falcon1a"])
@pytest.mark.parametrize("name,key", [("S0", "dS0"), ("v", "dv")])
def test_backward_affine_inputs_exact(rule, name, key):
    """o and S_T are affine in S0 and in v (the write is linear in r, and r
    is affine in v and S): a finite change D gives L(z + D) - L(z) =
    <dL/dz, D> exactly."""
    c, cot = _case(21, BH=2, T=9, m=5, dv=4)
    g = _grads(rule, c, cot, "l2", "given", True, True)
    D = np.random.default_rng(22).standard_normal(c[name].shape)
    L0 = _loss(rule, c, cot, "l2", "given", True, True)
    c[name] = c[name] + D
    L1 = _loss(rule, c, cot, "l2", "given", True, True)
    assert abs((L1 - L0) - (g[key] * D).sum()) < 1e-10 * max(1.0, abs(L1 - L0))


@pytest.mark.parametrize("rule", ["falcon1", "falcon1a"])
def test_backward_read_only_input_exact(rule):
    """q enters only the read o_t = S_t^T phi(q_t); with phi the identity the
    loss is linear in q."""
    c, cot = _case(31, BH=1, T=7, m=4, dv=5)
    g = _grads(rule, c, cot, "identity", "given", False, True)
    D = np.random.default_rng(32).standard_normal(c["q"].shape)
    L0 = _loss(rule, c, cot, "identity", "given", False, True)
    c["q"] = c["q"] + D
    L1 = _loss(rule, c, cot, "identity", "given", False, True)
    assert abs((L1 - L0) - (g["dq"] * D).sum()) < 1e-10 * max(1.0, abs(L1 - L0))


def test_falcon1a_value_gradient_closed_form():
    """Falcon-1A with lambda = 0: o_t = sum_{j<=t} eta_j <phi(q_t), x_j> v_j
    with x_j = phi(k_{j-1}), x_1 = 0, eta_1 = 0 (p1 Eq. (4.6), Eq. (4.8)), so
    dv_j = eta_j sum_{t>=j} <phi(q_t), x_j> dO_t."""
    c, cot = _case(41, BH=2, T=10, m=6, dv=3)
    c["lam"][:] = 0.0
    eps = 1e-6
    g = _grads("falcon1a", c, cot, "l2", "given", False, False)
    qf = c["q"] / np.linalg.norm(c["q"], axis=-1, keepdims=True)
    kf = c["k"] / np.linalg.norm(c["k"], axis=-1, keepdims=True)
    x = np.zeros_like(kf)
    x[:, 1:] = kf[:, :-1]
    eta = c["beta"] / ((x * x).sum(-1) + eps)
    eta[:, 0] = 0.0
    want = np.zeros_like(c["v"])
    T = c["q"].shape[1]
    for b in range(c["q"].shape[0]):
        for j in range(T):
            for t in range(j, T):
                want[b, j] += eta[b, j] * (qf[b, t] @ x[b, j]) * cot["dO"][b, t]
    np.testing.assert_allclose(g["dv"], want, rtol=1e-12, atol=1e-14)


def test_backward_empty_and_zero_cotangent():
    """T = 0 gives dS0 = dS_T and dx_prev = dx_last (S_T = S0 and
    x_last = x_prev); zero cotangents give zero gradients."""
    c, cot = _case(51, T=0)
    g = _grads("falcon1", c, cot, "l2", "given", True, True)
    np.testing.assert_array_equal(g["dS0"], cot["dS_T"])
    np.testing.assert_array_equal(g["dx_prev"], cot["dx_last"])
    c, cot = _case(52)
    cot = {k: np.zeros_like(v) for k, v in cot.items()}
    g = _grads("falcon1", c, cot, "l2", "given", True, True)
    assert all(np.all(v == 0) for v in g.values())
