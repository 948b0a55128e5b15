"""GPU parity of the chunked Falcon-2 forward (falcon2_fwd_chunked: the
blocked per-column solve in chunk form on the tensor cores for bf16
m = d_v = 64, the token-recurrent kernel otherwise) against the fp64 oracle,
through the C ABI.  Error measure as in test_gpu_parity.py: ||err||_F /
||ref||_F per head, max over heads; <= 1e-4 for fp32 inputs, <= 2e-2 for
bf16 inputs."""
import numpy as np
import pytest
import torch

import oracle
from delta_rule_attention_gb300 import workloads

from test_gpu_parity import TOL, head_err

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]


@pytest.fixture(scope="module")
def falcon():
    import delta_rule_attention_gb300 as f
    f.load_library()
    return f


def run2c(falcon, x, phi="l2", ridge="given", eps_gamma=1e-6):
    o, S, xl = falcon.falcon2_fwd_chunked(x["q"], x["k"], x["v"], x["beta"], x["lambda"],
                                          S0=x.get("S0"), x_prev=x.get("x_prev"), phi=phi,
                                          ridge=ridge, eps_gamma=eps_gamma)
    assert falcon.falcon_sync_check() == 0
    return o.float().cpu(), S.cpu(), xl.cpu()


def ref2(x, phi="l2", ridge="given", eps_gamma=1e-6):
    return oracle.forward2("falcon2", x["q"], x["k"], x["v"], x["beta"], x["lambda"],
                           S0=x.get("S0"), x_prev=x.get("x_prev"), phi=phi, ridge=ridge,
                           eps_gamma=eps_gamma)


CASES = [
    # B, H, T, dtype, phi (m = d_v = 64; bf16: tensor cores, fp32: recurrent)
    (2, 3, 3 * 64 + 5, torch.bfloat16, "l2"),   # several chunks, ragged tail
    (1, 2, 64, torch.bfloat16, "identity"),     # exactly one chunk
    (1, 2, 65, torch.bfloat16, "rms"),          # one token into the second chunk
    (3, 2, 7, torch.bfloat16, "l2"),            # shorter than a chunk
    (1, 2, 1, torch.bfloat16, "l2"),            # a single token
    (1, 4, 700, torch.bfloat16, "l2"),          # eleven chunks (the input ring wraps)
    (2, 2, 150, torch.float32, "l2"),           # fp32: the recurrent kernel
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c[:3])) + str(c[3])[-4:])
@pytest.mark.parametrize("carried", [False, True])
def test_falcon2_chunked_small_shapes(falcon, case, carried):
    B, H, T, dt, phi = case
    x = workloads.random_case(B, H, T, 64, 64, dt, seed=700 + CASES.index(case), device="cuda",
                              with_state=carried, with_x_prev=carried, per_column=True)
    o, S, xl = run2c(falcon, x, phi)
    ref = ref2(x, phi)
    assert head_err(o, ref["o"]) < TOL[dt]
    assert head_err(S, ref["S"]) < TOL[dt]
    np.testing.assert_allclose(xl.numpy(), ref["x_last"], rtol=1e-6, atol=1e-6)


@pytest.mark.parametrize("lam_shift", [1.0, 3.0])
def test_falcon2_chunked_clamped_and_strong_decay(falcon, lam_shift):
    """lambda = softplus(n + 1) and softplus(n + 3) with per-column gains up to
    2: the clamp fires on some (token, column) pairs and not on others, and the
    decay products inside a chunk underflow; the blocked solve uses products of
    gammas only."""
    x = workloads.random_case(2, 3, 400, 64, 64, torch.bfloat16, seed=719, lam_shift=lam_shift,
                              device="cuda", with_state=True, with_x_prev=True, per_column=True)
    o, S, _ = run2c(falcon, x)
    ref = ref2(x)
    eta_lam = (x["beta"] * (x["lambda"] / (1.0 + x["lambda"]))[..., None]).cpu()
    assert (eta_lam >= 1 - 1e-6).any(), "the clamp must fire somewhere"
    assert np.isfinite(o.numpy()).all() and np.isfinite(S.numpy()).all()
    assert head_err(o, ref["o"]) < 2e-2
    assert head_err(S, ref["S"]) < 2e-2


def test_falcon2_chunked_scaled_ridge(falcon):
    x = workloads.random_case(2, 2, 300, 64, 64, torch.bfloat16, seed=731, device="cuda",
                              with_state=True, per_column=True)
    o, S, _ = run2c(falcon, x, ridge="scaled")
    ref = ref2(x, ridge="scaled")
    assert head_err(o, ref["o"]) < 2e-2
    assert head_err(S, ref["S"]) < 2e-2


def test_falcon2_chunked_lm_workload_all_heads(falcon):
    """B8 H12 T2048 d64 bf16 with one gain per column (the lm-2 workload),
    every head compared in full."""
    w = workloads.LM_2
    x = workloads.generate(w, device="cuda")
    o, S, _ = run2c(falcon, x, w.phi)
    ref = ref2(x, w.phi)
    assert head_err(o, ref["o"]) < 2e-2
    assert head_err(S, ref["S"]) < 2e-2


def test_falcon2_chunked_matches_recurrent_kernel(falcon):
    """The chunk form and the token-recurrent kernel agree within the bf16
    tolerance on the same inputs (more heads than SMs: every CTA slot reused)."""
    x = workloads.random_case(4, 48, 256, 64, 64, torch.bfloat16, seed=733, device="cuda",
                              with_state=True, per_column=True)
    oc, Sc, _ = falcon.falcon2_fwd_chunked(x["q"], x["k"], x["v"], x["beta"], x["lambda"],
                                           S0=x["S0"])
    orr, Sr, _ = falcon.falcon2_fwd_recurrent(x["q"], x["k"], x["v"], x["beta"], x["lambda"],
                                              S0=x["S0"])
    assert falcon.falcon_sync_check() == 0
    assert head_err(oc.float().cpu(), orr.float().cpu().numpy()) < 2e-2
    assert head_err(Sc.cpu(), Sr.cpu().numpy()) < 2e-2


def test_falcon2_chunked_repeatable(falcon):
    """Two calls on the same inputs give bit-identical outputs (no atomics,
    fixed order of every sum)."""
    x = workloads.random_case(2, 4, 333, 64, 64, torch.bfloat16, seed=737, device="cuda",
                              with_state=True, with_x_prev=True, per_column=True)
    o1, S1, _ = run2c(falcon, x)
    o2, S2, _ = run2c(falcon, x)
    assert torch.equal(o1, o2) and torch.equal(S1, S2)
