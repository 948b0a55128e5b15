"""GPU parity of the feature and ridge variants (page hyper.ai/fr/papers/2608.27763,
Section 4.1): phi = RMSNorm and the scale-coupled ridge lambda_t = lambda_bar_t
||x_t||^2, on every path (generic fp32 chunked, tensor-core chunked m = 64 and
128, Falcon-2 recurrent, decode), against the fp64 oracle.  Error measure and
tolerances as in test_gpu_parity.py."""
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


VARIANTS = [("rms", "given"), ("rms", "scaled"), ("l2", "scaled")]
SHAPES = [  # B, H, T, m, dv, chunk, dtype: generic fp32, tensor-core m = 64 and 128
    (1, 2, 130, 32, 32, 32, torch.float32),
    (2, 2, 3 * 64 + 9, 64, 64, 64, torch.bfloat16),
    (1, 2, 2 * 64 + 30, 128, 128, 64, torch.bfloat16),
]


@pytest.mark.parametrize("rule", ["falcon1", "falcon1a"])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda c: f"m{c[3]}{str(c[6])[-4:]}")
@pytest.mark.parametrize("phi,ridge", VARIANTS)
def test_chunked_variants(falcon, rule, shape, phi, ridge):
    B, H, T, m, dv, C, dt = shape
    x = workloads.random_case(B, H, T, m, dv, dt, seed=T + m, device="cuda", with_state=True,
                              with_x_prev=True, lam_shift=0.0 if ridge == "scaled" else -2.0)
    fn = falcon.falcon1_fwd_chunked if rule == "falcon1" else falcon.falcon1a_fwd_chunked
    o, S, xl = fn(x["q"], x["k"], x["v"], x["beta"], x["lambda"], S0=x["S0"], x_prev=x["x_prev"],
                  chunk=C, phi=phi, ridge=ridge)
    assert falcon.falcon_sync_check() == 0
    ref = oracle.forward(rule, x["q"], x["k"], x["v"], x["beta"], x["lambda"], S0=x["S0"],
                         x_prev=x["x_prev"], phi=phi, ridge=ridge)
    assert head_err(o.float().cpu(), ref["o"]) < TOL[dt]
    assert head_err(S.cpu(), ref["S"]) < TOL[dt]
    np.testing.assert_allclose(xl.cpu().numpy(), ref["x_last"], rtol=2e-6, atol=2e-6)


@pytest.mark.parametrize("rule", ["falcon2", "falcon2a"])
@pytest.mark.parametrize("phi,ridge", VARIANTS)
def test_falcon2_variants(falcon, rule, phi, ridge):
    x = workloads.random_case(2, 2, 100, 64, 64, torch.bfloat16, seed=11, device="cuda",
                              with_state=True, with_x_prev=True, per_column=True,
                              lam_shift=0.0 if ridge == "scaled" else -2.0)
    fn = falcon.falcon2_fwd_recurrent if rule == "falcon2" else falcon.falcon2a_fwd_recurrent
    o, S, _ = fn(x["q"], x["k"], x["v"], x["beta"], x["lambda"], S0=x["S0"], x_prev=x["x_prev"],
                 phi=phi, ridge=ridge)
    assert falcon.falcon_sync_check() == 0
    ref = oracle.forward2(rule, x["q"], x["k"], x["v"], x["beta"], x["lambda"], S0=x["S0"],
                          x_prev=x["x_prev"], phi=phi, ridge=ridge)
    assert head_err(o.float().cpu(), ref["o"]) < 2e-2
    assert head_err(S.cpu(), ref["S"]) < 2e-2


@pytest.mark.parametrize("rule", ["falcon1", "falcon1a"])
@pytest.mark.parametrize("phi,ridge", VARIANTS)
def test_decode_variants(falcon, rule, phi, ridge):
    N, m, dv = 64, 128, 128
    g = torch.Generator().manual_seed(17)
    q, k, v = (torch.randn((N, d), generator=g).to(torch.bfloat16).cuda() for d in (m, m, dv))
    beta = (2 * torch.sigmoid(torch.randn(N, generator=g))).cuda()
    lam = torch.nn.functional.softplus(torch.randn(N, generator=g)).cuda()
    S = (0.3 * torch.randn((N, m, dv), generator=g)).cuda()
    xp = torch.randn((N, m), generator=g)
    xp = (xp / xp.norm(dim=-1, keepdim=True) * (m ** 0.5 if phi == "rms" else 1.0)).cuda()
    S_ref = S.double().cpu().numpy().copy()
    xp_ref = xp.double().cpu().numpy().copy()
    fn = falcon.falcon1_decode_step if rule == "falcon1" else falcon.falcon1a_decode_step
    o = fn(q, k, v, beta, lam, S, xp, phi=phi, ridge=ridge)
    assert falcon.falcon_sync_check() == 0
    o_ref = oracle.decode_step(rule, q, k, v, beta, lam, S_ref, xp_ref, phi=phi, ridge=ridge)
    assert head_err(o.float().cpu(), o_ref, head_dims=1) < 2e-2
    assert head_err(S.cpu(), S_ref) < 1e-4
    np.testing.assert_allclose(xp.cpu().numpy(), xp_ref, rtol=2e-6, atol=2e-6)
