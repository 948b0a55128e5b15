"""GPU parity of Falcon-2 / Falcon-2A (per-column step sizes, token-recurrent
kernel) against the fp64 oracle, through the C ABI.

Error measure as in test_gpu_parity.py: ||err||_F / ||ref||_F per head, max
over heads; <= 1e-4 for fp32 inputs, <= 2e-2 for bf16 inputs.
"""
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


def run2(falcon, rule, x, phi, eps=1e-6, eps_gamma=1e-6):
    fn = falcon.falcon2_fwd_recurrent if rule == "falcon2" else falcon.falcon2a_fwd_recurrent
    o, S, xl = fn(x["q"], x["k"], x["v"], x["beta"], x["lambda"], S0=x.get("S0"),
                  x_prev=x.get("x_prev"), phi=phi, eps=eps, eps_gamma=eps_gamma)
    assert falcon.falcon_sync_check() == 0
    return o.float().cpu(), S.cpu(), xl.cpu()


def ref2(rule, x, phi, eps=1e-6, eps_gamma=1e-6):
    return oracle.forward2(rule, x["q"], x["k"], x["v"], x["beta"], x["lambda"],
                           S0=x.get("S0"), x_prev=x.get("x_prev"), phi=phi, eps=eps,
                           eps_gamma=eps_gamma)


CASES2 = [
    # B, H, T, m, dv, dtype, phi
    (1, 2, 64, 16, 16, torch.float32, "identity"),
    (2, 3, 3 * 32 + 5, 64, 64, torch.bfloat16, "l2"),   # several token blocks, ragged tail
    (1, 2, 70, 32, 128, torch.float32, "l2"),           # four column groups
    (2, 1, 100, 128, 32, torch.bfloat16, "l2"),
    (1, 3, 257, 128, 128, torch.bfloat16, "l2"),
    (1, 2, 40, 16, 64, torch.float32, "identity"),
    (3, 2, 7, 64, 16, torch.float32, "l2"),             # shorter than one token block
    (1, 2, 1, 64, 64, torch.bfloat16, "l2"),            # a single token
]


@pytest.mark.parametrize("rule", ["falcon2", "falcon2a"])
@pytest.mark.parametrize("case", CASES2, ids=lambda c: "x".join(map(str, c[:5])) + str(c[5])[-4:])
@pytest.mark.parametrize("carried", [False, True])
def test_falcon2_small_shapes(falcon, rule, case, carried):
    B, H, T, m, dv, dt, phi = case
    x = workloads.random_case(B, H, T, m, dv, dt, seed=100 + CASES2.index(case), device="cuda",
                              with_state=carried, with_x_prev=carried, per_column=True)
    o, S, xl = run2(falcon, rule, x, phi)
    ref = ref2(rule, x, phi)
    assert head_err(o, ref["o"]) < TOL[dt]
    assert head_err(S, ref["S"]) < TOL[dt]
    np.testing.assert_allclose(xl.numpy(), ref["x_last"], rtol=1e-6, atol=1e-6)


@pytest.mark.parametrize("rule", ["falcon2", "falcon2a"])
def test_falcon2_clamp_active(falcon, rule):
    """lambda = softplus(n + 3) with gains up to 2: the per-column clamp fires
    on some columns of a token and not on others."""
    x = workloads.random_case(2, 2, 200, 64, 64, torch.float32, seed=177, lam_shift=3.0,
                              device="cuda", with_state=True, per_column=True)
    o, S, _ = run2(falcon, rule, x, "l2")
    ref = ref2(rule, x, "l2")
    assert np.isfinite(o.numpy()).all() and np.isfinite(S.numpy()).all()
    assert head_err(o, ref["o"]) < 1e-4
    assert head_err(S, ref["S"]) < 1e-4


@pytest.mark.parametrize("w", [workloads.LM_2, workloads.LM_2A], ids=lambda w: w.name)
def test_falcon2_lm_workloads_all_heads(falcon, w):
    """B8 H12 T2048 d64 bf16, one gain per column, every head compared in full."""
    x = workloads.generate(w, device="cuda")
    o, S, _ = run2(falcon, w.rule, x, w.phi)
    ref = ref2(w.rule, x, w.phi)
    assert head_err(o, ref["o"]) < 2e-2
    assert head_err(S, ref["S"]) < 2e-2


def test_falcon2_tied_gains_match_falcon1_kernels(falcon):
    """Tied gains reduce Falcon-2 to Falcon-1 (p1 Section 4.2): the recurrent
    per-column kernel and the chunked tensor-core kernel agree within the bf16
    tolerance on the same inputs."""
    x = workloads.random_case(2, 4, 512, 64, 64, torch.bfloat16, seed=5, device="cuda",
                              with_state=True)
    x2 = dict(x)
    x2["beta"] = x["beta"][..., None].expand(-1, -1, -1, 64).contiguous()
    o2, S2, _ = falcon.falcon2_fwd_recurrent(x2["q"], x2["k"], x2["v"], x2["beta"], x2["lambda"],
                                             S0=x2["S0"])
    o1, S1, _ = falcon.falcon1_fwd_chunked(x["q"], x["k"], x["v"], x["beta"], x["lambda"],
                                           S0=x["S0"], chunk=64)
    assert falcon.falcon_sync_check() == 0
    assert head_err(o2.float().cpu(), o1.float().cpu()) < 2e-2
    assert head_err(S2.cpu(), S1.cpu()) < 2e-2


def test_falcon2_zero_length(falcon):
    """T = 0: S_T = S0 and x_last = x_prev; nothing is launched."""
    x = workloads.random_case(1, 2, 0, 64, 64, torch.bfloat16, seed=9, device="cuda",
                              with_state=True, with_x_prev=True, per_column=True)
    o, S, xl = run2(falcon, "falcon2", x, "l2")
    np.testing.assert_array_equal(S.numpy(), x["S0"].cpu().numpy())
    np.testing.assert_array_equal(xl.numpy(), x["x_prev"].cpu().numpy())
