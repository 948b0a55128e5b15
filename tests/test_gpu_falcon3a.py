"""GPU parity of Falcon-3A (sliding-window inner-product rule, token-recurrent
kernel) against the fp64 oracle, through the C ABI.  Error measure as in
test_gpu_parity.py: ||err||_F / ||ref||_F per head, max over heads; <= 1e-4
for fp32 inputs, <= 2e-2 for bf16 inputs."""
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


def run3(falcon, x, window, phi="l2", ridge="given"):
    o, S, xl = falcon.falcon3a_fwd_recurrent(x["q"], x["k"], x["v"], x["beta"], x["lambda"],
                                             window, S0=x.get("S0"), phi=phi, ridge=ridge)
    assert falcon.falcon_sync_check() == 0
    return o.float().cpu(), S.cpu(), xl.cpu()


def ref3(x, window, phi="l2", ridge="given"):
    return oracle.forward3a(x["q"], x["k"], x["v"], x["beta"], x["lambda"], window,
                            S0=x.get("S0"), phi=phi, ridge=ridge)


CASES3 = [
    # B, H, T, m, dv, dtype, phi
    (1, 2, 64, 16, 16, torch.float32, "identity"),
    (2, 3, 3 * 32 + 5, 64, 64, torch.bfloat16, "l2"),   # several token blocks, ragged tail
    (1, 2, 150, 32, 128, torch.float32, "l2"),          # four column groups
    (1, 3, 257, 128, 128, torch.bfloat16, "rms"),
    (3, 2, 7, 64, 16, torch.float32, "l2"),             # shorter than the window
    (1, 2, 1, 64, 64, torch.bfloat16, "l2"),            # a single token
]


@pytest.mark.parametrize("window", [1, 3, 17, 32])
@pytest.mark.parametrize("case", CASES3, ids=lambda c: "x".join(map(str, c[:5])) + str(c[5])[-4:])
@pytest.mark.parametrize("with_state", [False, True])
def test_falcon3a_small_shapes(falcon, window, case, with_state):
    B, H, T, m, dv, dt, phi = case
    x = workloads.random_case(B, H, T, m, dv, dt, seed=200 + CASES3.index(case), device="cuda",
                              with_state=with_state)
    o, S, xl = run3(falcon, x, window, phi)
    ref = ref3(x, window, phi)
    assert head_err(o, ref["o"]) < TOL[dt]
    assert head_err(S, ref["S"]) < TOL[dt]
    np.testing.assert_allclose(xl.numpy(), ref["x_last"], rtol=2e-6, atol=2e-6)


def test_falcon3a_window_one_matches_falcon1a_kernels(falcon):
    """A window of one pair is Falcon-1A (p1 Section 4.5): the recurrent
    windowed kernel and the chunked tensor-core kernel agree."""
    x = workloads.random_case(2, 4, 512, 64, 64, torch.bfloat16, seed=8, device="cuda",
                              with_state=True)
    o3, S3, _ = falcon.falcon3a_fwd_recurrent(x["q"], x["k"], x["v"], x["beta"], x["lambda"], 1,
                                              S0=x["S0"])
    o1, S1, _ = falcon.falcon1a_fwd_chunked(x["q"], x["k"], x["v"], x["beta"], x["lambda"],
                                            S0=x["S0"], chunk=64)
    assert falcon.falcon_sync_check() == 0
    assert head_err(o3.float().cpu(), o1.float().cpu()) < 2e-2
    assert head_err(S3.cpu(), S1.cpu()) < 2e-2


@pytest.mark.parametrize("ridge", ["given", "scaled"])
def test_falcon3a_clamp_and_ridge(falcon, ridge):
    """lambda = softplus(n + 3) with gains up to 2: the clamp fires on many
    tokens; the scale-coupled ridge uses the window energy."""
    x = workloads.random_case(2, 2, 200, 64, 64, torch.float32, seed=277, lam_shift=3.0,
                              device="cuda", with_state=True)
    o, S, _ = run3(falcon, x, 5, "l2", ridge)
    ref = ref3(x, 5, "l2", ridge)
    assert np.isfinite(o.numpy()).all()
    assert head_err(o, ref["o"]) < 1e-4
    assert head_err(S, ref["S"]) < 1e-4


def test_falcon3a_lm_workload_all_heads(falcon):
    """B8 H12 T2048 d64 bf16, window 4, every head compared in full."""
    w = workloads.LM_3A
    x = workloads.generate(w, device="cuda")
    o, S, _ = run3(falcon, x, workloads.LM_3A_WINDOW, w.phi)
    ref = ref3(x, workloads.LM_3A_WINDOW, w.phi)
    assert head_err(o, ref["o"]) < 2e-2
    assert head_err(S, ref["S"]) < 2e-2


def test_falcon3a_rejects_bad_window_and_x_prev(falcon):
    x = workloads.random_case(1, 1, 16, 64, 64, torch.bfloat16, seed=1, device="cuda")
    for bad in (0, 33):
        with pytest.raises(falcon.FalconError):
            falcon.falcon3a_fwd_recurrent(x["q"], x["k"], x["v"], x["beta"], x["lambda"], bad)
