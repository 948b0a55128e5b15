"""GPU parity of the chunked Falcon-3A forward (falcon3a_fwd_chunked: the
masked-attention form of page hyper.ai/fr/papers/2608.27763 Section 4.6 on the
tensor cores for bf16 m = d_v = 64, the token-recurrent kernel otherwise)
against the fp64 oracle, through the C ABI.  Error measure as in
test_gpu_parity.py: ||err||_F / ||ref||_F per head, max over heads; <= 1e-4 for
fp32 inputs, <= 2e-2 for bf16 inputs."""
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


def run3c(falcon, x, window, phi="l2", ridge="given"):
    o, S, xl = falcon.falcon3a_fwd_chunked(x["q"], x["k"], x["v"], x["beta"], x["lambda"],
                                           window, S0=x.get("S0"), phi=phi, ridge=ridge)
    assert falcon.falcon_sync_check() == 0
    return o.float().cpu(), S.cpu(), xl.cpu()


def ref3(x, window, phi="l2", ridge="given"):
    return oracle.forward3a(x["q"], x["k"], x["v"], x["beta"], x["lambda"], window,
                            S0=x.get("S0"), phi=phi, ridge=ridge)


CASES = [
    # B, H, T, dtype, phi: m = d_v = 64 (bf16: tensor cores; fp32: recurrent)
    (2, 3, 3 * 64 + 5, torch.bfloat16, "l2"),   # several chunks, ragged tail
    (1, 2, 64, torch.bfloat16, "l2"),           # exactly one chunk
    (1, 2, 65, torch.bfloat16, "rms"),          # one token into the second chunk
    (3, 2, 7, torch.bfloat16, "identity"),      # shorter than the window
    (1, 2, 1, torch.bfloat16, "l2"),            # a single token
    (1, 4, 700, torch.bfloat16, "l2"),          # eleven chunks
    (2, 2, 150, torch.float32, "l2"),           # fp32: the recurrent kernel
]


@pytest.mark.parametrize("window", [1, 2, 4, 17, 32])
@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c[:3])) + str(c[3])[-4:])
@pytest.mark.parametrize("with_state", [False, True])
def test_falcon3a_chunked_small_shapes(falcon, window, case, with_state):
    B, H, T, dt, phi = case
    x = workloads.random_case(B, H, T, 64, 64, dt, seed=400 + CASES.index(case), device="cuda",
                              with_state=with_state)
    o, S, xl = run3c(falcon, x, window, phi)
    ref = ref3(x, window, phi)
    assert head_err(o, ref["o"]) < TOL[dt]
    assert head_err(S, ref["S"]) < TOL[dt]
    np.testing.assert_allclose(xl.numpy(), ref["x_last"], rtol=2e-6, atol=2e-6)


@pytest.mark.parametrize("ridge", ["given", "scaled"])
def test_falcon3a_chunked_clamp_and_ridge(falcon, ridge):
    """lambda = softplus(n + 3) with gains up to 2: the clamp fires on many
    tokens (decays down to eps_gamma inside a chunk); the scale-coupled ridge
    uses the window energy."""
    x = workloads.random_case(2, 2, 300, 64, 64, torch.bfloat16, seed=277, lam_shift=3.0,
                              device="cuda", with_state=True)
    x["beta"] = torch.full_like(x["beta"], 1.95)
    o, S, _ = run3c(falcon, x, 5, "l2", ridge)
    ref = ref3(x, 5, "l2", ridge)
    assert np.isfinite(o.numpy()).all()
    assert head_err(o, ref["o"]) < 2e-2
    assert head_err(S, ref["S"]) < 2e-2


def test_falcon3a_chunked_matches_recurrent_kernel(falcon):
    """GPU vs GPU on the lm-3A shape: the chunked and the token-recurrent
    kernels agree."""
    w = workloads.LM_3A
    x = workloads.generate(w, device="cuda")
    oc, Sc, _ = run3c(falcon, x, workloads.LM_3A_WINDOW, w.phi)
    o, S, _ = falcon.falcon3a_fwd_recurrent(x["q"], x["k"], x["v"], x["beta"], x["lambda"],
                                            workloads.LM_3A_WINDOW, phi=w.phi)
    assert falcon.falcon_sync_check() == 0
    assert head_err(oc, o.float().cpu()) < 2e-2
    assert head_err(Sc, S.cpu()) < 2e-2


def test_falcon3a_chunked_lm_workload_all_heads(falcon):
    """B8 H12 T2048 d64 bf16, window 4, every head against the oracle."""
    w = workloads.LM_3A
    x = workloads.generate(w, device="cuda")
    o, S, _ = run3c(falcon, x, workloads.LM_3A_WINDOW, w.phi)
    ref = ref3(x, workloads.LM_3A_WINDOW, w.phi)
    assert head_err(o, ref["o"]) < 2e-2
    assert head_err(S, ref["S"]) < 2e-2
