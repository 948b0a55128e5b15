"""GPU parity of the chunked Falcon-2A forward (falcon2a_fwd_chunked: per-column
decays in chunk form on the tensor cores for bf16 m = d_v = 64, the
token-recurrent kernel otherwise) against the fp64 oracle, through the C ABI.
Error measure as in test_gpu_parity.py: ||err||_F / ||ref||_F per head, max
over heads; <= 1e-4 for fp32 inputs, <= 2e-2 for bf16 inputs."""
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


def run2c(falcon, x, phi="l2", ridge="given"):
    o, S, xl = falcon.falcon2a_fwd_chunked(x["q"], x["k"], x["v"], x["beta"], x["lambda"],
                                           S0=x.get("S0"), x_prev=x.get("x_prev"), phi=phi,
                                           ridge=ridge)
    assert falcon.falcon_sync_check() == 0
    return o.float().cpu(), S.cpu(), xl.cpu()


def ref2(x, phi="l2", ridge="given"):
    return oracle.forward2("falcon2a", x["q"], x["k"], x["v"], x["beta"], x["lambda"],
                           S0=x.get("S0"), x_prev=x.get("x_prev"), phi=phi, ridge=ridge)


CASES = [
    # B, H, T, dtype, phi (m = d_v = 64; bf16: tensor cores, fp32: recurrent)
    (2, 3, 3 * 64 + 5, torch.bfloat16, "l2"),   # several chunks, ragged tail
    (1, 2, 64, torch.bfloat16, "identity"),     # exactly one chunk
    (1, 2, 65, torch.bfloat16, "rms"),          # one token into the second chunk
    (3, 2, 7, torch.bfloat16, "l2"),            # shorter than a chunk
    (1, 2, 1, torch.bfloat16, "l2"),            # a single token
    (1, 4, 700, torch.bfloat16, "l2"),          # eleven chunks
    (2, 2, 150, torch.float32, "l2"),           # fp32: the recurrent kernel
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c[:3])) + str(c[3])[-4:])
@pytest.mark.parametrize("carried", [False, True])
def test_falcon2a_chunked_small_shapes(falcon, case, carried):
    B, H, T, dt, phi = case
    x = workloads.random_case(B, H, T, 64, 64, dt, seed=500 + CASES.index(case), device="cuda",
                              with_state=carried, with_x_prev=carried, per_column=True)
    o, S, xl = run2c(falcon, x, phi)
    ref = ref2(x, phi)
    assert head_err(o, ref["o"]) < TOL[dt]
    assert head_err(S, ref["S"]) < TOL[dt]
    np.testing.assert_allclose(xl.numpy(), ref["x_last"], rtol=2e-6, atol=2e-6)


@pytest.mark.parametrize("ridge", ["given", "scaled"])
@pytest.mark.parametrize("lam_shift", [-1.0, 3.0])
def test_falcon2a_chunked_decay_and_ridge(falcon, ridge, lam_shift):
    """lam_shift 3 with gains up to 2: the clamp fires on most (token, column)
    pairs, chunk decay spans far beyond the factored range (the CUDA-core
    form of the intra-chunk part); the scale-coupled ridge uses ||x_t||^2."""
    x = workloads.random_case(2, 2, 300, 64, 64, torch.bfloat16, seed=577, lam_shift=lam_shift,
                              device="cuda", with_state=True, with_x_prev=True, per_column=True)
    if lam_shift > 0:
        x["beta"] = torch.full_like(x["beta"], 1.95)
    o, S, _ = run2c(falcon, x, "l2", ridge)
    ref = ref2(x, "l2", ridge)
    assert np.isfinite(o.numpy()).all()
    assert head_err(o, ref["o"]) < 2e-2
    assert head_err(S, ref["S"]) < 2e-2


def test_falcon2a_chunked_matches_recurrent_and_oracle_lm(falcon):
    """B8 H12 T2048 d64 bf16, one gain per column: every head against the
    oracle, and against the token-recurrent kernel."""
    w = workloads.LM_2A
    x = workloads.generate(w, device="cuda")
    o, S, _ = run2c(falcon, x, w.phi)
    ref = ref2(x, w.phi)
    assert head_err(o, ref["o"]) < 2e-2
    assert head_err(S, ref["S"]) < 2e-2
    orr, Sr, _ = falcon.falcon2a_fwd_recurrent(x["q"], x["k"], x["v"], x["beta"], x["lambda"],
                                               phi=w.phi)
    assert falcon.falcon_sync_check() == 0
    assert head_err(o, orr.float().cpu()) < 2e-2
    assert head_err(S, Sr.cpu()) < 2e-2
