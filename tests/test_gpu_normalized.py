"""GPU parity of Falcon-1A with the normalised read against the fp64 oracle.

o_t = S_t^T phi(q_t) / (z_t^T phi(q_t) + eps_attn), z_t = gamma_t z_{t-1} +
eta_t x_t (page hyper.ai/fr/papers/2608.27763, Section 2.2, Eq. (2.1)-(2.3),
with the Falcon-1A gain and clamped decay on the normaliser).  The inputs
have positive entries, the setting in which the pages call the normalised
read attention-like (a nonnegative normaliser).  Errors are ||err||_F /
||ref||_F per head: 1e-4 for fp32 inputs, 2e-2 for bf16 (o, S_T); z_T is fp32
arithmetic on exact inputs on every path (1e-4).
"""
import numpy as np
import pytest
import torch

import oracle
from delta_rule_attention_gb300 import workloads

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

TOL = {torch.float32: 1e-4, torch.bfloat16: 2e-2}


def head_err(got, ref, head_dims=2):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    g = got.reshape(-1, int(np.prod(got.shape[-head_dims:])))
    r = ref.reshape(g.shape)
    return float((np.linalg.norm(g - r, axis=1) / np.maximum(np.linalg.norm(r, axis=1), 1e-30))
                 .max())


def positive_case(B, H, T, m, dv, dt, seed, carried, lam_shift=-2.0):
    """Seeded inputs with positive q, k (|N(0,1)| + 0.05), carried state and
    normaliser when asked."""
    x = workloads.random_case(B, H, T, m, dv, torch.float32, seed=seed, lam_shift=lam_shift,
                              with_state=carried, with_x_prev=carried)
    x["q"] = (x["q"].abs() + 0.05).to(dt)
    x["k"] = (x["k"].abs() + 0.05).to(dt)
    x["v"] = x["v"].to(dt)
    if carried:
        g = torch.Generator().manual_seed(seed + 7)
        x["z0"] = torch.rand((B, H, m), generator=g) + 0.1
        x["x_prev"] = x["x_prev"].abs()
        x["x_prev"] = x["x_prev"] / x["x_prev"].norm(dim=-1, keepdim=True)
    return {n: t.cuda() for n, t in x.items()}


def run(x, chunk, phi="l2", eps_attn=1e-6):
    import delta_rule_attention_gb300 as falcon
    o, S, z, xl = falcon.falcon1a_fwd_chunked_normalized(
        x["q"], x["k"], x["v"], x["beta"], x["lambda"], S0=x.get("S0"), z0=x.get("z0"),
        x_prev=x.get("x_prev"), eps_attn=eps_attn, chunk=chunk, phi=phi)
    assert falcon.falcon_sync_check() == 0
    return o.float().cpu(), S.cpu(), z.cpu(), xl.cpu()


def ref_of(x, phi="l2", eps_attn=1e-6):
    return oracle.forward_normalized(x["q"], x["k"], x["v"], x["beta"], x["lambda"],
                                     S0=x.get("S0"), z0=x.get("z0"), x_prev=x.get("x_prev"),
                                     phi=phi, eps_attn=eps_attn)


CASES = [
    # B, H, T, m, dv, chunk, dtype, phi
    (1, 2, 64, 16, 16, 16, torch.float32, "identity"),
    (2, 2, 2 * 32 + 17, 32, 64, 32, torch.float32, "l2"),
    (1, 3, 3 * 64 + 5, 64, 64, 64, torch.bfloat16, "l2"),      # tensor-core numerator
    (1, 2, 257, 128, 128, 64, torch.bfloat16, "l2"),           # tensor-core, m = 128
    (2, 2, 100, 64, 32, 64, torch.bfloat16, "rms"),            # generic path, bf16
    (1, 2, 1, 64, 64, 64, torch.bfloat16, "l2"),               # a single token
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c[:6])) + str(c[6])[-4:])
@pytest.mark.parametrize("carried", [False, True])
def test_normalized_read_against_oracle(case, carried):
    B, H, T, m, dv, C, dt, phi = case
    x = positive_case(B, H, T, m, dv, dt, seed=CASES.index(case) + 40, carried=carried)
    eps_attn = 1e-3 if T == 1 and not carried else 1e-6  # token 1 of a fresh sequence: z_1 = 0
    o, S, z, xl = run(x, C, phi, eps_attn)
    ref = ref_of(x, phi, eps_attn)
    assert np.isfinite(o.numpy()).all()
    assert head_err(o, ref["o"]) < TOL[dt]
    assert head_err(S, ref["S"]) < TOL[dt]
    assert head_err(z, ref["z"], 1) < 1e-4
    np.testing.assert_allclose(xl.numpy(), ref["x_last"], rtol=1e-6, atol=1e-6)


def test_normalized_read_with_clamped_decay():
    """lambda = softplus(n + 2), gains near 2: the clamp fires, the decays
    underflow within chunks; tensor-core numerator (bf16, m = d_v = 64)."""
    x = positive_case(1, 3, 300, 64, 64, torch.bfloat16, seed=77, carried=True, lam_shift=2.0)
    x["beta"] = torch.full_like(x["beta"], 1.9)
    o, S, z, _ = run(x, 64)
    ref = ref_of(x)
    assert head_err(o, ref["o"]) < 2e-2
    assert head_err(S, ref["S"]) < 2e-2
    assert head_err(z, ref["z"], 1) < 1e-4


def test_normalized_read_lm_shape_all_heads():
    """B8 H12 T2048 d64 bf16 (the lm workload's shape and ridge) with positive
    q, k: every head compared in full."""
    w = workloads.LM
    x = positive_case(w.B, w.H, w.T, w.m, w.dv, w.dtype, seed=123, carried=False,
                      lam_shift=w.lam_shift)
    o, S, z, _ = run(x, w.chunk)
    ref = ref_of(x)
    assert head_err(o, ref["o"]) < 2e-2
    assert head_err(S, ref["S"]) < 2e-2
    assert head_err(z, ref["z"], 1) < 1e-4


def test_normalized_split_run_equals_full_run():
    """Carrying (S_T, z_T, x_last) across two calls equals one call (fp32)."""
    x = positive_case(2, 2, 200, 32, 32, torch.float32, seed=9, carried=False)
    o_f, S_f, z_f, _ = run(x, 32)
    for T1 in (1, 64, 77):
        a = {n: t[:, :, :T1].contiguous() for n, t in x.items()}
        b = {n: t[:, :, T1:].contiguous() for n, t in x.items()}
        o_a, S_a, z_a, xl_a = run(a, 32)
        b["S0"], b["z0"], b["x_prev"] = S_a.cuda(), z_a.cuda(), xl_a.cuda()
        o_b, S_b, z_b, _ = run(b, 32)
        assert head_err(torch.cat([o_a, o_b], 2), o_f) < 1e-5
        assert head_err(S_b, S_f) < 1e-5
        assert head_err(z_b, z_f, 1) < 1e-5


def test_normalized_read_many_chunks_chain_launch():
    """71 chunks of two heads (bf16, m = d_v = 64, ragged tail): the
    normaliser's chain runs as its own launch, and the tensor-core maps (which
    write the denominator's per-chunk terms) run in chunk ranges."""
    x = positive_case(1, 2, 70 * 64 + 9, 64, 64, torch.bfloat16, seed=61, carried=True)
    o, S, z, _ = run(x, 64)
    ref = ref_of(x)
    assert head_err(o, ref["o"]) < 2e-2
    assert head_err(S, ref["S"]) < 2e-2
    assert head_err(z, ref["z"], 1) < 1e-4


def test_normalized_read_z_out_aliases_z0():
    """z_out given as z0's own buffer (in place) on a few-chunk call: the
    result equals the call with separate buffers."""
    import delta_rule_attention_gb300 as falcon
    x = positive_case(2, 3, 5 * 64 + 11, 64, 64, torch.bfloat16, seed=62, carried=True)
    o_ref, S_ref, z_ref, _ = run(x, 64)
    z_buf = x["z0"].clone()
    o, S, z, _ = falcon.falcon1a_fwd_chunked_normalized(
        x["q"], x["k"], x["v"], x["beta"], x["lambda"], S0=x["S0"], z0=z_buf,
        x_prev=x["x_prev"], z_out=z_buf)
    assert falcon.falcon_sync_check() == 0
    assert z.data_ptr() == z_buf.data_ptr()
    assert torch.equal(z.cpu(), z_ref)
    assert torch.equal(o.float().cpu(), o_ref)
    assert torch.equal(S.cpu(), S_ref)
