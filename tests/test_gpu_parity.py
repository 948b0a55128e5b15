"""GPU parity: the CUDA library (through the C ABI) against the fp64 oracle.

Error measure: ||err||_F / ||ref||_F per head, for o over (T x dv) and for the
final state over (m x dv); the maximum over heads must stay within 1e-4 for
fp32 inputs and 2e-2 for bf16 inputs (fp32 accumulation).  Both sides see the
same seeded, already-rounded inputs.
"""
import numpy as np
import pytest
import torch

import oracle
from delta_rule_attention_gb300 import workloads

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

TOL = {torch.float32: 1e-4, torch.bfloat16: 2e-2}


@pytest.fixture(scope="module")
def falcon():
    import delta_rule_attention_gb300 as f
    f.load_library()
    return f


def head_err(got, ref, head_dims=2):
    """max over heads of ||got - ref||_F / ||ref||_F; the last `head_dims`
    dims form one head's block."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    g = got.reshape(-1, int(np.prod(got.shape[-head_dims:])))
    r = ref.reshape(g.shape)
    num = np.linalg.norm(g - r, axis=1)
    den = np.maximum(np.linalg.norm(r, axis=1), 1e-30)
    return float((num / den).max())


def run(falcon, rule, x, chunk, phi, eps=1e-6, eps_gamma=1e-6):
    fn = falcon.falcon1_fwd_chunked if rule == "falcon1" else falcon.falcon1a_fwd_chunked
    o, S, xl = fn(x["q"], x["k"], x["v"], x["beta"], x["lambda"], S0=x.get("S0"),
                  x_prev=x.get("x_prev"), chunk=chunk, phi=phi, eps=eps, eps_gamma=eps_gamma)
    assert falcon.falcon_sync_check() == 0
    return o.float().cpu(), S.cpu(), xl.cpu()


def ref_of(rule, x, phi, eps=1e-6, eps_gamma=1e-6):
    return oracle.forward(rule, x["q"], x["k"], x["v"], x["beta"], x["lambda"],
                          S0=x.get("S0"), x_prev=x.get("x_prev"), phi=phi, eps=eps,
                          eps_gamma=eps_gamma)


CASES = [
    # B, H, T, m, dv, chunk, dtype, phi
    (1, 2, 64, 16, 16, 16, torch.float32, "identity"),
    (2, 3, 3 * 64 + 5, 64, 64, 64, torch.bfloat16, "l2"),
    (1, 2, 2 * 32 + 17, 32, 128, 32, torch.float32, "l2"),
    (2, 1, 100, 128, 32, 64, torch.bfloat16, "l2"),
    (1, 3, 257, 128, 128, 64, torch.bfloat16, "l2"),
    (1, 2, 40, 16, 64, 16, torch.float32, "identity"),
    (3, 2, 7, 64, 16, 64, torch.float32, "l2"),       # shorter than one chunk
    (3, 2, 7, 64, 64, 64, torch.bfloat16, "l2"),      # tensor-core path, one partial chunk
    (1, 2, 1, 64, 64, 64, torch.bfloat16, "l2"),      # a single token
    (2, 2, 4 * 64, 64, 64, 64, torch.bfloat16, "identity"),
]


@pytest.mark.parametrize("rule", ["falcon1", "falcon1a"])
@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c[:6])) + str(c[6])[-4:])
@pytest.mark.parametrize("carried", [False, True])
def test_small_shapes_against_oracle(falcon, rule, case, carried):
    B, H, T, m, dv, C, dt, phi = case
    x = workloads.random_case(B, H, T, m, dv, dt, seed=CASES.index(case), device="cuda",
                              with_state=carried, with_x_prev=carried)
    o, S, xl = run(falcon, rule, x, C, phi)
    ref = ref_of(rule, x, phi)
    assert head_err(o, ref["o"]) < TOL[dt]
    assert head_err(S, ref["S"]) < TOL[dt]
    np.testing.assert_allclose(xl.numpy(), ref["x_last"], rtol=1e-6, atol=1e-6)


@pytest.mark.parametrize("rule", ["falcon1", "falcon1a"])
def test_clamp_active_large_ridge(falcon, rule):
    """lambda = softplus(n + 3): the decay clamp fires on many tokens and
    chunk decay products underflow; o and S stay finite and match."""
    x = workloads.random_case(2, 2, 300, 64, 64, torch.float32, seed=77, lam_shift=3.0,
                              device="cuda", with_state=True)
    x["beta"] = torch.full_like(x["beta"], 1.95)
    o, S, _ = run(falcon, rule, x, 64, "l2")
    ref = ref_of(rule, x, "l2")
    assert np.isfinite(o.numpy()).all() and np.isfinite(S.numpy()).all()
    assert head_err(o, ref["o"]) < 1e-4
    assert head_err(S, ref["S"]) < 1e-4


def _chunk_log_decay_spans(x, chunk, phi):
    """-(sum of log gamma_t) over every chunk of every head, and the share of
    tokens on the clamped branch, from the inputs by the step-size and clamp
    definitions (test-data check only)."""
    k = x["k"].double().cpu().numpy()
    if phi == "l2":
        k = k / np.maximum(np.linalg.norm(k, axis=-1, keepdims=True), 1e-12)
    xs = np.zeros_like(k)
    xs[..., 1:, :] = k[..., :-1, :]
    if x.get("x_prev") is not None:
        xs[..., 0, :] = x["x_prev"].double().cpu().numpy()
    E = (xs ** 2).sum(-1)
    beta, lam = x["beta"].double().cpu().numpy(), x["lambda"].double().cpu().numpy()
    eta = beta / (E + lam + 1e-6)
    if x.get("x_prev") is None:
        eta[..., 0] = 0.0
    a = np.minimum(eta * lam, 1.0 - 1e-6)
    lg = np.log1p(-a)
    T = lg.shape[-1]
    pad = (-T) % chunk
    lg = np.concatenate([lg, np.zeros(lg.shape[:-1] + (pad,))], -1)
    spans = -lg.reshape(lg.shape[:-1] + (-1, chunk)).sum(-1)
    return spans, float((eta * lam >= 1.0 - 1e-6).mean())


@pytest.mark.parametrize("rule", ["falcon1", "falcon1a"])
@pytest.mark.parametrize("m", [64, 128])
def test_tensor_core_strong_decay(falcon, rule, m):
    """bf16, m = d_v in {64, 128}, chunk 64 (the tensor-core forward) with gains
    near 2 and ridges that make the clamp fire: head 0 keeps the workload's
    mild ridge (chunk log-decay spans near 10: the factored decay form), heads
    1 and 2 take lambda = softplus(n + 1) and softplus(n + 3) (spans far above
    80: per-element decays of non-positive exponents).  Carried state and
    x_prev, ragged T; o, S_T and x_last against the oracle."""
    T = 4 * 64 + 29
    x = workloads.random_case(1, 3, T, m, m, torch.bfloat16, seed=400 + m, device="cuda",
                              with_state=True, with_x_prev=True)
    g = torch.Generator().manual_seed(500 + m)
    n_l = torch.randn((1, 3, T), generator=g)
    shift = torch.tensor([-3.0, 1.0, 3.0]).view(1, 3, 1)
    x["lambda"] = torch.nn.functional.softplus(n_l + shift).cuda()
    x["beta"] = (1.9 + 0.09 * torch.tanh(torch.randn((1, 3, T), generator=g))).cuda()
    spans, clamped = _chunk_log_decay_spans(x, 64, "l2")
    assert spans[0, 0].max() < 80.0 and spans[0, 1:].min() > 80.0
    assert clamped > 0.05
    o, S, xl = run(falcon, rule, x, 64, "l2")
    ref = ref_of(rule, x, "l2")
    assert np.isfinite(o.numpy()).all() and np.isfinite(S.numpy()).all()
    assert head_err(o, ref["o"]) < 2e-2
    assert head_err(S, ref["S"]) < 2e-2
    np.testing.assert_allclose(xl.numpy(), ref["x_last"], rtol=1e-6, atol=1e-6)


def test_tiny_workload(falcon):
    """Falcon-1 tiny: B1 H2 T64 d16 fp32, phi = identity, lambda_1 = 0, C = 16."""
    w = workloads.TINY
    x = workloads.generate(w, device="cuda")
    o, S, _ = run(falcon, w.rule, x, w.chunk, w.phi)
    ref = ref_of(w.rule, x, w.phi)
    assert head_err(o, ref["o"]) < 1e-4
    assert head_err(S, ref["S"]) < 1e-4


@pytest.mark.parametrize("w", [workloads.LM, workloads.LM_1A], ids=lambda w: w.name)
def test_lm_workloads_all_heads(falcon, w):
    """B8 H12 T2048 d64 bf16, every head compared in full."""
    x = workloads.generate(w, device="cuda")
    o, S, _ = run(falcon, w.rule, x, w.chunk, w.phi)
    ref = ref_of(w.rule, x, w.phi)
    assert head_err(o, ref["o"]) < 2e-2
    assert head_err(S, ref["S"]) < 2e-2


def test_long_context_all_heads(falcon):
    """B1 H16 T65536 d128 bf16 with lambda = softplus(n + 1) (the decay
    underflow stress case): whole run on the GPU, every head recomputed by the
    oracle in full."""
    import os
    w = workloads.LONG
    x = workloads.generate(w, device="cuda")
    o, S, xl = run(falcon, w.rule, x, w.chunk, w.phi)
    sub = {n: t.cpu() for n, t in x.items()}
    ref = oracle.forward(w.rule, sub["q"], sub["k"], sub["v"], sub["beta"], sub["lambda"],
                         phi=w.phi, threads=min(16, os.cpu_count() or 1))
    assert np.isfinite(o.numpy()).all()
    assert head_err(o, ref["o"]) < 2e-2
    assert head_err(S, ref["S"]) < 2e-2
    np.testing.assert_allclose(xl.numpy(), ref["x_last"], rtol=1e-6, atol=1e-6)


def test_decode_workload_one_state_per_cta(falcon):
    """256 x 32 states, d128, fp32 state, 4096 bf16 steps; the first step is a
    sequence start (sentinel).  The persistent kernel strides the states over
    one CTA per SM, so the states followed by the oracle include one of every
    CTA (at different depths of its stride) and the two of the ragged last
    round; each is checked over all 4096 steps (the oracle runs them as
    sequences: a decode loop from a fresh start is the sequence recurrence)."""
    import os
    w = workloads.DECODE
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    rounds = w.N // sms
    pick = sorted({c + sms * (c % rounds) for c in range(sms)} | {w.N - 2, w.N - 1})
    assert len(pick) >= sms
    pick_d = torch.tensor(pick, device="cuda")
    stream = workloads.DecodeStream(w, device="cuda")
    S = stream.initial_state()
    S0_pick = S[pick_d].cpu()
    xp = torch.zeros((w.N, w.m), device="cuda")
    fresh_all = torch.ones(w.N, dtype=torch.uint8, device="cuda")
    seq = {n: [] for n in ("q", "k", "v", "beta", "lambda")}
    outs = []
    for s in range(w.steps):
        x = stream.step()
        o = falcon.falcon1_decode_step(x["q"], x["k"], x["v"], x["beta"], x["lambda"], S, xp,
                                       fresh=fresh_all if s == 0 else None, phi=w.phi,
                                       eps=w.eps, eps_gamma=w.eps_gamma)
        for n in seq:
            seq[n].append(x[n][pick_d])
        outs.append(o[pick_d])
    assert falcon.falcon_sync_check() == 0
    # [P, steps, ...]: one sequence per followed state
    seqs = {n: torch.stack(t, 1).cpu() for n, t in seq.items()}
    o_got = torch.stack(outs, 1).float().cpu()
    ref = oracle.forward("falcon1", seqs["q"], seqs["k"], seqs["v"], seqs["beta"],
                         seqs["lambda"], S0=S0_pick, phi=w.phi, eps=w.eps,
                         eps_gamma=w.eps_gamma, threads=min(16, os.cpu_count() or 1))
    assert head_err(o_got, ref["o"]) < 2e-2
    assert head_err(S[pick_d].cpu(), ref["S"]) < 2e-2
    np.testing.assert_allclose(xp[pick_d].cpu().numpy(), ref["x_last"], rtol=1e-5, atol=1e-6)


@pytest.mark.parametrize("rule", ["falcon1", "falcon1a"])
@pytest.mark.parametrize("dt", [torch.float32, torch.bfloat16])
def test_decode_small_against_oracle(falcon, rule, dt):
    N, m, dv, T = 6, 32, 64, 9
    x = workloads.random_case(1, N, T, m, dv, dt, seed=91, device="cuda", with_state=True)
    S = x["S0"][0].clone()
    xp = torch.zeros((N, m), device="cuda")
    S_ref = S.double().cpu().numpy().copy()
    xp_ref = np.zeros((N, m))
    fn = falcon.falcon1_decode_step if rule == "falcon1" else falcon.falcon1a_decode_step
    fresh = torch.tensor([1, 0, 1, 0, 1, 1], dtype=torch.uint8, device="cuda")
    for t in range(T):
        args = [x[n][0, :, t].contiguous() for n in ("q", "k", "v", "beta", "lambda")]
        o = fn(*args, S, xp, fresh=fresh if t == 0 else None)
        o_ref = oracle.decode_step(rule, *[a.cpu() for a in args], S_ref, xp_ref,
                                   fresh=fresh.cpu().numpy() if t == 0 else None)
        assert head_err(o.float().cpu(), o_ref, 1) < TOL[dt]
    assert falcon.falcon_sync_check() == 0
    assert head_err(S.cpu(), S_ref) < TOL[dt]


@pytest.mark.parametrize("m,dv", [(64, 64), (128, 64), (64, 128), (128, 32), (32, 128),
                                  (128, 128), (16, 64), (32, 32), (16, 16), (32, 16),
                                  (16, 128)])
@pytest.mark.parametrize("dt", [torch.float32, torch.bfloat16])
def test_decode_many_states_per_cta(falcon, m, dv, dt):
    """Many states per persistent CTA (64 MB of state, or 4 per SM at least)
    with a ragged last round: every state after three steps against the
    oracle.  Fresh states at the first step get NaN in x_prev, which the
    sentinel must ignore (x_t = 0)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    N = max(sms * 4, (1 << 26) // (m * dv * 4)) + 37
    g = torch.Generator().manual_seed(m * 1000 + dv)
    S = (0.3 * torch.randn((N, m, dv), generator=g)).cuda()
    xp = torch.randn((N, m), generator=g)
    xp = (xp / xp.norm(dim=-1, keepdim=True)).cuda()
    fresh = (torch.rand(N, generator=g) < 0.3).to(torch.uint8)
    xp_ref = xp.double().cpu().numpy().copy()
    xp_ref[fresh.numpy() != 0] = 0.0
    xp[fresh.cuda() != 0] = float("nan")
    S_ref = S.double().cpu().numpy().copy()
    fresh = fresh.cuda()
    for step in range(3):
        q, k, v = (torch.randn((N, d), generator=g).to(dt).cuda() for d in (m, m, dv))
        beta = (2 * torch.sigmoid(torch.randn(N, generator=g))).cuda()
        lam = torch.nn.functional.softplus(torch.randn(N, generator=g) - 1.0).cuda()
        f = fresh if step == 0 else None
        o = falcon.falcon1_decode_step(q, k, v, beta, lam, S, xp, fresh=f)
        o_ref = oracle.decode_step("falcon1", q, k, v, beta, lam, S_ref, xp_ref,
                                   fresh=None if f is None else f.cpu().numpy())
        assert head_err(o.float().cpu(), o_ref, head_dims=1) < TOL[dt]
    assert falcon.falcon_sync_check() == 0
    assert head_err(S.cpu(), S_ref) < TOL[dt]
    np.testing.assert_allclose(xp.cpu().numpy(), xp_ref, rtol=2e-6, atol=2e-6)


@pytest.mark.parametrize("rule", ["falcon1", "falcon1a"])
def test_decode_loop_equals_chunked(falcon, rule):
    """GPU vs GPU: T single-token steps (fresh at the first) reproduce the
    chunked forward."""
    B, H, T, m, dv = 1, 4, 80, 64, 64
    x = workloads.random_case(B, H, T, m, dv, torch.float32, seed=5, device="cuda",
                              with_state=True)
    o_c, S_c, xl_c = run(falcon, rule, x, 32, "l2")
    fn = falcon.falcon1_decode_step if rule == "falcon1" else falcon.falcon1a_decode_step
    S = x["S0"][0].clone()
    xp = torch.zeros((H, m), device="cuda")
    outs = []
    for t in range(T):
        args = [x[n][0, :, t].contiguous() for n in ("q", "k", "v", "beta", "lambda")]
        fresh = torch.ones(H, dtype=torch.uint8, device="cuda") if t == 0 else None
        outs.append(fn(*args, S, xp, fresh=fresh).cpu())
    o_d = torch.stack(outs, 1)[None]
    assert head_err(o_d, o_c) < 1e-4
    assert head_err(S.cpu()[None], S_c) < 1e-4
    np.testing.assert_allclose(xp.cpu().numpy()[None], xl_c.numpy(), rtol=1e-6, atol=1e-7)


@pytest.mark.parametrize("rule", ["falcon1", "falcon1a"])
def test_split_run_equals_full_run(falcon, rule):
    """Carrying (S_T, x_last) across two calls equals one call (the exact
    continuation state of Falcon-1/1A)."""
    x = workloads.random_case(2, 2, 200, 64, 32, torch.float32, seed=9, device="cuda")
    o_f, S_f, xl_f = run(falcon, rule, x, 64, "l2")
    for T1 in (1, 64, 77):
        a = {n: t[:, :, :T1].contiguous() for n, t in x.items()}
        b = {n: t[:, :, T1:].contiguous() for n, t in x.items()}
        o_a, S_a, xl_a = run(falcon, rule, a, 64, "l2")
        b["S0"], b["x_prev"] = S_a.cuda(), xl_a.cuda()
        o_b, S_b, xl_b = run(falcon, rule, b, 64, "l2")
        assert head_err(torch.cat([o_a, o_b], 2), o_f) < 1e-5
        assert head_err(S_b, S_f) < 1e-5
        np.testing.assert_array_equal(xl_b.numpy(), xl_f.numpy())


@pytest.mark.parametrize("rule", ["falcon1", "falcon1a"])
def test_chunk_size_changes_only_rounding(falcon, rule):
    x = workloads.random_case(1, 3, 190, 32, 32, torch.float32, seed=13, device="cuda",
                              with_state=True)
    res = [run(falcon, rule, x, C, "l2") for C in (16, 32, 64)]
    for o, S, _ in res[1:]:
        assert head_err(o, res[0][0]) < 1e-5
        assert head_err(S, res[0][1]) < 1e-5


def test_zero_length_and_inplace_state(falcon):
    """T = 0 returns S0 and x_prev; S_out may alias S0."""
    x = workloads.random_case(1, 2, 0, 16, 16, torch.float32, seed=3, device="cuda",
                              with_state=True, with_x_prev=True)
    o, S, xl = run(falcon, "falcon1", x, 16, "l2")
    assert o.numel() == 0
    np.testing.assert_array_equal(S.numpy(), x["S0"].cpu().numpy())
    np.testing.assert_array_equal(xl.numpy(), x["x_prev"].cpu().numpy())
    x = workloads.random_case(1, 2, 50, 16, 16, torch.float32, seed=4, device="cuda",
                              with_state=True)
    ref = ref_of("falcon1", x, "l2")
    S_io = x["S0"].clone()
    falcon.falcon1_fwd_chunked(x["q"], x["k"], x["v"], x["beta"], x["lambda"], S0=S_io,
                               chunk=16, S_out=S_io)
    assert falcon.falcon_sync_check() == 0
    assert head_err(S_io.cpu(), ref["S"]) < 1e-4


def test_zero_denominator_is_a_no_op(falcon):
    """eps = 0, lambda = 0 and a zero key make the step-size denominator
    vanish for the next token: eta := 0, no write (Eq. (3.4))."""
    x = workloads.random_case(1, 1, 20, 16, 16, torch.float32, seed=8, device="cuda",
                              with_state=True)
    x["lambda"].zero_()
    x["k"][:, :, 4] = 0
    o, S, _ = run(falcon, "falcon1", x, 16, "identity", eps=0.0)
    ref = ref_of("falcon1", x, "identity", eps=0.0)
    assert np.isfinite(o.numpy()).all()
    assert head_err(o, ref["o"]) < 1e-4
    assert head_err(S, ref["S"]) < 1e-4


@pytest.mark.parametrize("rule", ["falcon1", "falcon1a"])
@pytest.mark.parametrize("m", [64, 128])
def test_chunk_range_pieces(falcon, rule, m):
    """Few heads and many chunks: the call runs as chunk-range pieces (maps on
    the caller's stream, scans on a second stream, the running state through
    S_out).  Ragged tail, carried state and x_prev, and S_out aliasing S0."""
    T = 64 * 64 + 17
    x = workloads.random_case(1, 2, T, m, m, torch.bfloat16, seed=300 + m, device="cuda",
                              with_state=True, with_x_prev=True)
    ref = ref_of(rule, x, "l2")
    S_alias = x["S0"].clone()
    fn = falcon.falcon1_fwd_chunked if rule == "falcon1" else falcon.falcon1a_fwd_chunked
    o, S, xl = fn(x["q"], x["k"], x["v"], x["beta"], x["lambda"], S0=S_alias,
                  x_prev=x["x_prev"], chunk=64, phi="l2", S_out=S_alias)
    assert falcon.falcon_sync_check() == 0
    assert S.data_ptr() == S_alias.data_ptr()
    assert head_err(o.float().cpu(), ref["o"]) < 2e-2
    assert head_err(S.cpu(), ref["S"]) < 2e-2
    np.testing.assert_allclose(xl.cpu().numpy(), ref["x_last"], rtol=1e-6, atol=1e-6)
