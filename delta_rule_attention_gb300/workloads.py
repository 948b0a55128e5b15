"""Seeded synthetic workloads (inputs only; none of the method's arithmetic).

The workloads are shaped like the 124M-130M-parameter language-model
layers of the experiments on the pages (heads of width 64, about 12 heads,
sequence 1024-2048) plus a long-context stress case and a batched decode.
The pages train on FineWeb-Edu and evaluate on lm-eval tasks and a digit-
addition set; no dataset or trained weight is used here: q, k, v are iid
N(0, 1), and the gain and ridge are fixed transforms of N(0, 1) draws:

    beta_t   = 2 * sigmoid(n)          (in (0, 2), as the pages require)
    lambda_t = softplus(n + shift)     (>= 0)

Draw order for one workload: q, k, v, then the beta normals, then the lambda
normals, all in float32 row-major [B, H, T, .] from one torch.Generator seeded
with the workload's seed; q, k, v are then rounded to the workload dtype.  The
per-column workloads (Falcon-2, Falcon-2A) draw one beta normal per value
column, [B, H, T, d_v], in the same place of the order.
Workloads small enough for the host (tiny, lm, lm-1A, lm-2, lm-2A, lm-3A) draw on the CPU
generator, so they are the same on every machine; the long-context and decode
workloads (hundreds of millions of draws) draw on the device's generator.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    rule: str             # "falcon1" | "falcon1a"
    B: int
    H: int
    T: int
    m: int
    dv: int
    dtype: torch.dtype
    phi: str
    chunk: int
    lam_shift: float
    seed: int
    lambda_first_zero: bool = False
    host_rng: bool = True
    eps: float = 1e-6
    eps_gamma: float = 1e-6
    per_column: bool = False  # Falcon-2/2A: one gain per value column, beta [B, H, T, dv]

    @property
    def tokens(self) -> int:
        return self.B * self.T


TINY = Workload("falcon1_tiny_B1H2T64_d16_f32", "falcon1", 1, 2, 64, 16, 16, torch.float32,
                "identity", 16, -2.0, 0, lambda_first_zero=True)
LM = Workload("falcon1_lm_B8H12T2048_d64_bf16", "falcon1", 8, 12, 2048, 64, 64, torch.bfloat16,
              "l2", 64, -3.0, 1)
LM_1A = Workload("falcon1a_lm_B8H12T2048_d64_bf16", "falcon1a", 8, 12, 2048, 64, 64,
                 torch.bfloat16, "l2", 64, -3.0, 2)
LONG = Workload("falcon1_long_B1H16T65536_d128_bf16", "falcon1", 1, 16, 65536, 128, 128,
                torch.bfloat16, "l2", 64, 1.0, 3, host_rng=False)
# Falcon-2 / Falcon-2A (per-column step sizes) on the lm shape.
LM_2 = Workload("falcon2_lm_B8H12T2048_d64_bf16", "falcon2", 8, 12, 2048, 64, 64, torch.bfloat16,
                "l2", 64, -3.0, 5, per_column=True)
LM_2A = Workload("falcon2a_lm_B8H12T2048_d64_bf16", "falcon2a", 8, 12, 2048, 64, 64,
                 torch.bfloat16, "l2", 64, -3.0, 6, per_column=True)
# Falcon-3A (sliding window of 4 write pairs: the pages give no window for
# their runs; 4 is the reading taken) on the lm shape.
LM_3A = Workload("falcon3a_lm_B8H12T2048_d64_bf16_w4", "falcon3a", 8, 12, 2048, 64, 64,
                 torch.bfloat16, "l2", 64, -3.0, 7)
LM_3A_WINDOW = 4
WORKLOADS = {w.name: w for w in (TINY, LM, LM_1A, LONG, LM_2, LM_2A, LM_3A)}


@dataclass(frozen=True)
class DecodeWorkload:
    name: str = "falcon1_decode_N8192_d128_bf16"
    n_seq: int = 256
    H: int = 32
    m: int = 128
    dv: int = 128
    steps: int = 4096
    dtype: torch.dtype = torch.bfloat16
    phi: str = "l2"
    lam_shift: float = -3.0
    s0_std: float = 0.1     # S0 ~ N(0, 0.1^2): 0.1 read as a standard deviation
    seed: int = 4
    eps: float = 1e-6
    eps_gamma: float = 1e-6

    @property
    def N(self) -> int:
        return self.n_seq * self.H


DECODE = DecodeWorkload()


def gain_and_ridge(nb: torch.Tensor, nl: torch.Tensor, lam_shift: float):
    """beta = 2 sigmoid(n), lambda = softplus(n + shift): the workload recipe."""
    return 2.0 * torch.sigmoid(nb), torch.nn.functional.softplus(nl + lam_shift)


def generate(w: Workload, device="cpu"):
    """Inputs of a chunked-forward workload as a dict of tensors on `device`."""
    gen_dev = "cpu" if w.host_rng else device
    g = torch.Generator(device=gen_dev)
    g.manual_seed(w.seed)
    B, H, T, m, dv = w.B, w.H, w.T, w.m, w.dv
    q = torch.randn((B, H, T, m), generator=g, device=gen_dev)
    k = torch.randn((B, H, T, m), generator=g, device=gen_dev)
    v = torch.randn((B, H, T, dv), generator=g, device=gen_dev)
    nb = torch.randn((B, H, T, dv) if w.per_column else (B, H, T), generator=g, device=gen_dev)
    nl = torch.randn((B, H, T), generator=g, device=gen_dev)
    beta, lam = gain_and_ridge(nb, nl, w.lam_shift)
    if w.lambda_first_zero and T > 0:
        lam[..., 0] = 0.0
    out = {"q": q.to(w.dtype), "k": k.to(w.dtype), "v": v.to(w.dtype),
           "beta": beta.contiguous(), "lambda": lam.contiguous()}
    return {n: t.to(device).contiguous() for n, t in out.items()}


def random_case(B, H, T, m, dv, dtype=torch.float32, seed=0, lam_shift=-2.0, device="cpu",
                with_state=False, with_x_prev=False, per_column=False):
    """Small seeded case for parity tests of arbitrary shape (CPU generator);
    per_column draws one gain per value column (beta [B, H, T, dv])."""
    g = torch.Generator().manual_seed(seed)
    q = torch.randn((B, H, T, m), generator=g)
    k = torch.randn((B, H, T, m), generator=g)
    v = torch.randn((B, H, T, dv), generator=g)
    beta, lam = gain_and_ridge(torch.randn((B, H, T, dv) if per_column else (B, H, T),
                                           generator=g),
                               torch.randn((B, H, T), generator=g), lam_shift)
    out = {"q": q.to(dtype), "k": k.to(dtype), "v": v.to(dtype), "beta": beta, "lambda": lam}
    if with_state:
        out["S0"] = 0.5 * torch.randn((B, H, m, dv), generator=g)
    if with_x_prev:
        xp = torch.randn((B, H, m), generator=g)
        out["x_prev"] = xp / xp.norm(dim=-1, keepdim=True)
    return {n: t.to(device).contiguous() for n, t in out.items()}


def cotangents(B, H, T, m, dv, dtype=torch.float32, seed=0, device="cpu", ends=False):
    """Seeded cotangents for the backward pass: dO [B,H,T,dv] N(0,1) in `dtype`
    and, with ``ends``, dS_T [B,H,m,dv] and dx_last [B,H,m] N(0,1) fp32 (a
    training step on a fresh, final segment has zero end cotangents)."""
    g = torch.Generator().manual_seed(10_000 + seed)
    out = {"dO": torch.randn((B, H, T, dv), generator=g).to(dtype)}
    if ends:
        out["dS_T"] = torch.randn((B, H, m, dv), generator=g)
        out["dx_last"] = torch.randn((B, H, m), generator=g)
    return {n: t.to(device).contiguous() for n, t in out.items()}


class DecodeStream:
    """Per-step inputs of the decode workload, drawn step after step from one
    generator on `device` (the initial state first, then for every step q, k,
    v, the beta normals and the lambda normals)."""

    def __init__(self, w: DecodeWorkload = DECODE, device="cuda"):
        self.w = w
        self.device = device
        self.g = torch.Generator(device=device)
        self.g.manual_seed(w.seed)

    def initial_state(self):
        w = self.w
        return w.s0_std * torch.randn((w.N, w.m, w.dv), generator=self.g, device=self.device)

    def step(self):
        w = self.w
        q = torch.randn((w.N, w.m), generator=self.g, device=self.device).to(w.dtype)
        k = torch.randn((w.N, w.m), generator=self.g, device=self.device).to(w.dtype)
        v = torch.randn((w.N, w.dv), generator=self.g, device=self.device).to(w.dtype)
        nb = torch.randn((w.N,), generator=self.g, device=self.device)
        nl = torch.randn((w.N,), generator=self.g, device=self.device)
        beta, lam = gain_and_ridge(nb, nl, w.lam_shift)
        return {"q": q, "k": k, "v": v, "beta": beta, "lambda": lam}
