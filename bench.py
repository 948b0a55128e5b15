"""Benchmark: Falcon-1 chunked forward, B8 H12 T2048 d64 bf16 (tokens/s).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step is one pass of the whole hot path over one batch: the Falcon-1
chunk-parallel forward on the B=8, H=12, T=2048, m=dv=64, bf16 workload
(tokens = B*T per step), inputs resident in HBM.  Under torchrun every rank
runs the same per-rank workload on its own GPU (independent problems, no
data-path collective: weak scaling); the time is the max over ranks.

The line also carries
  e2e          the same metric through the public API from pinned host
               buffers, with host->device inputs and device->host outputs
               inside the timed region;
  roofline     achieved algorithmic HBM bytes per launch / launch time of
               the dominant kernel against the measured copy bandwidth;
  cpu_baseline the fp64 oracle on this host's cores on a bounded sample;
  also         the other workloads (Falcon-1A, long context, Falcon-2 and Falcon-2A
               in chunk form, Falcon-3A, Falcon-1A with the normalised read, the
               backward, decode).

`--impl reference` times the fp64 CPU oracle (the only reference this method
has) on the same workload: the whole lm workload (all 96 heads) per step.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from delta_rule_attention_gb300 import workloads  # noqa: E402

L2_BYTES = 129 * 1024 * 1024
METRIC = "Falcon-1 chunked fwd tokens/s (B8 H12 T2048 d64 bf16) and % of roofline"


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"], "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "fallback"}


# The sources that define the headline path's two kernels (the tensor-core
# map and scan launches): profiled counters are tied to them.
TC_PATH_SOURCES = ("chunk_tc.cu", "tc_ptx.cuh", "tc_util.cuh", "tmap.cu", "tmap.cuh",
                   "common.cuh")


def kernel_sources_digest():
    """sha256 over the headline path's CUDA sources, to tie profiled counters
    to them."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "delta_rule_attention_gb300", "csrc")
    for name in TC_PATH_SOURCES:
        h.update(name.encode())
        h.update(open(os.path.join(csrc, name), "rb").read())
    return h.hexdigest()


def profiled_traffic():
    """DRAM bytes per call (read + write, both launches) from the committed ncu
    summary, or None when the kernels changed since it was taken."""
    p = os.path.join(ROOT, "profiles", "falcon1_fwd_chunked_lm_traffic.txt")
    if not os.path.exists(p):
        return None
    fields = {}
    for line in open(p):
        parts = line.split()
        if len(parts) == 2 and not line.startswith("#"):
            fields[parts[0]] = parts[1]
    if fields.get("csrc_sha256") != kernel_sources_digest():
        return None
    return float(fields["dram_bytes_per_call"])


def algorithmic_bytes(w, with_S0=False):
    """Bytes one forward call must move: q, k, v read, beta, lambda read (beta
    per value column for Falcon-2/2A), o written, S_T (and x_last) written, S0
    read if given."""
    es = torch.finfo(w.dtype).bits // 8
    BH = w.B * w.H
    gains = 4 * w.dv if w.per_column else 4  # beta per value column (Falcon-2/2A) or per token
    b = BH * w.T * (2 * w.m + w.dv) * es + BH * w.T * (gains + 4) + BH * w.T * w.dv * es
    b += BH * w.m * w.dv * 4 + BH * w.m * 4
    if with_S0:
        b += BH * w.m * w.dv * 4
    return b


def algorithmic_bytes_bwd(w):
    """Bytes one backward call must move at the least: q, k, v, dO read, beta,
    lambda read; dq, dk, dv written, dbeta, dlambda written, dS0 and dx_prev
    written (fresh sequences, zero end cotangents)."""
    es = torch.finfo(w.dtype).bits // 8
    BH = w.B * w.H
    b = BH * w.T * (2 * w.m + 2 * w.dv) * es + BH * w.T * 8          # q, k, v, dO; beta, lambda
    b += BH * w.T * (2 * w.m + w.dv) * es + BH * w.T * 8             # dq, dk, dv; dbeta, dlambda
    b += BH * w.m * w.dv * 4 + BH * w.m * 4                          # dS0, dx_prev
    return b


def algorithmic_flops(w):
    """Triangle-aware flops of the chunk form per call (Falcon-1), per chunk
    and head: C(C-1)m (X X^T) + C(C+1)m (Q X^T) + C^3/3 (solve) + C^2 (m+dv)
    (T X, T V) + 6 C m dv (state products) + C(C+1) dv (P U)."""
    C, m, dv = w.chunk, w.m, w.dv
    per = C * (C - 1) * m + C * (C + 1) * m + C ** 3 / 3 + C * C * (m + dv) + 6 * C * m * dv \
        + C * (C + 1) * dv
    if w.rule == "falcon1a":
        per = C * (C + 1) * (m + dv) + 4 * C * m * dv
    return per * w.B * w.H * ((w.T + C - 1) // C)


class ClockSampler:
    """nvidia-smi clock/throttle samples during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.proc = None

    def __enter__(self):
        self.edge = [self.query_once()]  # right before the timed region
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()
        self.edge.append(self.query_once())  # right after it
        return False

    def query_once(self):
        """One nvidia-smi sample now (a CSV line, or "" if it cannot be taken)."""
        try:
            out = subprocess.run(["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.Q}",
                                  "--format=csv,noheader,nounits"], capture_output=True,
                                 text=True, timeout=10).stdout
            return out.strip().splitlines()[0] if out.strip() else ""
        except (OSError, IndexError, subprocess.TimeoutExpired):
            return ""

    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def parse(self, lines):
        sm, mx, reasons = [], [], set()
        for line in lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, val in zip(self.NAMES, f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(n)
        return sm, mx, reasons

    def summary(self):
        """Median SM clock and the throttle reasons seen in the samples taken
        during the timed region; with fewer than three of those (a region
        shorter than the sampling period) the samples taken right before and
        right after it are included, and the note says so."""
        sm, mx, reasons = self.parse((self.out or "").strip().splitlines())
        self.in_region = len(sm)
        out = {}
        if len(sm) < 3:
            e_sm, e_mx, e_r = self.parse(self.edge)
            sm, mx, reasons = sm + e_sm, mx + e_mx, reasons | e_r
            out["note"] = ("timed region shorter than the 200 ms sampling period: samples "
                           "right before and right after it are included")
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no_samples"]}
        out.update({"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                    "reasons": sorted(reasons), "samples": len(sm),
                    "samples_in_region": self.in_region})
        return out


def barrier(ws):
    if ws > 1:
        torch.distributed.barrier()


def max_over_ranks(x, ws):
    """The slowest rank's time (NCCL on the GPU machine, gloo on a CPU host)."""
    if ws > 1:
        dev = "cuda" if torch.distributed.get_backend() == "nccl" else "cpu"
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        return float(t.item())
    return x


def input_sets(w, n_sets, device):
    """n_sets independent copies of the workload (different seeds) so that
    consecutive timed steps never find their inputs in L2."""
    sets = []
    for s in range(n_sets):
        sets.append(workloads.generate(dataclasses.replace(w, seed=w.seed + 1000 * s),
                                       device=device))
    return sets


def time_device(fn, sets, steps, warmup, ws):
    """Run fn(set) for warmup + steps steps; time exactly `steps` on the
    device with events on the current stream, barrier + sync both sides."""
    for i in range(warmup):
        fn(sets[i % len(sets)])
    torch.cuda.synchronize()
    barrier(ws)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record()
    for i in range(steps):
        fn(sets[i % len(sets)])
    ev1.record()
    torch.cuda.synchronize()
    barrier(ws)
    torch.cuda.synchronize()
    return ev0.elapsed_time(ev1) / 1e3


def time_e2e(falcon, w, inputs, workspace, steps, warmup, ws, dev):
    """End-to-end steps through falcon1_fwd_chunked with pinned host buffers.
    Streams: h2d copies, compute, d2h copies; two buffer sets alternate.
    Returns (seconds for `steps` steps, h2d bytes per step, d2h bytes per step)."""
    host_in = [{n: t.cpu().pin_memory() for n, t in inputs.items()} for _ in range(2)]
    host_o = [torch.empty((w.B, w.H, w.T, w.dv), dtype=w.dtype).pin_memory() for _ in range(2)]
    host_S = [torch.empty((w.B, w.H, w.m, w.dv), dtype=torch.float32).pin_memory()
              for _ in range(2)]
    dev_in = [{n: torch.empty_like(t, device=dev) for n, t in inputs.items()} for _ in range(2)]
    dev_o = [torch.empty((w.B, w.H, w.T, w.dv), dtype=w.dtype, device=dev) for _ in range(2)]
    dev_S = [torch.empty((w.B, w.H, w.m, w.dv), dtype=torch.float32, device=dev)
             for _ in range(2)]
    s_h2d, s_cmp, s_d2h = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    in_ready = [torch.cuda.Event() for _ in range(2)]
    cmp_done = [torch.cuda.Event() for _ in range(2)]
    out_free = [torch.cuda.Event() for _ in range(2)]

    def run(n, first):
        for i in range(first, first + n):
            b = i & 1
            with torch.cuda.stream(s_h2d):
                if i >= 2:
                    s_h2d.wait_event(cmp_done[b])  # compute(i-2) is done with dev_in[b]
                for name, t in dev_in[b].items():
                    t.copy_(host_in[b][name], non_blocking=True)
                in_ready[b].record(s_h2d)
            with torch.cuda.stream(s_cmp):
                s_cmp.wait_event(in_ready[b])
                if i >= 2:
                    s_cmp.wait_event(out_free[b])  # d2h(i-2) is done with dev_o[b]
                x = dev_in[b]
                falcon.falcon1_fwd_chunked(x["q"], x["k"], x["v"], x["beta"], x["lambda"],
                                           chunk=w.chunk, phi=w.phi, eps=w.eps,
                                           eps_gamma=w.eps_gamma, o=dev_o[b], S_out=dev_S[b],
                                           workspace=workspace, stream=s_cmp,
                                           want_x_last=False)
                cmp_done[b].record(s_cmp)
            with torch.cuda.stream(s_d2h):
                s_d2h.wait_event(cmp_done[b])
                host_o[b].copy_(dev_o[b], non_blocking=True)
                host_S[b].copy_(dev_S[b], non_blocking=True)
                out_free[b].record(s_d2h)

    run(warmup, 0)
    torch.cuda.synchronize()
    barrier(ws)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(s_h2d)
    s_cmp.wait_stream(s_h2d)
    s_d2h.wait_stream(s_h2d)
    run(steps, 0)
    s_h2d.wait_stream(s_d2h)
    ev1.record(s_h2d)
    torch.cuda.synchronize()
    barrier(ws)
    torch.cuda.synchronize()
    h2d = sum(t.numel() * t.element_size() for t in host_in[0].values())
    d2h = host_o[0].numel() * host_o[0].element_size() + host_S[0].numel() * 4
    return ev0.elapsed_time(ev1) / 1e3, h2d, d2h


def workload_config(w, ws):
    """The config object of the bench line (the same for both arms)."""
    return {"workload": w.name, "rule": w.rule, "B": w.B, "H": w.H, "T": w.T, "m": w.m,
            "dv": w.dv, "chunk": w.chunk, "phi": w.phi, "tokens_per_step": w.tokens,
            "parallelism": f"replica x{ws} (independent batches, no collective)"}


def run_ours(args):
    import delta_rule_attention_gb300 as falcon
    import numpy as np

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if ws > 1:
        torch.distributed.init_process_group("nccl", device_id=dev)
    w = workloads.LM
    per_set = algorithmic_bytes(w)
    n_sets = max(2, -(-2 * L2_BYTES // per_set) + 1)
    sets = input_sets(w, n_sets, dev)
    outs = [(torch.empty((w.B, w.H, w.T, w.dv), dtype=w.dtype, device=dev),
             torch.empty((w.B, w.H, w.m, w.dv), dtype=torch.float32, device=dev),
             torch.empty((w.B, w.H, w.m), dtype=torch.float32, device=dev))
            for _ in range(n_sets)]
    shape = falcon.make_shape(w.B, w.H, w.T, w.m, w.dv, w.chunk, w.dtype, w.phi, w.eps,
                              w.eps_gamma)
    ws_bytes = falcon.falcon_workspace_bytes(shape)
    workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    launches_per_step = 2
    counter = {"i": 0}

    def step(x):
        i = counter["i"] % n_sets
        counter["i"] += 1
        o, S, xl = outs[i]
        falcon.falcon1_fwd_chunked(x["q"], x["k"], x["v"], x["beta"], x["lambda"],
                                   chunk=w.chunk, phi=w.phi, eps=w.eps, eps_gamma=w.eps_gamma,
                                   o=o, S_out=S, x_last=xl, workspace=workspace)

    # Calibrate the step count so the timed region lasts ~3 s unless given.
    for i in range(3):
        step(sets[i % n_sets])
    torch.cuda.synchronize()
    steps = args.steps
    if steps is None:
        t = time_device(step, sets, 20, 0, 1)
        steps = int(min(200000, max(100, 3.0 / max(t / 20, 1e-7))))
    with ClockSampler(local) as clk:
        secs = time_device(step, sets, steps, args.warmup, ws)
    secs = max_over_ranks(secs, ws)
    assert falcon.falcon_sync_check() == 0
    clocks = clk.summary()
    if clocks.get("samples_in_region", 0) < 3:
        # A short timed region: the clocks under the same load are sampled for
        # about a second right after it (untimed steps of the same call).
        with ClockSampler(local) as clk2:
            t_end = time.perf_counter() + 1.0
            while time.perf_counter() < t_end:
                for i in range(64):
                    step(sets[i % n_sets])
                torch.cuda.synchronize()
        clocks["under_same_load"] = clk2.summary()
    ms = secs * 1e3 / steps
    value = w.tokens * ws * steps / secs

    # e2e: the public API fed from pinned host buffers.  Every step copies its
    # inputs host->device and its outputs (o, S_T) device->host inside the timed
    # region; copies run on their own streams, double-buffered, so step i's
    # copies overlap the compute of its neighbours.
    e2e_steps = max(10, min(steps, 200))
    e2e_secs, h2d, d2h = time_e2e(falcon, w, sets[0], workspace, e2e_steps, 3, ws, dev)
    e2e_secs = max_over_ranks(e2e_secs, ws)

    pk = peaks()
    achieved = per_set / (secs / steps) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1) q,k,v; "
        "beta=2*sigmoid(n), lambda=softplus(n-3))",
        "config": dict(workload_config(w, ws),
                       l2=f"{n_sets} rotating input sets of {per_set / 1e6:.1f} MB (> L2)"),
        "clocks": clocks,
        "e2e": {"value": w.tokens * ws * e2e_steps / e2e_secs, "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": launches_per_step * (steps + 0),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"],
                     "unit": "GB/s", "frac": achieved / pk["hbm_gbs"],
                     "traffic": profiled_traffic(),
                     "peak_source": pk["source"],
                     "kernel": "falcon1_fwd_chunked = tc_chunk_map_kernel + tc_chunk_scan_kernel "
                               "(2 launches per call, timed together)",
                     "bytes_per_launch": per_set,
                     # the same call against the bf16 tensor-core peak: the path is
                     # HBM-bound (88 flop/B, below the ~286 flop/B ridge), so this
                     # fraction is at most ~0.3 even at the HBM bound
                     "tensor": {"achieved": algorithmic_flops(w) / (secs / steps) / 1e12,
                                "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                                "frac": algorithmic_flops(w) / (secs / steps) / 1e12
                                / pk["bf16_tflops"],
                                "frac_at_hbm_bound": algorithmic_flops(w) * pk["hbm_gbs"] * 1e9
                                / per_set / 1e12 / pk["bf16_tflops"]}},
        "flops_per_step": algorithmic_flops(w),
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, budget_s=args.cpu_budget)
    if rank == 0 and not args.no_extra:
        line["also"] = extra_workloads(falcon, dev)
    if ws > 1:
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(line))


def extra_workloads(falcon, dev):
    """The other workloads, timed the same way (device-resident inputs)."""
    out = []
    pk = peaks()
    for w, steps in ((workloads.LM_1A, 200), (workloads.LONG, 5), (workloads.LM_2, 20),
                     (workloads.LM_2A, 20), (workloads.LM_3A, 20)):
        sets = input_sets(w, 1 if w is workloads.LONG else 2, dev)
        o = torch.empty((w.B, w.H, w.T, w.dv), dtype=w.dtype, device=dev)
        S = torch.empty((w.B, w.H, w.m, w.dv), dtype=torch.float32, device=dev)
        if w.rule == "falcon3a":
            shape = falcon.make_shape(w.B, w.H, w.T, w.m, w.dv, w.chunk, w.dtype, w.phi)
            wsb = torch.empty(max(falcon.falcon_workspace_bytes(shape), 1), dtype=torch.uint8,
                              device=dev)

            def step(x):
                falcon.falcon3a_fwd_chunked(x["q"], x["k"], x["v"], x["beta"], x["lambda"],
                                            workloads.LM_3A_WINDOW, phi=w.phi, o=o, S_out=S,
                                            workspace=wsb, want_x_last=False)
        elif w.per_column:
            shape = falcon.make_shape(w.B, w.H, w.T, w.m, w.dv, w.chunk, w.dtype, w.phi)
            wsb = torch.empty(max(falcon.falcon_workspace_bytes(shape), 1), dtype=torch.uint8,
                              device=dev)
            if w.rule == "falcon2a":
                def step(x):
                    falcon.falcon2a_fwd_chunked(x["q"], x["k"], x["v"], x["beta"], x["lambda"],
                                                phi=w.phi, o=o, S_out=S, workspace=wsb,
                                                want_x_last=False)
            else:
                def step(x):
                    falcon.falcon2_fwd_chunked(x["q"], x["k"], x["v"], x["beta"], x["lambda"],
                                               phi=w.phi, o=o, S_out=S, want_x_last=False)
        else:
            fn = falcon.falcon1_fwd_chunked if w.rule == "falcon1" else falcon.falcon1a_fwd_chunked
            shape = falcon.make_shape(w.B, w.H, w.T, w.m, w.dv, w.chunk, w.dtype, w.phi)
            wsb = torch.empty(max(falcon.falcon_workspace_bytes(shape), 1), dtype=torch.uint8,
                              device=dev)

            def step(x):
                fn(x["q"], x["k"], x["v"], x["beta"], x["lambda"], chunk=w.chunk, phi=w.phi,
                   o=o, S_out=S, workspace=wsb, want_x_last=False)
        secs = time_device(step, sets, steps, 2, 1)
        b = algorithmic_bytes(w)
        out.append({"workload": w.name, "tokens_per_s": w.tokens * steps / secs,
                    "ms_per_call": secs * 1e3 / steps,
                    "hbm_frac": b / (secs / steps) / 1e9 / pk["hbm_gbs"]})
        del sets
    # Falcon-1A with the normalised read (z) on the lm-1A shape, positive q, k
    # (the setting in which the normaliser is attention-like); its bytes add
    # z_T to the forward's
    w = workloads.LM_1A
    sets = input_sets(w, 2, dev)
    for x in sets:
        x["q"] = x["q"].abs() + 0.05
        x["k"] = x["k"].abs() + 0.05
    o = torch.empty((w.B, w.H, w.T, w.dv), dtype=w.dtype, device=dev)
    S = torch.empty((w.B, w.H, w.m, w.dv), dtype=torch.float32, device=dev)
    z = torch.empty((w.B, w.H, w.m), dtype=torch.float32, device=dev)
    xl = torch.empty((w.B, w.H, w.m), dtype=torch.float32, device=dev)
    shape = falcon.make_shape(w.B, w.H, w.T, w.m, w.dv, w.chunk, w.dtype, w.phi)
    wsb = torch.empty(max(falcon.falcon_normalized_workspace_bytes(shape), 1), dtype=torch.uint8,
                      device=dev)

    def nstep(x):
        falcon.falcon1a_fwd_chunked_normalized(x["q"], x["k"], x["v"], x["beta"], x["lambda"],
                                               chunk=w.chunk, phi=w.phi, o=o, S_out=S, z_out=z,
                                               x_last=xl, workspace=wsb)
    steps = 200
    secs = time_device(nstep, sets, steps, 3, 1)
    b = algorithmic_bytes(w) + w.B * w.H * w.m * 4
    out.append({"workload": w.name.replace("falcon1a_", "falcon1a_normalized_"),
                "tokens_per_s": w.tokens * steps / secs, "ms_per_call": secs * 1e3 / steps,
                "hbm_frac": b / (secs / steps) / 1e9 / pk["hbm_gbs"]})
    del sets, wsb
    # backward of the chunked forward (lm shapes): gradients for q, k, v, beta,
    # lambda, S0 and x_prev from a seeded dO
    for w in (workloads.LM, workloads.LM_1A):
        sets = input_sets(w, 2, dev)
        for k, x in enumerate(sets):
            x.update(workloads.cotangents(w.B, w.H, w.T, w.m, w.dv, w.dtype, seed=w.seed + 7 * k,
                                          device=dev))
        fnb = falcon.falcon1_bwd_chunked if w.rule == "falcon1" else falcon.falcon1a_bwd_chunked
        shape = falcon.make_shape(w.B, w.H, w.T, w.m, w.dv, w.chunk, w.dtype, w.phi)
        wsb = torch.empty(max(falcon.falcon_bwd_workspace_bytes(shape), 1), dtype=torch.uint8,
                          device=dev)
        grads = {}

        def bstep(x):
            fnb(x["q"], x["k"], x["v"], x["beta"], x["lambda"], x["dO"], chunk=w.chunk,
                phi=w.phi, workspace=wsb, grads=grads)
        steps = 50
        secs = time_device(bstep, sets, steps, 3, 1)
        b = algorithmic_bytes_bwd(w)
        out.append({"workload": w.name.replace("_lm_", "_lm_bwd_"),
                    "tokens_per_s": w.tokens * steps / secs, "ms_per_call": secs * 1e3 / steps,
                    "hbm_frac": b / (secs / steps) / 1e9 / pk["hbm_gbs"]})
        del sets, wsb, grads
    # decode: rotating per-step inputs, state resident
    d = workloads.DECODE
    stream = workloads.DecodeStream(d, device=dev)
    S = stream.initial_state()
    xp = torch.zeros((d.N, d.m), device=dev)
    steps_in = [stream.step() for _ in range(8)]
    o = torch.empty((d.N, d.dv), dtype=d.dtype, device=dev)

    def dstep(x):
        falcon.falcon1_decode_step(x["q"], x["k"], x["v"], x["beta"], x["lambda"], S, xp,
                                   phi=d.phi, o=o)
    n = 512
    secs = time_device(dstep, steps_in, n, 4, 1)
    state_bytes = 2 * d.N * d.m * d.dv * 4
    step_bytes = state_bytes + d.N * ((2 * d.m + 2 * d.dv) * 2 + 8 + 2 * d.m * 4)
    out.append({"workload": d.name, "tokens_per_s": d.N * n / secs,
                "us_per_step": secs * 1e6 / n,
                "hbm_frac": step_bytes / (secs / n) / 1e9 / pk["hbm_gbs"]})
    return out


def host_cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else platform)."""
    import platform
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.TimeoutExpired):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu model")):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.processor() or platform.machine()


def cpu_baseline(w, budget_s=12.0, reps_max=20):
    """The fp64 oracle on this host's cores: whole LM workload per rep (all
    heads), repeated until ~budget_s of CPU time; plus one thread on two heads
    (the single-thread rate)."""
    import oracle
    x = workloads.generate(w, device="cpu")
    cores = os.cpu_count() or 1
    t0 = time.perf_counter()
    reps = 0
    while True:
        oracle.forward(w.rule, x["q"], x["k"], x["v"], x["beta"], x["lambda"], phi=w.phi,
                       eps=w.eps, eps_gamma=w.eps_gamma, threads=cores)
        reps += 1
        el = time.perf_counter() - t0
        if el > budget_s or reps >= reps_max:
            break
    one = {n: t[:1, :2].contiguous() for n, t in x.items()}
    t1 = time.perf_counter()
    oracle.forward(w.rule, one["q"], one["k"], one["v"], one["beta"], one["lambda"], phi=w.phi,
                   eps=w.eps, eps_gamma=w.eps_gamma, threads=1)
    el1 = time.perf_counter() - t1
    return {"value": w.tokens * reps / el, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "cpu_model": host_cpu_model(),
            "sample": f"{reps} x full {w.name} (all {w.B * w.H} heads, fp64, {cores} threads)",
            "single_thread": {"value": 2 * w.T / el1 / w.H, "unit": "tokens/s",
                              "sample": f"2 heads of {w.name} on 1 thread, as B*T tokens/s of "
                                        f"the {w.H}-head workload"}}


def run_reference(args):
    """The fp64 oracle timed on the host cores, rank 0 only: one step is the
    whole workload (all B*H heads, T tokens each), the same config as ours."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    w = workloads.LM
    x = workloads.generate(w, device="cpu")
    cores = os.cpu_count() or 1
    steps = args.steps if args.steps is not None else 5

    def one():
        oracle.forward(w.rule, x["q"], x["k"], x["v"], x["beta"], x["lambda"],
                       phi=w.phi, eps=w.eps, eps_gamma=w.eps_gamma, threads=cores)
    for _ in range(args.warmup):
        one()
    t0 = time.perf_counter()
    for _ in range(steps):
        one()
    secs = time.perf_counter() - t0
    value = w.tokens * steps / secs
    sample = (f"the whole {w.name} workload per step ({w.B * w.H} heads x {w.T} tokens), fp64, "
              f"{cores} threads")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": ws, "steps": steps, "warmup": args.warmup,
            "ms_per_step": secs * 1e3 / steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(w, ws),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores,
                             "kind": "oracle", "sample": sample,
                             "cpu_model": host_cpu_model()},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line))


def run_profile(args):
    """Profiler target: one workload's library calls only (no timing line), so
    that ncu captures run committed code on a chosen, possibly reduced, size."""
    import delta_rule_attention_gb300 as falcon
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    calls = args.steps or 3
    if args.profile == "decode":
        d = workloads.DECODE
        if args.profile_size:
            d = dataclasses.replace(d, n_seq=max(1, args.profile_size // d.H))
        stream = workloads.DecodeStream(d, device=dev)
        S = stream.initial_state()
        xp = torch.zeros((d.N, d.m), device=dev)
        o = torch.empty((d.N, d.dv), dtype=d.dtype, device=dev)
        for _ in range(calls):
            x = stream.step()
            falcon.falcon1_decode_step(x["q"], x["k"], x["v"], x["beta"], x["lambda"], S, xp,
                                       phi=d.phi, o=o)
        name, size = d.name, d.N
    else:
        bwd = args.profile.endswith("bwd")
        norm = args.profile == "lm1anorm"
        w = {"lm": workloads.LM, "lm1a": workloads.LM_1A, "long": workloads.LONG,
             "lm2": workloads.LM_2, "lm2a": workloads.LM_2A, "lm3a": workloads.LM_3A,
             "lmbwd": workloads.LM, "lm1abwd": workloads.LM_1A,
             "lm1anorm": workloads.LM_1A}[args.profile]
        if args.profile_size:
            w = dataclasses.replace(w, T=args.profile_size)
        x = workloads.generate(w, device=dev)
        if bwd:
            x.update(workloads.cotangents(w.B, w.H, w.T, w.m, w.dv, w.dtype, seed=w.seed,
                                          device=dev))
        for _ in range(calls):
            if norm:
                falcon.falcon1a_fwd_chunked_normalized(x["q"], x["k"], x["v"], x["beta"],
                                                       x["lambda"], chunk=w.chunk, phi=w.phi)
            elif bwd:
                fnb = (falcon.falcon1_bwd_chunked if w.rule == "falcon1"
                       else falcon.falcon1a_bwd_chunked)
                fnb(x["q"], x["k"], x["v"], x["beta"], x["lambda"], x["dO"], chunk=w.chunk,
                    phi=w.phi)
            elif w.rule == "falcon3a":
                falcon.falcon3a_fwd_chunked(x["q"], x["k"], x["v"], x["beta"], x["lambda"],
                                            workloads.LM_3A_WINDOW, phi=w.phi)
            elif w.per_column:
                fn2 = (falcon.falcon2_fwd_chunked if w.rule == "falcon2"
                       else falcon.falcon2a_fwd_chunked)
                fn2(x["q"], x["k"], x["v"], x["beta"], x["lambda"], phi=w.phi)
            else:
                fn = (falcon.falcon1_fwd_chunked if w.rule == "falcon1"
                      else falcon.falcon1a_fwd_chunked)
                fn(x["q"], x["k"], x["v"], x["beta"], x["lambda"], chunk=w.chunk, phi=w.phi)
        name, size = w.name, w.T
    torch.cuda.synchronize()
    assert falcon.falcon_sync_check() == 0
    print(json.dumps({"profile": name, "size": size, "calls": calls, "ok": True}))


def host_link(args):
    """Pinned host <-> device copy bandwidth at the e2e step's sizes (the lm
    workload's inputs host->device, o and S_T device->host): each direction
    alone, then both at once on two streams.  Prints one JSON line."""
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    w = workloads.LM
    x = workloads.generate(w, device="cpu")
    h_in = [t.pin_memory() for t in x.values()]
    d_in = [torch.empty_like(t, device=dev) for t in h_in]
    d_out = [torch.empty((w.B, w.H, w.T, w.dv), dtype=w.dtype, device=dev),
             torch.empty((w.B, w.H, w.m, w.dv), dtype=torch.float32, device=dev)]
    h_out = [torch.empty_like(t, device="cpu").pin_memory() for t in d_out]
    b_in = sum(t.numel() * t.element_size() for t in h_in)
    b_out = sum(t.numel() * t.element_size() for t in h_out)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    reps = args.steps or 50

    def h2d():
        with torch.cuda.stream(s1):
            for d, h in zip(d_in, h_in):
                d.copy_(h, non_blocking=True)

    def d2h():
        with torch.cuda.stream(s2):
            for h, d in zip(h_out, d_out):
                h.copy_(d, non_blocking=True)

    def timed(fns):
        for _ in range(3):
            for f in fns:
                f()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(reps):
            for f in fns:
                f()
        torch.cuda.synchronize()
        return (time.perf_counter() - t0) / reps

    t_in, t_out, t_both = timed([h2d]), timed([d2h]), timed([h2d, d2h])
    print(json.dumps({
        "host_link": True, "reps": reps, "h2d_bytes": b_in, "d2h_bytes": b_out,
        "h2d_gbs": b_in / t_in / 1e9, "d2h_gbs": b_out / t_out / 1e9,
        "h2d_us": t_in * 1e6, "d2h_us": t_out * 1e6, "both_us": t_both * 1e6,
        "both_gbs": (b_in + b_out) / t_both / 1e9,
        "gpu": torch.cuda.get_device_name(dev), "cpu_model": host_cpu_model()}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-extra", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--profile",
                    choices=["lm", "lm1a", "long", "decode", "lm2", "lm2a", "lm3a", "lmbwd",
                             "lm1abwd", "lm1anorm"], default=None,
                    help="profiler target: run --steps calls of one workload, print no timing")
    ap.add_argument("--host-link", action="store_true",
                    help="measure pinned host<->device copy bandwidth at the e2e sizes")
    ap.add_argument("--profile-size", type=int, default=None,
                    help="with --profile: tokens per head (chunked) or states (decode)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.host_link:
        host_link(args)
    elif args.profile:
        run_profile(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
