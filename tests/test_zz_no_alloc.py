"""The fixed-scratch Falcon-1 forward (falcon1_fwd_chunked_fixed_scratch).

Some callers cannot allocate device memory at the call site: a C host
program or plugin that only receives input and output buffers, a framework
whose allocator is out of reach, a serving loop that forbids allocation after
start-up.  For them the library offers this entry point, which takes no
workspace and uses a fixed scratch array built into the library instead.

The GPU tests call it twice in a row through the C ABI (the second call sees
the first call's leftovers in the shared array) and compare each result with
the regular workspace entry point, within the parity tolerances used
everywhere else (1e-4 for fp32 inputs, 2e-2 for bf16).  The tensor-core cases
(bf16, m = d_v = 64 or 128, chunk 64; one of them long enough for the
chunk-range pieces on the second stream) are also compared with the fp64
oracle.  This file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

from delta_rule_attention_gb300 import workloads


def _rel(a, b):
    a = a.double().cpu().numpy().reshape(-1, a.shape[-2] * a.shape[-1])
    b = b.double().cpu().numpy().reshape(a.shape)
    return float((np.linalg.norm(a - b, axis=1) / np.maximum(np.linalg.norm(b, axis=1), 1e-30))
                 .max())


def test_scratch_limit_is_rejected_on_the_host():
    """A shape whose scratch exceeds the fixed array is refused before any
    device work (no GPU needed)."""
    import shutil
    if shutil.which("nvcc") is None:
        pytest.skip("needs nvcc to build the library")
    from delta_rule_attention_gb300 import _build
    _build.build()
    import delta_rule_attention_gb300 as falcon
    lib = falcon.load_library()
    big = falcon.make_shape(8, 12, 2048, 64, 64, 64, torch.bfloat16)
    assert lib.falcon_workspace_bytes(ctypes.byref(big)) > falcon.FALCON_FIXED_SCRATCH_BYTES
    p = ctypes.c_void_p(0x10000)
    rc = lib.falcon1_fwd_chunked_fixed_scratch(ctypes.byref(big), p, p, p, p, p, None, None, p,
                                               p, None, None)
    assert rc == falcon.FALCON_ERR_SCRATCH_LIMIT
    assert b"fixed" in lib.falcon_strerror(rc)


@pytest.mark.gpu
@pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_fixed_scratch_matches_workspace_entry_point(dtype):
    import delta_rule_attention_gb300 as falcon
    tol = 1e-4 if dtype == torch.float32 else 2e-2
    # Two different problems back to back; the second is larger and carries state.
    cases = [
        workloads.random_case(1, 2, 64, 16, 16, dtype, seed=101, device="cuda"),
        workloads.random_case(2, 3, 200, 64, 32, dtype, seed=102, device="cuda",
                              with_state=True, with_x_prev=True),
    ]
    for x, C in zip(cases, (16, 64)):
        B, H, T, m = x["q"].shape
        dv = x["v"].shape[-1]
        shape = falcon.make_shape(B, H, T, m, dv, C, dtype)
        assert falcon.falcon_workspace_bytes(shape) <= falcon.FALCON_FIXED_SCRATCH_BYTES
        o = torch.empty((B, H, T, dv), dtype=dtype, device="cuda")
        S = torch.empty((B, H, m, dv), dtype=torch.float32, device="cuda")
        xl = torch.empty((B, H, m), dtype=torch.float32, device="cuda")
        falcon.falcon1_fwd_chunked_fixed_scratch(
            x["q"], x["k"], x["v"], x["beta"], x["lambda"], S0=x.get("S0"),
            x_prev=x.get("x_prev"), chunk=C, o=o, S_out=S, x_last=xl)
        assert falcon.falcon_sync_check() == 0
        o_ref, S_ref, xl_ref = falcon.falcon1_fwd_chunked(
            x["q"], x["k"], x["v"], x["beta"], x["lambda"], S0=x.get("S0"),
            x_prev=x.get("x_prev"), chunk=C)
        assert falcon.falcon_sync_check() == 0
        assert _rel(o.float(), o_ref.float()) < tol
        assert _rel(S, S_ref) < tol
        np.testing.assert_allclose(xl.cpu().numpy(), xl_ref.cpu().numpy(), rtol=1e-6, atol=1e-7)


@pytest.mark.gpu
@pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")
def test_fixed_scratch_tensor_core_path_against_oracle():
    """bf16, m = d_v = 64 and 128, chunk 64: the tensor-core kernels read and
    write their chunk maps in the fixed array.  B1 H2 T8192 at m = 64 runs as
    chunk-range pieces (maps on the caller's stream, scans on the library's
    second stream).  Three calls in a row, each against the oracle and against
    the workspace entry point."""
    import oracle
    import delta_rule_attention_gb300 as falcon
    cases = [
        (workloads.random_case(1, 2, 256, 64, 64, torch.bfloat16, seed=111, device="cuda",
                               with_state=True, with_x_prev=True), "falcon1"),
        (workloads.random_case(1, 2, 8192 + 17, 64, 64, torch.bfloat16, seed=112,
                               device="cuda", with_state=True), "falcon1"),
        (workloads.random_case(1, 2, 1000, 128, 128, torch.bfloat16, seed=113, device="cuda",
                               with_x_prev=True), "falcon1"),
    ]
    for x, rule in cases:
        B, H, T, m = x["q"].shape
        shape = falcon.make_shape(B, H, T, m, m, 64, torch.bfloat16)
        assert falcon.falcon_workspace_bytes(shape) <= falcon.FALCON_FIXED_SCRATCH_BYTES
        o = torch.empty((B, H, T, m), dtype=torch.bfloat16, device="cuda")
        S = torch.empty((B, H, m, m), dtype=torch.float32, device="cuda")
        xl = torch.empty((B, H, m), dtype=torch.float32, device="cuda")
        falcon.falcon1_fwd_chunked_fixed_scratch(
            x["q"], x["k"], x["v"], x["beta"], x["lambda"], S0=x.get("S0"),
            x_prev=x.get("x_prev"), chunk=64, o=o, S_out=S, x_last=xl)
        assert falcon.falcon_sync_check() == 0
        o_ws, S_ws, _ = falcon.falcon1_fwd_chunked(
            x["q"], x["k"], x["v"], x["beta"], x["lambda"], S0=x.get("S0"),
            x_prev=x.get("x_prev"), chunk=64)
        assert falcon.falcon_sync_check() == 0
        ref = oracle.forward(rule, x["q"], x["k"], x["v"], x["beta"], x["lambda"],
                             S0=x.get("S0"), x_prev=x.get("x_prev"), phi="l2")
        assert _rel(o.float(), o_ws.float()) < 2e-2
        assert _rel(S, S_ws) < 2e-2
        assert _rel(o.float(), torch.from_numpy(ref["o"])) < 2e-2
        assert _rel(S, torch.from_numpy(ref["S"])) < 2e-2
        np.testing.assert_allclose(xl.cpu().numpy(), ref["x_last"], rtol=1e-6, atol=1e-6)
