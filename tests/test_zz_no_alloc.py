"""The fixed-scratch Falcon-1 forward (falcon1_fwd_chunked_fixed_scratch).

Some callers cannot allocate device memory at the call site: a C host
program or plugin that only receives input and output buffers, a framework
whose allocator is out of reach, a serving loop that forbids allocation after
start-up.  For them the library offers this entry point, which takes no
workspace and uses a fixed scratch array built into the library instead.

The GPU test calls it twice in a row through the C ABI (the second call sees
the first call's leftovers in the shared array) and compares each result with
the regular workspace entry point, within the parity tolerances used
everywhere else (1e-4 for fp32 inputs, 2e-2 for bf16).  This file is named so
that pytest collects it last.
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
