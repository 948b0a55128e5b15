"""Failure detection without a GPU fault.

Every device-side wait of the library is bounded in time; when one runs out,
the kernel records the expiry in the library's device error word and returns
(no trap, no hang), and falcon_sync_check reports FALCON_ERR_TIMEOUT.  The GPU
test makes a wait run out on purpose (a barrier that nothing completes, with a
20 ms limit) and checks the status, that the word is cleared by the read, and
that the context still runs a forward call correctly afterwards.
"""
import ctypes

import numpy as np
import pytest
import torch

FALCON_ERR_TIMEOUT = -7


def test_selftest_rejects_bad_limits_without_a_device():
    import shutil
    if shutil.which("nvcc") is None:
        pytest.skip("needs nvcc to build the library")
    from delta_rule_attention_gb300 import _build
    _build.build()
    import delta_rule_attention_gb300 as falcon
    lib = falcon.load_library()
    assert lib.falcon_selftest_wait_timeout(0, None) == -8
    assert lib.falcon_selftest_wait_timeout(10_000_001, None) == -8


@pytest.mark.gpu
@pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")
def test_lost_wait_reports_timeout_and_context_survives():
    import oracle
    import delta_rule_attention_gb300 as falcon
    from delta_rule_attention_gb300 import workloads
    assert falcon.falcon_sync_check() == 0
    falcon.falcon_selftest_wait_timeout(20000)
    assert falcon.falcon_sync_check() == FALCON_ERR_TIMEOUT
    assert falcon.falcon_sync_check() == 0  # the read cleared the word
    x = workloads.random_case(1, 2, 130, 64, 64, torch.bfloat16, seed=3, device="cuda")
    o, S, _ = falcon.falcon1_fwd_chunked(x["q"], x["k"], x["v"], x["beta"], x["lambda"], chunk=64)
    assert falcon.falcon_sync_check() == 0
    ref = oracle.forward("falcon1", x["q"], x["k"], x["v"], x["beta"], x["lambda"])
    err = np.linalg.norm(o.float().cpu().numpy() - ref["o"]) / np.linalg.norm(ref["o"])
    assert err < 2e-2
