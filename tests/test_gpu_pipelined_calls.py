"""Back-to-back calls on one stream, sharing one workspace, with no
synchronisation between them, give exactly the outputs of the same calls run
one at a time.

The chunked forwards launch their map kernel as a programmatic dependent
launch behind whatever kernel precedes it on the stream, and their scans let
the next launch start early, so a call's map CTAs can be resident while the
previous call's scan is still reading the workspace they will overwrite.  The
map kernel waits for the preceding grid before it reads or writes anything;
this test holds it to that.  The forwards are deterministic (no atomics), so
the comparison is bit for bit.
"""
import pytest
import torch

from delta_rule_attention_gb300 import workloads

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

CALLS = 3


@pytest.fixture(scope="module")
def falcon():
    import delta_rule_attention_gb300 as f
    f.load_library()
    return f


def _inputs(B, H, T, m, dv, seed, per_column=False):
    return workloads.random_case(B, H, T, m, dv, dtype=torch.bfloat16, seed=seed,
                                 lam_shift=-3.0, device="cuda", per_column=per_column)


def _call(falcon, rule, x, outs, workspace):
    o, S, xl = outs
    args = (x["q"], x["k"], x["v"], x["beta"], x["lambda"])
    if rule == "falcon1":
        falcon.falcon1_fwd_chunked(*args, chunk=64, phi="l2", o=o, S_out=S, x_last=xl,
                                   workspace=workspace)
    elif rule == "falcon1a":
        falcon.falcon1a_fwd_chunked(*args, chunk=64, phi="l2", o=o, S_out=S, x_last=xl,
                                    workspace=workspace)
    elif rule == "falcon2a":
        falcon.falcon2a_fwd_chunked(*args, phi="l2", o=o, S_out=S, x_last=xl,
                                    workspace=workspace)
    else:
        falcon.falcon3a_fwd_chunked(*args, 4, phi="l2", o=o, S_out=S, x_last=xl,
                                    workspace=workspace)


# rule, B, H, T, m (= dv); the long-sequence case runs as chunk-range pieces
# (few heads, many chunks) with its scans on a second stream.
CASES = [
    ("falcon1", 2, 12, 1024 + 37, 64),
    ("falcon1a", 2, 12, 1024, 64),
    ("falcon1", 1, 4, 8192, 128),
    ("falcon2a", 2, 8, 1024, 64),
    ("falcon3a", 2, 8, 1024 + 5, 64),
]


@pytest.mark.parametrize("rule,B,H,T,m", CASES)
def test_back_to_back_calls_match_isolated_calls(falcon, rule, B, H, T, m):
    xs = [_inputs(B, H, T, m, m, seed=100 + i, per_column=rule == "falcon2a")
          for i in range(CALLS)]

    def outs():
        return (torch.empty((B, H, T, m), dtype=torch.bfloat16, device="cuda"),
                torch.empty((B, H, m, m), dtype=torch.float32, device="cuda"),
                torch.empty((B, H, m), dtype=torch.float32, device="cuda"))

    shape = falcon.make_shape(B, H, T, m, m, 64, torch.bfloat16, "l2")
    ws_bytes = falcon.falcon_workspace_bytes(shape)

    # One call at a time, each with its own workspace, synchronised.
    ref = []
    for x in xs:
        o = outs()
        ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device="cuda")
        _call(falcon, rule, x, o, ws)
        torch.cuda.synchronize()
        assert falcon.falcon_sync_check() == 0
        ref.append(o)

    # The same calls back to back on one stream, sharing one workspace that
    # still holds the previous call's data, synchronised only at the end.
    shared = torch.full((max(ws_bytes, 1),), 0x7F, dtype=torch.uint8, device="cuda")
    got = [outs() for _ in xs]
    torch.cuda.synchronize()
    for x, o in zip(xs, got):
        _call(falcon, rule, x, o, shared)
    torch.cuda.synchronize()
    assert falcon.falcon_sync_check() == 0

    for i, (r, g) in enumerate(zip(ref, got)):
        for name, a, b in zip(("o", "S_T", "x_last"), r, g):
            assert torch.equal(a, b), f"call {i}: {name} differs from the isolated call"
