"""A bounded device wait that runs out, on the GPU, without faulting it.

The tensor-core prefill kernels hand chunks between their warp roles through
mbarrier waits bounded in wall time.  gla_set_wait_limit_ns shortens that bound
for the hand-off waits only (not the teardown drain), so a normal call hits it:
some role gives up, flags the abort, every role stops at its next wait, the
producer waits for its own tile copies and the MMA issuers for their own
matrix products, tensor memory is released and the kernel returns.  The call
must then report GLA_ERR_TIMEOUT through status_sync, and the next call, with
the default limit back, must be correct.  Nothing here waits on a flag that
nothing sets: every wait ends, by its limit or by the abort flag.  (The abort
protocol itself is modelled on the CPU in test_prefill_protocol.py.)
"""
import pytest
import torch

import gla_inputs
from parity import cuda, rel_max, to_np, out_tol, TOL_STATE
import oracle

pytestmark = pytest.mark.gpu

GLA_ERR_TIMEOUT = 5


def _gla():
    import gated_linear_attention_gla_gb300 as gla
    return gla


ATTEMPTS = 20


@pytest.mark.parametrize("workload", ["prefill", "vector"])
def test_wait_that_runs_out_reports_timeout_then_next_call_is_correct(cuda_ok, workload):
    """With a 1 ns limit, a hand-off wait that is still open once its first
    barrier test returns runs out.  A barrier test may hold a warp until the
    hand-off completes (up to a hardware-defined time), so a call can also
    finish normally; the call is repeated until one reports the timeout (each
    attempt either times out or is a normal call)."""
    gla = _gla()
    x = gla_inputs.prefill_inputs(gla_inputs.WORKLOADS[workload], seed=5, B=2, T=4000, H=8)
    args = (cuda(x["q"]), cuda(x["k"]), cuda(x["v"]), cuda(x["g"]))
    kw = dict(scale=x["scale"], init_state=cuda(x["init_state"]), chunk=128,
              output_final_state=True, out_dtype=torch.float32)
    flags = gla.GLA_FLAG_VECTOR_GATE if workload == "vector" else 0
    assert gla.lib().gla_chunk_fwd_kernel(128, 128, 128, flags) == b"tensor_core"
    gla.status_sync()
    prev = gla.set_wait_limit_ns(1)
    timed_out = 0
    try:
        for attempt in range(ATTEMPTS):
            gla.chunk_fwd(*args, **kw)
            try:
                gla.status_sync()
            except gla.GlaError as e:
                assert e.status == GLA_ERR_TIMEOUT
                timed_out = attempt + 1
                break
    finally:
        gla.set_wait_limit_ns(prev)
    print(f"timed out on attempt {timed_out}")
    assert timed_out, f"no wait ran out in {ATTEMPTS} calls"
    assert gla.status_sync() == 0  # reported once, then cleared
    out, fin = gla.chunk_fwd(*args, **kw)
    assert gla.status_sync() == 0
    o_ref, s_ref = oracle.recurrent(x["q"], x["k"], x["v"], x["g"], x["scale"],
                                    init_state=x["init_state"])
    assert rel_max(to_np(out), o_ref) <= out_tol(torch.bfloat16)
    assert rel_max(to_np(fin), s_ref) <= TOL_STATE
