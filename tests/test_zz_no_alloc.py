"""gla_chunk_bwd_fixed_workspace: the backward for callers that cannot allocate.

Some callers cannot call cudaMalloc when they need a gradient -- code running
inside a caching allocator's callbacks, real-time threads that must not take
the driver's allocation lock, embedders whose device memory is reserved up
front.  For them the library's tensor-core backward takes its workspace from a
fixed static device buffer (384 MiB) instead of a caller-provided one.

These tests call that entry point straight through the C ABI (ctypes, device
pointers only; the outputs are allocated by the test beforehand, as such a
caller would have them) and compare it with gla_chunk_bwd given a caller
workspace, on two calls in a row with different inputs: the second call must
not see anything of the first one's contents of the shared buffer.  A call
whose workspace need exceeds the buffer must be rejected before anything is
enqueued, with the limit in gla_last_error_string().

The file is named to be collected last, so that a run that stops at the first
failure has run every other test before this one; it also builds and loads the
library itself, so it passes when run alone in a fresh process.
"""
import ctypes

import pytest
import torch

import gla_inputs

pytestmark = pytest.mark.gpu

NAMES = ("dq", "dk", "dv", "dg", "d_init")


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gated_linear_attention_gla_gb300 import build as glabuild
    glabuild.build()
    from gated_linear_attention_gla_gb300 import _binding
    return _binding.lib()


def _p(t):
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _device_inputs(seed, B=4, T=2048, H=16):
    x = gla_inputs.prefill_inputs(gla_inputs.WORKLOADS["prefill"], seed=seed, B=B, T=T, H=H)
    gr = gla_inputs.grad_inputs(x, seed=seed)
    d = {n: x[n].cuda() for n in ("q", "k", "v", "g", "init_state")}
    d["d_out"] = gr["d_out"].cuda()
    d["d_final"] = gr["d_final_state"].cuda()
    d["scale"] = x["scale"]
    d["B"], d["T"], d["H"] = B, T, H
    return d


def _outputs(d):
    dq = torch.full_like(d["q"], float("nan"))
    dk = torch.full_like(d["k"], float("nan"))
    dv = torch.full_like(d["v"], float("nan"))
    dg = torch.full_like(d["g"], float("nan"))
    d_init = torch.full_like(d["init_state"], float("nan"))
    return dq, dk, dv, dg, d_init


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _call_fixed(L, d, outs):
    dq, dk, dv, dg, d_init = outs
    return L.gla_chunk_bwd_fixed_workspace(
        _p(d["q"]), _p(d["k"]), _p(d["v"]), _p(d["g"]), ctypes.c_float(d["scale"]),
        _p(d["init_state"]), _p(d["d_out"]), _p(d["d_final"]), _p(dq), _p(dk), _p(dv),
        _p(dg), _p(d_init), _p(None), d["B"], d["H"], d["T"], 128, 128, _stream(), 0)


def _call_with_workspace(L, d, outs):
    dq, dk, dv, dg, d_init = outs
    need = L.gla_chunk_bwd_workspace_size(d["B"], d["H"], d["T"], 128, 128, 0, 0)
    assert need > 0
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    rc = L.gla_chunk_bwd(
        _p(d["q"]), _p(d["k"]), _p(d["v"]), _p(d["g"]), ctypes.c_float(d["scale"]),
        _p(d["init_state"]), _p(d["d_out"]), _p(d["d_final"]), _p(dq), _p(dk), _p(dv),
        _p(dg), _p(d_init), _p(None), d["B"], d["H"], d["T"], 128, 128, _p(ws),
        ctypes.c_size_t(need), _stream(), 0)
    torch.cuda.synchronize()
    return rc


def _status(L):
    return L.gla_status_sync(_stream())


def test_two_calls_in_a_row_match_the_caller_workspace_entry_point(L):
    """Two calls with different inputs at the prefill workload's sizes (B = 4,
    T = 2048, H = 16, d = 128: 152 MB of the 384 MiB buffer): each equals
    gla_chunk_bwd on a caller workspace -- dq, dk, dv and d_init bit for bit
    (the same kernels on the same operands), dg within the order of its fp32
    atomic additions (1e-5 of its largest magnitude)."""
    for seed in (101, 202):
        d = _device_inputs(seed)
        mine, ref = _outputs(d), _outputs(d)
        assert _call_fixed(L, d, mine) == 0
        assert _status(L) == 0
        assert _call_with_workspace(L, d, ref) == 0
        assert _status(L) == 0
        for name, a, b in zip(NAMES, mine, ref):
            assert not torch.isnan(a).any(), f"seed {seed}: {name} left unwritten"
            if name == "dg":
                torch.testing.assert_close(a, b, rtol=1e-5, atol=1e-5 * float(b.abs().max()))
            else:
                assert torch.equal(a, b), f"seed {seed}: {name} differs"


def test_a_call_beyond_the_buffer_is_rejected_before_anything_runs(L):
    """B = 16, T = 2048, H = 16 needs about 606 MB of workspace: the call
    returns GLA_ERR_UNSUPPORTED, names the need and the limit, and writes
    nothing."""
    B, T, H = 16, 2048, 16
    need = L.gla_chunk_bwd_workspace_size(B, H, T, 128, 128, 0, 0)
    assert need > 384 << 20
    w = gla_inputs.WORKLOADS["prefill"]
    z = lambda *s, dt=torch.bfloat16: torch.zeros(*s, dtype=dt, device="cuda")  # noqa: E731
    d = dict(q=z(B, T, H, 128), k=z(B, T, H, 128), v=z(B, T, H, 128),
             g=z(B, T, H, dt=torch.float32), init_state=z(B, H, 128, 128, dt=torch.float32),
             d_out=z(B, T, H, 128), d_final=z(B, H, 128, 128, dt=torch.float32),
             scale=w.dk ** -0.5, B=B, T=T, H=H)
    outs = _outputs(d)
    rc = _call_fixed(L, d, outs)
    assert rc == 2  # GLA_ERR_UNSUPPORTED
    L.gla_last_error_string.restype = ctypes.c_char_p
    msg = L.gla_last_error_string().decode()
    assert str(need) in msg and str(384 << 20) in msg, msg
    torch.cuda.synchronize()
    assert _status(L) == 0
    for name, t in zip(NAMES, outs):
        assert torch.isnan(t).all(), f"{name} was written by a rejected call"
