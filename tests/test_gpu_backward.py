"""GPU chunked backward (gla_chunk_bwd) against the fp64 oracle's gradient.

Both paths behind the entry point: the fp32 CUDA-core kernels (every test
without ``tc``) and the tensor-core path (bf16, per-head gate, d = 128: three
runs of the tcgen05 prefill kernel on exchanged operands; the ``tc`` tests).

The oracle's gradient (reverse mode through the recurrence, token by token)
is itself pinned to finite differences of the forward in
``test_oracle_backward_pins.py``.  Here the GPU path is compared with it at
sizes the oracle finishes in seconds that span several 64-token chunks and a
ragged tail, for both gate shapes, every head size, packed batches with empty
sequences, fp32 I/O, the optional inputs and outputs left out, strong decays,
and at the prefill workload's full size, every element.

Error norm: ``max |x - ref| / RMS(ref)`` per gradient.  Tolerances (fp32
arithmetic throughout; no tolerance is stated for the gradient, so these are
derived from the arithmetic): dq, dk, dv and d_init 1e-4 -- each element is an
fp32 sum of at most 64 + d products of exactly represented inputs and decay
factors accurate to a few ulp, so the expected error is ~1e-6 of the RMS;
dg 1e-3 -- every dg_t is a suffix sum over up to T per-token terms, each
itself carrying the error above.  bf16 gradients must equal the fp32 ones
rounded once to nearest-even.
"""
import numpy as np
import pytest
import torch

import gla_inputs
import oracle
from parity import cuda, rel_max, to_np

pytestmark = pytest.mark.gpu

TOL_GRAD = 1e-4
TOL_DG = 1e-3
# tensor-core paths.  The per-key-channel dv run (its prefill rounds P' once
# off the diagonal blocks): the bf16 output tolerance applied to fp32 results.
TOL_GRAD_TC = 2e-2
# The per-head path (three runs of the per-head prefill, whose S', P' and W V
# enter as bf16 hi + lo): gradients measured within 4.5e-5 of their RMS on
# every case below, dg within 1.8e-4 (a suffix sum over up to T tokens of
# 128-channel dot products; full size, T = 2048); bounds about five times the
# measurements.
TOL_GRAD_TC_HEAD = 3e-4
TOL_DG_TC = 1e-3
# strong decays: the reference is the oracle at the clamped gate, and d_init
# (the gradient through the first token's decay) measured 1.3e-3 there
TOL_GRAD_TC_STRONG = 5e-3


def _gla():
    import gated_linear_attention_gla_gb300 as gla
    return gla


def run_gpu(x, gr, grad_dtype=None, need_dg=True, need_d_init=True, init=True, final=True,
            tc=False):
    """The CUDA-core path by default; ``tc`` takes the tensor-core path where it
    covers the call."""
    gla = _gla()
    res = gla.chunk_bwd(cuda(x["q"]), cuda(x["k"]), cuda(x["v"]), cuda(x["g"]),
                        cuda(gr["d_out"]), scale=x["scale"],
                        init_state=cuda(x["init_state"]) if init else None,
                        d_final_state=cuda(gr["d_final_state"]) if final else None,
                        cu_seqlens=cuda(x["cu_seqlens"]), grad_dtype=grad_dtype,
                        need_dg=need_dg, need_d_init=need_d_init, tensor_cores=tc)
    gla.status_sync()
    return res


def run_ref(x, gr, init=True, final=True):
    return oracle.backward(x["q"], x["k"], x["v"], x["g"], x["scale"], gr["d_out"],
                           init_state=x["init_state"] if init else None,
                           d_final=gr["d_final_state"] if final else None,
                           cu_seqlens=x["cu_seqlens"])


NAMES = ("dq", "dk", "dv", "dg", "d_init")


def check(got, ref, tol=TOL_GRAD, tol_dg=TOL_DG, label=""):
    errs = {}
    for name, a, b in zip(NAMES, got, ref):
        if a is None:
            continue
        errs[name] = rel_max(to_np(a), b)
    print(label, {k: f"{v:.2e}" for k, v in errs.items()})
    for name, e in errs.items():
        lim = tol_dg if name == "dg" else tol
        assert e <= lim, f"{label} {name} error {e:.3e} > {lim:.0e}"


def inputs(name="prefill", seed=None, **over):
    x = gla_inputs.prefill_inputs(gla_inputs.WORKLOADS[name], seed=seed, **over)
    return x, gla_inputs.grad_inputs(x, seed=seed)


@pytest.mark.parametrize("gate", ["scalar", "vector"])
def test_backward_matches_oracle(gate):
    # 200 tokens: three full 64-token chunks and a ragged tail of 8
    x, gr = inputs(B=2, T=200, H=3, gate=gate, g_mu=2.0 if gate == "vector" else 3.0)
    got = run_gpu(x, gr, grad_dtype=torch.float32)
    check(got, run_ref(x, gr), label=gate)


@pytest.mark.parametrize("gate", ["scalar", "vector"])
def test_bf16_gradients_are_the_fp32_ones_rounded(gate):
    x, gr = inputs(B=1, T=130, H=2, gate=gate)
    g32 = run_gpu(x, gr, grad_dtype=torch.float32)
    g16 = run_gpu(x, gr)
    for a, b in zip(g16[:3], g32[:3]):
        assert a.dtype == torch.bfloat16
        assert torch.equal(a, b.to(torch.bfloat16))
    assert torch.equal(g16[4], g32[4])


@pytest.mark.parametrize("dk,dv", [(64, 64), (64, 192), (96, 192), (96, 128), (128, 64),
                                   (128, 192)])
@pytest.mark.parametrize("gate", ["scalar", "vector"])
def test_head_sizes(dk, dv, gate):
    x, gr = inputs(B=1, T=100, H=2, dk=dk, dv=dv, gate=gate)
    check(run_gpu(x, gr, grad_dtype=torch.float32), run_ref(x, gr), label=f"{gate} {dk}x{dv}")


@pytest.mark.parametrize("gate", ["scalar", "vector"])
def test_fp32_io(gate):
    x, gr = inputs("tiny", B=2, T=150, gate=gate, init_std=0.05)
    got = run_gpu(x, gr)
    assert got[0].dtype == torch.float32
    check(got, run_ref(x, gr), label=f"fp32 {gate}")


@pytest.mark.parametrize("gate", ["scalar", "vector"])
def test_packed_with_empty_and_short_sequences(gate):
    x, gr = inputs("varlen", lengths=[70, 0, 1, 129, 64, 5], H=2, gate=gate)
    got = run_gpu(x, gr, grad_dtype=torch.float32)
    ref = run_ref(x, gr)
    check(got, ref, label=f"packed {gate}")
    # the empty sequence hands d_final through to d_init
    assert torch.equal(got[4][1].cpu(), gr["d_final_state"][1])


def test_optional_inputs_and_outputs_left_out():
    x, gr = inputs(B=2, T=90, H=2)
    ref = run_ref(x, gr, init=False, final=False)
    got = run_gpu(x, gr, grad_dtype=torch.float32, init=False, final=False)
    check(got, ref, label="no init/final")
    dq, dk, dv, dg, d0 = run_gpu(x, gr, grad_dtype=torch.float32, need_dg=False,
                                 need_d_init=False, init=False, final=False)
    assert dg is None and d0 is None
    assert torch.equal(dq, got[0]) and torch.equal(dk, got[1]) and torch.equal(dv, got[2])


@pytest.mark.parametrize("gate", ["scalar", "vector"])
def test_strong_and_clamped_decays(gate):
    """Gates around -40 (down to -125).  The kernels raise gates below -30 to
    -30, so their gradients are those of the clamped gate: the reference is the
    oracle's gradient at max(g, -30) (it moves dq, dk, dv by ~1e-12 but d_init,
    the gradient through the first token's decay, by a few per cent).  dg comes
    from suffix sums of per-token terms x_t = q_t dq_t - k_t dk_t (summed over
    the key channels for the per-head gate) whose exact total is tiny here
    (RMS(dg) / RMS(x) ~ 1e-4), so its error is bounded in absolute terms: each
    x_t carries a relative error of a few 1e-6 and a suffix has up to T terms,
    hence max |dg - ref| <= 1e-4 RMS(x)."""
    x, gr = inputs(B=1, T=140, H=2, gate=gate, g_mu=-2.0, g_div=0.05)
    assert float(x["g"].min()) < -30
    xc = dict(x, g=x["g"].clamp(min=-30.0))
    got = run_gpu(x, gr, grad_dtype=torch.float32)
    ref = run_ref(xc, gr)
    check(got[:3] + (None,) + got[4:], ref, label=f"strong {gate}")
    terms = to_np(x["q"]) * ref[0] - to_np(x["k"]) * ref[1]
    if gate == "scalar":
        terms = terms.sum(-1)
    err = float(np.max(np.abs(to_np(got[3]) - ref[3])))
    scale_x = float(np.sqrt(np.mean(terms * terms)))
    print(f"strong {gate} dg: max err {err:.2e}, RMS(x) {scale_x:.2e}, "
          f"RMS(dg) {float(np.sqrt(np.mean(ref[3] ** 2))):.2e}")
    assert err <= 1e-4 * scale_x


def test_empty_batch_and_zero_length():
    gla = _gla()
    x, gr = inputs(B=2, T=0, H=2)
    res = gla.chunk_bwd(cuda(x["q"]), cuda(x["k"]), cuda(x["v"]), cuda(x["g"]),
                        cuda(gr["d_out"]), init_state=cuda(x["init_state"]),
                        d_final_state=cuda(gr["d_final_state"]))
    gla.status_sync()
    assert torch.equal(res[4].cpu(), gr["d_final_state"])


@pytest.mark.parametrize("gate", ["scalar", "vector"])
def test_full_size(gate):
    """The prefill workload at full size (B=4, H=16, T=2048) -- the launch
    configuration the benchmark times -- every element of every gradient
    against the oracle."""
    over = {} if gate == "scalar" else dict(gate="vector", g_mu=2.0, g_div=4.0)
    x, gr = inputs(**over)
    got = run_gpu(x, gr, grad_dtype=torch.float32)
    check(got, run_ref(x, gr), label=f"full {gate}")


# --------------------------------------------------------------------------
# tensor-core path
# --------------------------------------------------------------------------
def test_tc_path_is_taken_only_where_it_applies():
    from gated_linear_attention_gla_gb300 import _binding as b
    assert b.chunk_bwd_workspace_size(2, 3, 200, 128, 128, 0, 0) > 0
    assert b.chunk_bwd_workspace_size(2, 3, 200, 128, 128, 0, b.GLA_FLAG_VECTOR_GATE) > 0
    assert b.chunk_bwd_workspace_size(2, 3, 200, 96, 192, 0, 0) == 0
    assert b.chunk_bwd_workspace_size(2, 3, 200, 128, 128, 0, b.GLA_FLAG_FP32_IO) == 0


@pytest.mark.parametrize("T", [200, 300])
def test_tc_per_key_channel_gate(T):
    """Per-key-channel gate with a workspace: dq, dk, dg and d_init from the
    CUDA-core kernels (their tolerances), dv from the reversed run of the
    per-key-channel tensor-core prefill (the prefill's tolerance)."""
    x, gr = inputs(B=2, T=T, H=2, gate="vector", g_mu=2.0, g_div=4.0)
    got = run_gpu(x, gr, grad_dtype=torch.float32, tc=True)
    ref = run_ref(x, gr)
    check((got[0], got[1], None, got[3], got[4]), ref, label="tc vec (cuda-core part)")
    check((None, None, got[2], None, None), ref, tol=TOL_GRAD_TC, label="tc vec dv")
    g16 = run_gpu(x, gr, tc=True)
    assert torch.equal(g16[2], got[2].to(torch.bfloat16))


def test_tc_per_key_channel_gate_packed_and_full_size():
    x, gr = inputs("varlen", lengths=[300, 0, 1, 129], H=2, gate="vector", g_mu=2.0, g_div=4.0)
    got = run_gpu(x, gr, grad_dtype=torch.float32, tc=True)
    check((None, None, got[2], None, None), run_ref(x, gr), tol=TOL_GRAD_TC,
          label="tc vec packed dv")
    x, gr = inputs(gate="vector", g_mu=2.0, g_div=4.0)
    got = run_gpu(x, gr, grad_dtype=torch.float32, tc=True)
    check((None, None, got[2], None, None), run_ref(x, gr), tol=TOL_GRAD_TC,
          label="tc vec full-size dv")


def test_tc_backward_matches_oracle():
    x, gr = inputs(B=2, T=300, H=3)   # two full 128-token chunks and a ragged tail
    got = run_gpu(x, gr, grad_dtype=torch.float32, tc=True)
    check(got, run_ref(x, gr), tol=TOL_GRAD_TC_HEAD, tol_dg=TOL_DG_TC, label="tc")


def test_tc_bf16_gradients_are_the_fp32_ones_rounded():
    x, gr = inputs(B=1, T=260, H=2)
    g32 = run_gpu(x, gr, grad_dtype=torch.float32, tc=True)
    g16 = run_gpu(x, gr, tc=True)
    for a, b in zip(g16[:3], g32[:3]):
        assert a.dtype == torch.bfloat16 and torch.equal(a, b.to(torch.bfloat16))
    assert torch.equal(g16[4], g32[4])


def test_tc_packed_with_empty_and_short_sequences():
    x, gr = inputs("varlen", lengths=[300, 0, 1, 129, 128, 5], H=2)
    got = run_gpu(x, gr, grad_dtype=torch.float32, tc=True)
    check(got, run_ref(x, gr), tol=TOL_GRAD_TC_HEAD, tol_dg=TOL_DG_TC, label="tc packed")
    # the empty sequence hands d_final through (as (d_final / scale) * scale)
    torch.testing.assert_close(got[4][1].cpu(), gr["d_final_state"][1], rtol=1e-6, atol=0)


def test_tc_optional_inputs_and_outputs_left_out():
    x, gr = inputs(B=2, T=200, H=2)
    got = run_gpu(x, gr, grad_dtype=torch.float32, init=False, final=False, tc=True)
    check(got, run_ref(x, gr, init=False, final=False), tol=TOL_GRAD_TC_HEAD, tol_dg=TOL_DG_TC,
          label="tc no init/final")
    dq, dk, dv, dg, d0 = run_gpu(x, gr, grad_dtype=torch.float32, need_dg=False,
                                 need_d_init=False, init=False, final=False, tc=True)
    assert dg is None and d0 is None
    assert torch.equal(dq, got[0]) and torch.equal(dk, got[1]) and torch.equal(dv, got[2])


def test_tc_full_size():
    """The prefill workload at full size (B=4, H=16, T=2048) on the tensor-core
    path: every element of every gradient against the oracle."""
    x, gr = inputs()
    got = run_gpu(x, gr, grad_dtype=torch.float32, tc=True)
    check(got, run_ref(x, gr), tol=TOL_GRAD_TC_HEAD, tol_dg=TOL_DG_TC, label="tc full size")


@pytest.mark.parametrize("T", [1, 127, 128, 129, 256])
def test_tc_chunk_boundaries(T):
    x, gr = inputs(B=2, T=T, H=2)
    got = run_gpu(x, gr, grad_dtype=torch.float32, tc=True)
    check(got, run_ref(x, gr), tol=TOL_GRAD_TC_HEAD, tol_dg=TOL_DG_TC, label=f"tc T={T}")


@pytest.mark.parametrize("dk,dv", [(64, 64), (64, 128), (128, 64)])
def test_tc_head_sizes_64(dk, dv):
    """Head sizes 64 on the tensor-core path: the three runs take (d_v, d_k),
    (d_v, d_k) and (d_k, d_v) as their key and value sizes (a 64 key size runs
    zero-padded to 128, a 64 value size as one slice).  Packed sequences with an
    empty one and a ragged tail, fp32 and bf16 gradients."""
    x, gr = inputs("varlen", lengths=[300, 0, 129, 1], H=3, dk=dk, dv=dv)
    got = run_gpu(x, gr, grad_dtype=torch.float32, tc=True)
    check(got, run_ref(x, gr), tol=TOL_GRAD_TC_HEAD, tol_dg=TOL_DG_TC, label=f"tc {dk}x{dv}")
    g16 = run_gpu(x, gr, tc=True)
    for a, b in zip(g16[:3], got[:3]):
        assert a.dtype == torch.bfloat16 and torch.equal(a, b.to(torch.bfloat16))
    torch.testing.assert_close(got[4][1].cpu(), gr["d_final_state"][1], rtol=1e-6, atol=0)


def test_tc_head_size_64_strong_decays():
    """d_k = d_v = 64 with gates around -40 (every chunk wide in all three runs)."""
    x, gr = inputs(B=1, T=300, H=2, dk=64, dv=64, g_mu=-2.0, g_div=0.05)
    xc = dict(x, g=x["g"].clamp(min=-30.0))
    got = run_gpu(x, gr, grad_dtype=torch.float32, tc=True)
    check(got[:3] + (None,) + got[4:], run_ref(xc, gr), tol=TOL_GRAD_TC_STRONG,
          label="tc 64 strong")


def test_tc_zero_gate():
    """g = 0 (no decay): the gradients are those of causal linear attention."""
    x, gr = inputs(B=1, T=200, H=2)
    x["g"] = torch.zeros_like(x["g"])
    got = run_gpu(x, gr, grad_dtype=torch.float32, tc=True)
    check(got, run_ref(x, gr), tol=TOL_GRAD_TC_HEAD, tol_dg=TOL_DG_TC, label="tc g=0")


def test_tc_strong_decays_take_the_wide_path():
    """Gates around -40 make every chunk "wide" (decay span past 2^96) in the
    three prefill runs, forward and reversed.  As for the CUDA-core path, the
    reference is the oracle at max(g, -30).  dg is then ~1e-4 of its per-token
    terms x_t = sum_i (q dq - k dk), and its error is the suffix sum of those
    terms' own errors.  With the prefill's hi + lo operands the gradients are
    within ~4e-5 of their RMS, and the measured dg error is 1.0e-3 RMS(x) at
    T = 300 (it was 5.2e-2 with operands rounded once); the bound is three
    times the measurement."""
    T = 300
    x, gr = inputs(B=1, T=T, H=2, g_mu=-2.0, g_div=0.05)
    xc = dict(x, g=x["g"].clamp(min=-30.0))
    got = run_gpu(x, gr, grad_dtype=torch.float32, tc=True)
    ref = run_ref(xc, gr)
    check(got[:3] + (None,) + got[4:], ref, tol=TOL_GRAD_TC_STRONG, label="tc strong")
    terms = (to_np(x["q"]) * ref[0] - to_np(x["k"]) * ref[1]).sum(-1)
    err = float(np.max(np.abs(to_np(got[3]) - ref[3])))
    scale_x = float(np.sqrt(np.mean(terms * terms)))
    print(f"tc strong dg: max err {err / scale_x:.2e} RMS(x)")
    assert err <= 3e-3 * scale_x


def test_tc_minus_inf_gate_resets():
    """A gate of -inf at one token erases the state there (clamped to -30 on the
    GPU): the gradient reaching across it is below 1e-13."""
    x, gr = inputs(B=1, T=260, H=2)
    x["g"][0, 130, :] = float("-inf")
    xc = dict(x, g=x["g"].clamp(min=-30.0))
    got = run_gpu(x, gr, grad_dtype=torch.float32, tc=True)
    check(got, run_ref(xc, gr), tol=TOL_GRAD_TC_HEAD, tol_dg=TOL_DG_TC, label="tc -inf")


def test_tc_per_key_channel_strong_decays():
    """Per-key-channel gates around -1.3 make every chunk "wide" in the reversed
    per-key-channel prefill run that gives dv (token by token there); the
    reference is the oracle's gradient at max(g, -30)."""
    x, gr = inputs(B=1, T=300, H=2, gate="vector", g_mu=-1.0, g_div=1.0)
    xc = dict(x, g=x["g"].clamp(min=-30.0))
    got = run_gpu(x, gr, grad_dtype=torch.float32, tc=True)
    check((None, None, got[2], None, None), run_ref(xc, gr), tol=TOL_GRAD_TC,
          label="tc vec strong dv")
