"""The mixer's steps after the readout (self-augmentation, head RMSNorm, SiLU
output gate) on the GPU, against the fp64 oracle: after every prefill kernel
(gla_chunk_fwd_mixer: inside the per-key-channel kernel; a pass over the
output after the per-head and CUDA-core kernels) and fused into the decode
step.

The check is split in two.  The readout o itself must match the oracle within
the output tolerance (as everywhere); the epilogue, applied by the GPU to that
o, must match the oracle's epilogue applied to the same o (the GPU's fp32
readout, widened) within 1e-5 of the result's RMS -- fp32 arithmetic against
fp64.  A direct comparison of the two composites would charge the epilogue
with the readout's rounding, magnified elementwise by the gate (|silu(z)| up
to ~4 against an RMS of ~0.8) and row by row by the normalisation."""
import numpy as np
import pytest
import torch

import gla_inputs
import oracle
from parity import TOL_STATE, cuda, out_tol, rel_max, to_np

pytestmark = pytest.mark.gpu

STEPS = {"aug": ("aug",), "norm": ("norm_w", "eps"), "gate": ("z",),
         "all": ("aug", "norm_w", "eps", "z")}


def _gla():
    import gated_linear_attention_gla_gb300 as gla
    return gla


def _pick(m, which):
    return {k: m[k] for k in STEPS[which]}


def _ref_epilogue(o_ref, x, m, which, q=None, k=None, v=None):
    q = x["q"] if q is None else q
    k = x["k"] if k is None else k
    v = x["v"] if v is None else v
    return oracle.mixer_epilogue(o_ref, q, k, v, aug=m["aug"] if "aug" in STEPS[which] else None,
                                 norm_w=m["norm_w"] if "norm_w" in STEPS[which] else None,
                                 eps=m["eps"], z=m["z"] if "z" in STEPS[which] else None)


@pytest.mark.parametrize("which", sorted(STEPS))
@pytest.mark.parametrize("case", ["tc_scalar", "tc_vector", "laplace", "simt_fp32"])
def test_prefill_with_mixer_epilogue(cuda_ok, case, which):
    gla = _gla()
    if case == "tc_scalar":
        w, kw = gla_inputs.WORKLOADS["prefill"], dict(B=2, T=300, H=4)
    elif case == "tc_vector":
        w, kw = gla_inputs.WORKLOADS["vector"], dict(B=2, T=300, H=4, init_std=0.02)
    elif case == "laplace":
        w, kw = gla_inputs.WORKLOADS["laplace"], dict(B=2, T=300, H=16)
    else:
        w, kw = gla_inputs.WORKLOADS["tiny"], dict(B=2, T=150, H=2, chunk=64, init_std=0.1)
    x = gla_inputs.prefill_inputs(w, seed=31, **kw)
    m = gla_inputs.mixer_inputs(w, x["q"].shape[:-2], seed=31, **{k: kw[k] for k in ("H",)})
    mix = {k: cuda(v) if torch.is_tensor(v) else v for k, v in _pick(m, which).items()}
    args = (cuda(x["q"]), cuda(x["k"]), cuda(x["v"]), cuda(x["g"]))
    kw = dict(scale=x["scale"], init_state=cuda(x["init_state"]), chunk=x["chunk"],
              out_dtype=torch.float32)
    o, _ = gla.chunk_fwd(*args, **kw)
    y, fin = gla.chunk_fwd(*args, mixer=mix, **kw)
    gla.status_sync()
    o_ref, s_ref = oracle.recurrent(x["q"], x["k"], x["v"], x["g"], x["scale"],
                                    init_state=x["init_state"])
    tol = out_tol(x["q"].dtype)
    assert rel_max(to_np(o), o_ref) <= tol
    assert rel_max(to_np(fin), s_ref) <= (TOL_STATE if x["q"].dtype == torch.bfloat16 else 1e-5)
    if case == "tc_vector":
        _check_fused(o, y, o_ref, x, m, which)
    else:
        e = rel_max(to_np(y), _ref_epilogue(to_np(o), x, m, which))
        assert e <= 1e-5, f"epilogue error {e:.3e}"


def _check_fused(o, y, o_ref, x, m, which):
    """The per-key-channel kernel applies the steps inside the kernel (the
    augmentation through P''s diagonal, the RMSNorm and the gate before the
    store), so its readout is never stored on its own and cannot be fed to
    the oracle's epilogue.  Its composite is measured against the exact
    composite instead, next to the composite the two-step path would give
    (the oracle's epilogue applied exactly to this kernel's plain readout):
    both carry the readout's rounding, magnified by the gate."""
    y_ref = _ref_epilogue(o_ref, x, m, which)
    e_fused = rel_max(to_np(y), y_ref)
    e_two_step = rel_max(_ref_epilogue(to_np(o), x, m, which), y_ref)
    print(f"fused composite error {e_fused:.3e}, two-step {e_two_step:.3e}")
    assert e_fused <= 1.5 * e_two_step + 2e-3, (e_fused, e_two_step)


def test_epilogue_entry_point_matches_oracle_on_a_given_output(cuda_ok):
    """gla_mixer_epilogue alone, over an fp32 output that is the oracle's own
    readout: only the epilogue's arithmetic is measured (fp32 vs fp64)."""
    gla = _gla()
    from gated_linear_attention_gla_gb300 import _binding
    w = gla_inputs.WORKLOADS["laplace"]
    x = gla_inputs.prefill_inputs(w, seed=5, B=1, T=64, H=16)
    m = gla_inputs.mixer_inputs(w, x["q"].shape[:-2], seed=5)
    o_ref, _ = oracle.recurrent(x["q"], x["k"], x["v"], x["g"], x["scale"],
                                init_state=x["init_state"])
    out = torch.tensor(o_ref, dtype=torch.float32).cuda().contiguous()
    args = {n: cuda(x[n]) for n in ("q", "k", "v")}
    mix = {n: cuda(m[n]) for n in ("aug", "norm_w", "z")}
    rc = _binding.gla_mixer_epilogue(out.data_ptr(), args["q"].data_ptr(), args["k"].data_ptr(),
                                     args["v"].data_ptr(), mix["aug"].data_ptr(),
                                     mix["norm_w"].data_ptr(), m["eps"], mix["z"].data_ptr(),
                                     64, 16, 96, 192, torch.cuda.current_stream().cuda_stream,
                                     _binding.GLA_FLAG_FP32_OUT)
    assert rc == 0
    gla.status_sync()
    y_ref = _ref_epilogue(o_ref, x, m, "all")
    assert rel_max(to_np(out), y_ref) <= 1e-5


@pytest.mark.parametrize("which", sorted(STEPS))
@pytest.mark.parametrize("dk,dv,gate", [(128, 128, "scalar"), (96, 192, "scalar"),
                                        (128, 128, "vector")])
def test_decode_step_with_fused_mixer(cuda_ok, dk, dv, gate, which):
    gla = _gla()
    w = gla_inputs.WORKLOADS["decode"]
    d = gla_inputs.decode_inputs(w, steps=2, N=6, H=4, dk=dk, dv=dv, gate=gate)
    m = gla_inputs.mixer_inputs(w, (6,), seed=3, H=4, dk=dk, dv=dv)
    mix = {k: cuda(v) if torch.is_tensor(v) else v for k, v in _pick(m, which).items()}
    S = cuda(d["state"]).clone()
    S_ref = d["state"].double().numpy()
    for t in range(2):
        args = [cuda(d[n][t]) for n in ("q", "k", "v", "g")]
        S_plain = S.clone()
        o = gla.decode_step(*args, S_plain, scale=d["scale"], out_dtype=torch.float32)
        y = gla.decode_step(*args, S, scale=d["scale"], out_dtype=torch.float32, mixer=mix)
        gla.status_sync()
        assert torch.equal(S, S_plain), t  # the epilogue leaves the state step alone
        o_ref, S_ref = oracle.decode_step(d["q"][t], d["k"][t], d["v"][t], d["g"][t],
                                          d["scale"], S_ref)
        assert rel_max(to_np(o), o_ref) <= out_tol(torch.bfloat16), t
        y_ref = _ref_epilogue(to_np(o), None, m, which, d["q"][t], d["k"][t], d["v"][t])
        e = rel_max(to_np(y), y_ref)
        assert e <= 1e-5, f"step {t}: epilogue error {e:.3e}"
    assert rel_max(to_np(S), S_ref) <= 1e-5


def test_decode_mixer_on_slot_pages(cuda_ok):
    """The fused epilogue with slot-indexed pages and a padding row."""
    gla = _gla()
    w = gla_inputs.WORKLOADS["decode"]
    d = gla_inputs.decode_inputs(w, steps=1, N=3, H=2)
    m = gla_inputs.mixer_inputs(w, (3,), seed=4, H=2)
    mix = {k: cuda(v) if torch.is_tensor(v) else v for k, v in m.items()}
    pool = torch.zeros(5, 2, w.dk, w.dv)
    pool[[4, 1]] = d["state"][[0, 2]]
    pool_gpu = cuda(pool).contiguous()
    slots = cuda(torch.tensor([4, -1, 1], dtype=torch.int32))
    args = [cuda(d[n][0]) for n in ("q", "k", "v", "g")]
    o = torch.zeros(3, 2, w.dv, device="cuda")
    gla.decode_step(*args, pool_gpu.clone(), scale=d["scale"], out=o, slots=slots)
    out = torch.zeros(3, 2, w.dv, device="cuda")
    gla.decode_step(*args, pool_gpu, scale=d["scale"], out=out, slots=slots, mixer=mix)
    gla.status_sync()
    live = [0, 2]
    o_ref, _ = oracle.decode_step(d["q"][0][live], d["k"][0][live], d["v"][0][live],
                                  d["g"][0][live], d["scale"], d["state"][live])
    assert rel_max(to_np(o[live]), o_ref) <= out_tol(torch.bfloat16)
    y_ref = oracle.mixer_epilogue(to_np(o[live]), d["q"][0][live], d["k"][0][live],
                                  d["v"][0][live], aug=m["aug"], norm_w=m["norm_w"], eps=m["eps"],
                                  z=m["z"][live])
    assert rel_max(to_np(out[live]), y_ref) <= 1e-5
    assert (out[1] == 0).all()


def _vector_case(seed=41, **over):
    w = gla_inputs.WORKLOADS["vector"]
    kw = dict(B=2, T=300, H=4, init_std=0.02)
    kw.update(over)
    x = gla_inputs.prefill_inputs(w, seed=seed, **kw)
    m = gla_inputs.mixer_inputs(w, x["q"].shape[:-2], seed=seed, H=kw.get("H", 4))
    return x, m


def _run_vector(x, m, out_dtype):
    gla = _gla()
    mix = {k: cuda(v) if torch.is_tensor(v) else v for k, v in m.items()}
    args = (cuda(x["q"]), cuda(x["k"]), cuda(x["v"]), cuda(x["g"]))
    kw = dict(scale=x["scale"], init_state=cuda(x["init_state"]),
              cu_seqlens=cuda(x["cu_seqlens"]), chunk=128, out_dtype=out_dtype)
    o, _ = gla.chunk_fwd(*args, **kw)
    y, _ = gla.chunk_fwd(*args, mixer=mix, **kw)
    gla.status_sync()
    return o, y


def test_vector_mixer_on_wide_chunks(cuda_ok):
    """Strong per-channel decays make every chunk "wide" (processed token by
    token by the per-key-channel kernel); the steps follow as for any output."""
    x, m = _vector_case(g_mu=-1.0, g_div=1.0)
    o, y = _run_vector(x, m, torch.float32)
    o_ref, _ = oracle.recurrent(x["q"], x["k"], x["v"], x["g"], x["scale"],
                                init_state=x["init_state"])
    assert rel_max(to_np(o), o_ref) <= out_tol(torch.bfloat16)
    e = rel_max(to_np(y), _ref_epilogue(to_np(o), x, m, "all"))
    assert e <= 1e-5, f"epilogue error {e:.3e}"


def test_vector_mixer_packed(cuda_ok):
    w = gla_inputs.WORKLOADS["vector"]
    x = gla_inputs.prefill_inputs(w, seed=43, lengths=[300, 0, 1, 129], H=2, init_std=0.02)
    m = gla_inputs.mixer_inputs(w, x["q"].shape[:-2], seed=43, H=2)
    o, y = _run_vector(x, m, torch.float32)
    o_ref, _ = oracle.recurrent(x["q"], x["k"], x["v"], x["g"], x["scale"],
                                init_state=x["init_state"], cu_seqlens=x["cu_seqlens"])
    _check_fused(o, y, o_ref, x, m, "all")


@pytest.mark.parametrize("g_mu,g_div", [(2.0, 4.0), (-1.0, 1.0)], ids=["tensor_core", "wide"])
def test_vector_mixer_bf16_output_is_the_fp32_result_rounded(cuda_ok, g_mu, g_div):
    """The fused per-key-channel kernel computes the same fp32 values for either
    output type and rounds them once for a bf16 output (tensor-core chunks and
    wide chunks, which apply the steps in the token-by-token path)."""
    from parity import check_bf16_rounding
    x, m = _vector_case(seed=47, g_mu=g_mu, g_div=g_div)
    _, y32 = _run_vector(x, m, torch.float32)
    _, y16 = _run_vector(x, m, torch.bfloat16)
    check_bf16_rounding(y16, y32)


def test_vector_mixer_full_size(cuda_ok):
    """The fused per-key-channel mixer on the whole full-size vector workload
    (B=8, T=4096, H=16), every element: its composite against the exact one,
    next to the two-step composite of the same kernel's plain readout."""
    w = gla_inputs.WORKLOADS["vector"]
    x = gla_inputs.prefill_inputs(w)
    m = gla_inputs.mixer_inputs(w, x["q"].shape[:-2])
    o, y = _run_vector(x, m, torch.float32)
    o_ref, _ = oracle.recurrent(x["q"], x["k"], x["v"], x["g"], x["scale"],
                                init_state=x["init_state"])
    _check_fused(o, y, o_ref, x, m, "all")


def _per_head_case(seed=51, w="prefill", **over):
    w = gla_inputs.WORKLOADS[w]
    kw = dict(B=2, T=300, H=4)
    kw.update(over)
    x = gla_inputs.prefill_inputs(w, seed=seed, **kw)
    m = gla_inputs.mixer_inputs(w, x["q"].shape[:-2], seed=seed, H=kw["H"])
    return x, m


def _run_per_head(x, m):
    """The per-head kernel's plain readout and its mixer call (the kernel, then
    the pass over its output), fp32 outputs, and the oracle's readout."""
    gla = _gla()
    mix = {k: cuda(v) if torch.is_tensor(v) else v for k, v in m.items()}
    args = (cuda(x["q"]), cuda(x["k"]), cuda(x["v"]), cuda(x["g"]))
    kw = dict(scale=x["scale"], init_state=cuda(x["init_state"]), chunk=128,
              out_dtype=torch.float32)
    if x["cu_seqlens"] is not None:
        kw["cu_seqlens"] = cuda(x["cu_seqlens"])
    o, _ = gla.chunk_fwd(*args, **kw)
    y, _ = gla.chunk_fwd(*args, mixer=mix, **kw)
    gla.status_sync()
    o_ref, _ = oracle.recurrent(x["q"], x["k"], x["v"], x["g"], x["scale"],
                                init_state=x["init_state"], cu_seqlens=x["cu_seqlens"])
    return o, y, o_ref


def _check_two_step(o, y, o_ref, x, m):
    assert rel_max(to_np(o), o_ref) <= out_tol(torch.bfloat16)
    e = rel_max(to_np(y), _ref_epilogue(to_np(o), x, m, "all"))
    assert e <= 1e-5, f"epilogue error {e:.3e}"


@pytest.mark.parametrize("mu", [-3.0, 8.0], ids=["wide", "weak"])
def test_per_head_mixer_strong_and_weak_decay(cuda_ok, mu):
    """g = logsigmoid(N(mu, 1)): mu = -3 makes every chunk "wide" (the explicit
    decays), mu = 8 keeps nearly all memory."""
    x, m = _per_head_case()
    gen = torch.Generator().manual_seed(53)
    x["g"] = torch.nn.functional.logsigmoid(torch.randn(x["g"].shape, generator=gen) + mu)
    _check_two_step(*_run_per_head(x, m), x, m)


def test_per_head_mixer_packed(cuda_ok):
    """Packed sequences, an empty one and a one-token one among them."""
    x, m = _per_head_case(lengths=[300, 0, 1, 129], H=2)
    _check_two_step(*_run_per_head(x, m), x, m)


def test_per_head_mixer_zero_scale(cuda_ok):
    """scale = 0: the readout is exactly zero and the steps still apply (the
    self-augmentation term alone reaches the output)."""
    x, m = _per_head_case(seed=55)
    x["scale"] = 0.0
    o, y, o_ref = _run_per_head(x, m)
    assert float(o.abs().max()) == 0.0
    _check_two_step(o, y, o_ref, x, m)


@pytest.mark.parametrize("wname", ["prefill", "laplace"])
def test_per_head_mixer_full_size(cuda_ok, wname):
    """The per-head kernel and the pass on the whole full-size workload, every
    element."""
    w = gla_inputs.WORKLOADS[wname]
    x = gla_inputs.prefill_inputs(w)
    m = gla_inputs.mixer_inputs(w, x["q"].shape[:-2])
    _check_two_step(*_run_per_head(x, m), x, m)
