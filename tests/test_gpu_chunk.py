"""GPU chunked prefill (gla_chunk_fwd) against the fp64 oracle.

Covers both kernels behind the entry point -- the fp32 CUDA-core path (fp32
I/O, chunk sizes 16/32/64) and the bf16 tensor-core path (chunk 128) -- at
sizes the oracle finishes in seconds that still span several chunks and a
ragged tail, the edge cases (T = 1, T < chunk, empty and length-1 packed
sequences, no initial/final state, in-place state, g = -inf), the method's
invariants on the GPU path, and every workload at full size, every element
of the output and final state.
"""
import numpy as np
import pytest
import torch

import gla_inputs
import oracle
from parity import TOL_STATE, check_bf16_rounding, cuda, out_tol, rel_max, to_np

pytestmark = pytest.mark.gpu


def _gla():
    import gated_linear_attention_gla_gb300 as gla
    return gla


def run_gpu(x, chunk=None, init=True, final=True, pair=True):
    """Run the GPU path.  For bf16 inputs (``pair``) run it twice -- bf16 and
    fp32 output -- check the bf16 output is the fp32 one rounded once, and
    return the fp32 result (the one the tolerance applies to)."""
    gla = _gla()
    args = (cuda(x["q"]), cuda(x["k"]), cuda(x["v"]), cuda(x["g"]))
    kw = dict(scale=x["scale"], init_state=cuda(x["init_state"]) if init else None,
              cu_seqlens=cuda(x["cu_seqlens"]), chunk=chunk or x["chunk"],
              output_final_state=final)
    out, fin = gla.chunk_fwd(*args, **kw)
    gla.status_sync()
    if x["q"].dtype != torch.bfloat16 or not pair:
        return out, fin
    out32, fin32 = gla.chunk_fwd(*args, out_dtype=torch.float32, **kw)
    gla.status_sync()
    check_bf16_rounding(out, out32)
    if fin is not None:
        assert torch.equal(fin, fin32)
    return out32, fin


def run_ref(x, init=True):
    return oracle.recurrent(x["q"], x["k"], x["v"], x["g"], x["scale"],
                            init_state=x["init_state"] if init else None,
                            cu_seqlens=x["cu_seqlens"])


def check(x, out, fin, o_ref, s_ref, state_tol=None):
    """``out`` is the fp32 result (fp32 output mode for bf16 inputs)."""
    tol = out_tol(x["q"].dtype)
    e_o = rel_max(to_np(out), o_ref)
    assert e_o <= tol, f"output error {e_o:.3e} > {tol:.0e}"
    if fin is not None:
        st = state_tol if state_tol is not None else (
            TOL_STATE if x["q"].dtype == torch.bfloat16 else 1e-5)
        e_s = rel_max(to_np(fin), s_ref)
        assert e_s <= st, f"state error {e_s:.3e} > {st:.0e}"


def small(name="prefill", **kw):
    w = gla_inputs.WORKLOADS[name]
    return gla_inputs.prefill_inputs(w, seed=kw.pop("seed", 11), **kw)


# ---------------------------------------------------------------------------
# The tiny fp32 workload, whole (tolerance 1e-5).
# ---------------------------------------------------------------------------
def test_tiny_fp32_workload(cuda_ok):
    x = gla_inputs.prefill_inputs(gla_inputs.WORKLOADS["tiny"])
    out, fin = run_gpu(x)
    o_ref, s_ref = run_ref(x)
    assert out.dtype == torch.float32
    check(x, out, fin, o_ref, s_ref)


@pytest.mark.parametrize("chunk", [16, 32, 64, 128])
@pytest.mark.parametrize("gate", ["scalar", "vector"])
def test_fp32_path_chunk_sizes(cuda_ok, chunk, gate):
    x = small("tiny", B=2, T=203, H=3, gate=gate, init_std=0.05, chunk=chunk)
    out, fin = run_gpu(x)
    check(x, out, fin, *run_ref(x))


@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 128), (64, 128), (128, 64), (96, 192)])
def test_fp32_path_head_sizes(cuda_ok, dk, dv):
    x = small("tiny", B=1, T=150, H=2, dk=dk, dv=dv, init_std=0.1, chunk=64)
    out, fin = run_gpu(x)
    check(x, out, fin, *run_ref(x))


# ---------------------------------------------------------------------------
# bf16 I/O: tensor-core path (chunk 128) and CUDA-core path (chunk 64).
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("chunk", [128, 64])
@pytest.mark.parametrize("gate", ["scalar", "vector"])
@pytest.mark.parametrize("dk,dv", [(128, 128), (64, 64), (128, 64), (64, 128), (96, 192)])
def test_bf16_small(cuda_ok, chunk, gate, dk, dv):
    x = small(B=2, T=333, H=3, dk=dk, dv=dv, gate=gate, chunk=chunk,
              g_div=4.0 if gate == "vector" else 1.0)
    out, fin = run_gpu(x)
    check(x, out, fin, *run_ref(x))


@pytest.mark.parametrize("T", [1, 2, 127, 128, 129, 256, 257])
def test_bf16_lengths_around_the_chunk(cuda_ok, T):
    x = small(B=2, T=T, H=2)
    out, fin = run_gpu(x)
    check(x, out, fin, *run_ref(x))


def test_laplace_head_with_the_fixed_decay_schedule(cuda_ok):
    """The Laplace 3B head (d_k = 96, d_v = 192) with the page's fixed per-head
    decays, several chunks and a ragged tail, on the tensor-core path."""
    x = small("laplace", B=2, T=333, H=16)
    out, fin = run_gpu(x)
    check(x, out, fin, *run_ref(x))


@pytest.mark.parametrize("mu", [-3.0, 8.0, None])
def test_tensor_core_key_head_64(cuda_ok, mu):
    """d_k = 64 on the tensor-core kernel: the second 64-channel panel of Q and K
    lies wholly outside the tensor and is zero-filled, so state rows 64..127
    stay zero.  Packed sequences (an empty one, a length-1 one, one longer than
    several chunks) with very strong (mu = -3), very weak (mu = 8) and the
    workload's own decays."""
    x = small(B=0, lengths=[300, 1, 0, 129, 520], H=3, dk=64, dv=128, init_std=0.05)
    if mu is not None:
        gen = torch.Generator().manual_seed(6)
        x["g"] = torch.nn.functional.logsigmoid(torch.randn(x["g"].shape, generator=gen) + mu)
    out, fin = run_gpu(x)
    check(x, out, fin, *run_ref(x))
    assert torch.equal(fin[2].cpu(), x["init_state"][2])


@pytest.mark.parametrize("gate", ["scalar", "vector"])
def test_bf16_no_initial_state_no_final_state(cuda_ok, gate):
    x = small(B=2, T=300, H=2, gate=gate)
    out, fin = run_gpu(x, init=False, final=False)
    assert fin is None
    o_ref, _ = run_ref(x, init=False)
    check(x, out, None, o_ref, None)


@pytest.mark.parametrize("gate", ["scalar", "vector"])
def test_final_state_in_place_over_initial_state(cuda_ok, gate):
    gla = _gla()
    x = small(B=2, T=260, H=2, gate=gate, init_std=0.05)
    S = cuda(x["init_state"]).clone()
    out, fin = gla.chunk_fwd(cuda(x["q"]), cuda(x["k"]), cuda(x["v"]), cuda(x["g"]),
                             scale=x["scale"], init_state=S, final_state=S, chunk=128,
                             out_dtype=torch.float32)
    gla.status_sync()
    assert fin.data_ptr() == S.data_ptr()
    check(x, out, fin, *run_ref(x))


@pytest.mark.parametrize("gate", ["scalar", "vector"])
def test_minus_inf_gate_inside_chunks(cuda_ok, gate):
    x = small(B=1, T=300, H=2, gate=gate)
    g = x["g"].clone()
    g[:, 5] = float("-inf")          # first chunk
    g[:, 170] = float("-inf")        # second chunk, mid
    g[:, 256] = float("-inf")        # chunk start
    x["g"] = g
    out, fin = run_gpu(x)
    assert torch.isfinite(out.float()).all() and torch.isfinite(fin).all()
    check(x, out, fin, *run_ref(x))


@pytest.mark.parametrize("gate", ["scalar", "vector"])
@pytest.mark.parametrize("positions", [[5, 40, 90], [0, 1, 2, 127], [64, 65, 66, 200, 201, 202],
                                       [10, 20, 30, 40, 50]])
def test_several_resets_in_one_chunk(cuda_ok, positions, gate):
    """-inf gates (clamped at -30, 43 in log2 each): three or more in one chunk
    push its decay span past 2^96 -- two such chunks in a row in the third
    case -- so the per-head kernel takes its explicit-decay path for them and
    the per-key-channel kernel its token-by-token path."""
    x = small(B=2, T=300, H=2, gate=gate)
    g = x["g"].clone()
    g[:, positions] = float("-inf")
    x["g"] = g
    out, fin = run_gpu(x)
    assert torch.isfinite(out).all() and torch.isfinite(fin).all()
    check(x, out, fin, *run_ref(x))


@pytest.mark.parametrize("gate", ["scalar", "vector"])
@pytest.mark.parametrize("mu", [-3.0, 0.0, 8.0])
def test_strong_and_weak_decay(cuda_ok, mu, gate):
    """g = logsigmoid(N(mu, 1)): mu = -3 makes every chunk's decay span far wider
    than 2^96 (explicit / token-by-token path throughout), mu = 8 keeps nearly
    all memory (the lo half of the state update matters in every chunk)."""
    x = small(B=2, T=400, H=2, gate=gate)
    gen = torch.Generator().manual_seed(5)
    x["g"] = torch.nn.functional.logsigmoid(torch.randn(x["g"].shape, generator=gen) + mu)
    out, fin = run_gpu(x)
    check(x, out, fin, *run_ref(x))


def test_vector_gate_mixed_channel_decays(cuda_ok):
    """Per-key-channel decays from nearly none to very strong in the same head
    (channel i: g = logsigmoid(N(mu_i, 1)), mu_i from -4 to 8), and chunks that
    alternate between the tensor-core and the token-by-token path."""
    x = small(B=2, T=700, H=2, gate="vector")
    gen = torch.Generator().manual_seed(9)
    mu = torch.linspace(-4.0, 8.0, x["g"].shape[-1])
    g = torch.nn.functional.logsigmoid(torch.randn(x["g"].shape, generator=gen) + mu)
    g[:, 128:256] = torch.nn.functional.logsigmoid(
        torch.randn(g[:, 128:256].shape, generator=gen) + 4.0)   # a mild chunk
    g[:, 400:410] = float("-inf")                                 # a chunk with ten resets
    x["g"] = g
    out, fin = run_gpu(x)
    assert torch.isfinite(out).all() and torch.isfinite(fin).all()
    check(x, out, fin, *run_ref(x))


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_output_buffer_only_16_byte_aligned(cuda_ok, out_dtype):
    """An output that is 16- but not 32-byte aligned takes 128-bit stores; the
    result is bit-identical to the one written into a fresh (aligned) tensor."""
    gla = _gla()
    x = small(B=2, T=300, H=2)
    args = (cuda(x["q"]), cuda(x["k"]), cuda(x["v"]), cuda(x["g"]))
    kw = dict(scale=x["scale"], init_state=cuda(x["init_state"]), chunk=128)
    ref, _ = gla.chunk_fwd(*args, out_dtype=out_dtype, **kw)
    shift = 16 // torch.empty((), dtype=out_dtype).element_size()
    buf = torch.full((ref.numel() + 2 * shift,), float("nan"), dtype=out_dtype, device="cuda")
    out = buf[shift:shift + ref.numel()].view(ref.shape)
    assert out.data_ptr() % 32 == 16
    got, _ = gla.chunk_fwd(*args, out=out, out_dtype=out_dtype, **kw)
    gla.status_sync()
    assert got.data_ptr() == out.data_ptr()
    assert torch.equal(got, ref)
    assert torch.isnan(buf[:shift]).all() and torch.isnan(buf[shift + ref.numel():]).all()


def test_packed_sequences_with_empty_and_short_ones(cuda_ok):
    x = small(B=0, lengths=[300, 1, 0, 128, 129, 5, 700], H=3, init_std=0.05)
    out, fin = run_gpu(x)
    check(x, out, fin, *run_ref(x))
    # the empty sequence hands its initial state through unchanged
    assert torch.equal(fin[2].cpu(), x["init_state"][2])


@pytest.mark.parametrize("chunk", [128, 64])
def test_packed_vector_gate(cuda_ok, chunk):
    x = small(B=0, lengths=[77, 256, 130], H=2, gate="vector", g_div=4.0, chunk=chunk)
    out, fin = run_gpu(x)
    check(x, out, fin, *run_ref(x))


def test_bad_cu_seqlens_reported_by_status_sync(cuda_ok):
    gla = _gla()
    x = small(B=0, lengths=[10, 20, 30], H=2)
    cu = torch.tensor([0, 20, 10, 60], dtype=torch.int32)  # not monotone
    with pytest.raises(gla.GlaError) as e:
        gla.chunk_fwd(cuda(x["q"]), cuda(x["k"]), cuda(x["v"]), cuda(x["g"]),
                      scale=x["scale"], cu_seqlens=cuda(cu), chunk=128)
        gla.status_sync()
    assert e.value.status == 1
    gla.status_sync()  # cleared


def test_empty_dense_batch_copies_initial_state(cuda_ok):
    gla = _gla()
    x = small(B=3, T=0, H=2)
    out, fin = gla.chunk_fwd(cuda(x["q"]), cuda(x["k"]), cuda(x["v"]), cuda(x["g"]),
                             init_state=cuda(x["init_state"]), chunk=128)
    gla.status_sync()
    assert out.numel() == 0
    assert torch.equal(fin.cpu(), x["init_state"])


# ---------------------------------------------------------------------------
# The method's invariants on the GPU path.
# ---------------------------------------------------------------------------
def test_chunk_sizes_agree(cuda_ok):
    x = small(B=2, T=390, H=2)
    outs = [run_gpu(x, chunk=c) for c in (16, 32, 64, 128)]
    for o, f in outs[1:]:
        assert rel_max(to_np(o), to_np(outs[0][0])) <= 2 * out_tol(torch.bfloat16)
        assert rel_max(to_np(f), to_np(outs[0][1])) <= 2 * TOL_STATE


@pytest.mark.parametrize("gate", ["scalar", "vector"])
@pytest.mark.parametrize("chunk", [128, 64])
def test_prefill_equals_decode_steps(cuda_ok, chunk, gate):
    gla = _gla()
    x = small(B=3, T=140, H=2, chunk=chunk, gate=gate, init_std=0.05)
    out, fin = run_gpu(x)
    S = cuda(x["init_state"]).clone()
    for t in range(x["q"].shape[1]):
        o = gla.decode_step(cuda(x["q"][:, t]), cuda(x["k"][:, t]), cuda(x["v"][:, t]),
                            cuda(x["g"][:, t]), S, scale=x["scale"], out_dtype=torch.float32)
        assert rel_max(to_np(o), to_np(out[:, t])) <= 2 * out_tol(torch.bfloat16), t
    assert rel_max(to_np(S), to_np(fin)) <= 2 * TOL_STATE


def test_linear_in_v(cuda_ok):
    """Superposition in V: V1 and V2 have disjoint supports, so V1 + a V2 (a a
    power of two) is exact in bf16 and the outputs and states must add up."""
    x = small(B=2, T=300, H=2, init_std=0.0)
    mask = torch.rand(x["v"].shape, generator=torch.Generator().manual_seed(3)) < 0.5
    v1 = torch.where(mask, x["v"], torch.zeros_like(x["v"]))
    v2 = torch.where(mask, torch.zeros_like(x["v"]), x["v"])
    a = -0.5
    v3 = (v1.float() + a * v2.float()).to(torch.bfloat16)
    assert torch.equal(v3.float(), v1.float() + a * v2.float())
    o1, f1 = run_gpu(dict(x, v=v1))
    o2, f2 = run_gpu(dict(x, v=v2))
    o3, f3 = run_gpu(dict(x, v=v3))
    assert rel_max(to_np(o3), to_np(o1) + a * to_np(o2)) <= 2 * out_tol(torch.bfloat16)
    assert rel_max(to_np(f3), to_np(f1) + a * to_np(f2)) <= 2 * TOL_STATE
    check(dict(x, v=v3), o3, f3, *run_ref(dict(x, v=v3)))


def test_continuation_from_final_state(cuda_ok):
    gla = _gla()
    x = small(B=2, T=400, H=2)
    t1 = 200
    o_full, f_full = run_gpu(x)
    x1 = dict(x, q=x["q"][:, :t1].contiguous(), k=x["k"][:, :t1].contiguous(),
              v=x["v"][:, :t1].contiguous(), g=x["g"][:, :t1].contiguous())
    o1, f1 = run_gpu(x1)
    out2, f2 = gla.chunk_fwd(cuda(x["q"][:, t1:].contiguous()), cuda(x["k"][:, t1:].contiguous()),
                             cuda(x["v"][:, t1:].contiguous()), cuda(x["g"][:, t1:].contiguous()),
                             scale=x["scale"], init_state=f1, chunk=128,
                             out_dtype=torch.float32)
    gla.status_sync()
    o_ref, s_ref = run_ref(x)
    check(x, torch.cat([o1, out2], dim=1), f2, o_ref, s_ref)


# ---------------------------------------------------------------------------
# Full-size workloads, every element against the oracle.
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("name", ["prefill", "vector", "varlen", "laplace"])
def test_full_size_workload(cuda_ok, name):
    """The whole output and final-state tensors of each full-size workload
    against the oracle's token-by-token recurrence (in the launch
    configuration the bench times).  The tolerance applies to the fp32 output
    of the same call; the bf16 output is that result rounded once, and its own
    error is printed beside it for the reader."""
    gla = _gla()
    w = gla_inputs.WORKLOADS[name]
    x = gla_inputs.prefill_inputs(w)
    args = (cuda(x["q"]), cuda(x["k"]), cuda(x["v"]), cuda(x["g"]))
    kw = dict(scale=x["scale"], init_state=cuda(x["init_state"]),
              cu_seqlens=cuda(x["cu_seqlens"]), chunk=x["chunk"])
    out16, fin16 = gla.chunk_fwd(*args, **kw)
    out32, fin = gla.chunk_fwd(*args, out_dtype=torch.float32, **kw)
    gla.status_sync()
    check_bf16_rounding(out16, out32)
    assert torch.equal(fin16, fin)
    o_ref, s_ref = run_ref(x)
    e_o = rel_max(to_np(out32), o_ref)
    e_o16 = rel_max(to_np(out16), o_ref)
    e_s = rel_max(to_np(fin), s_ref)
    print(f"{name}: output (fp32 result) {e_o:.3e}, output (bf16 tensor) {e_o16:.3e}, "
          f"final state {e_s:.3e}")
    assert e_o <= out_tol(torch.bfloat16), f"output error {e_o:.3e}"
    assert e_s <= TOL_STATE, f"state error {e_s:.3e}"
    if name != "vector":
        # the per-head kernel's S', P' and W V enter as bf16 hi + lo: measured
        # 3.0e-5 .. 5.6e-5 (output) and 2.2e-5 .. 3.0e-5 (state); a regression
        # to operands rounded once (2.5e-2 here) fails these
        assert e_o <= 3e-4 and e_s <= 3e-4, (e_o, e_s)
