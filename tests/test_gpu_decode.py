"""GPU decode step (gla_decode_step) against the fp64 oracle."""
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


def _inputs(N, H, dk, dv, io, gate, steps, seed=7):
    w = gla_inputs.WORKLOADS["decode"]
    return gla_inputs.decode_inputs(w, seed=seed, N=N, H=H, dk=dk, dv=dv, io=io, gate=gate,
                                    steps=steps)


@pytest.mark.parametrize("io", ["bf16", "fp32"])
@pytest.mark.parametrize("gate", ["scalar", "vector"])
@pytest.mark.parametrize("dk,dv", [(128, 128), (64, 64), (64, 128), (128, 64), (96, 192), (128, 192)])
def test_decode_steps_match_oracle(cuda_ok, io, gate, dk, dv):
    gla = _gla()
    x = _inputs(37, 3, dk, dv, io, gate, steps=3)
    S_ref = to_np(x["state"])
    S = cuda(x["state"]).clone()
    for t in range(3):
        args = (cuda(x["q"][t]), cuda(x["k"][t]), cuda(x["v"][t]), cuda(x["g"][t]))
        if io == "bf16":
            # same step twice from the same state: bf16 output, then fp32 output
            S2 = S.clone()
            out16 = gla.decode_step(*args, S2, scale=x["scale"])
            out = gla.decode_step(*args, S, scale=x["scale"], out_dtype=torch.float32)
            torch.cuda.synchronize()
            check_bf16_rounding(out16, out)
            assert torch.equal(S, S2)
        else:
            out = gla.decode_step(*args, S, scale=x["scale"])
        o_ref, S_ref = oracle.decode_step(x["q"][t], x["k"][t], x["v"][t], x["g"][t],
                                          x["scale"], S_ref)
        torch.cuda.synchronize()
        assert rel_max(to_np(out), o_ref) <= out_tol(x["q"].dtype), t
        tol_s = TOL_STATE if io == "bf16" else 1e-5
        assert rel_max(to_np(S), S_ref) <= tol_s, t


def test_decode_minus_inf_gate_resets_state(cuda_ok):
    gla = _gla()
    x = _inputs(5, 2, 128, 128, "fp32", "scalar", steps=1)
    g = torch.full_like(x["g"][0], float("-inf"))
    S = cuda(x["state"]).clone()
    out = gla.decode_step(cuda(x["q"][0]), cuda(x["k"][0]), cuda(x["v"][0]), cuda(g), S,
                          scale=1.0)
    kv = torch.einsum("nhi,nhj->nhij", x["k"][0].double(), x["v"][0].double())
    # 0 * S + k v^T is exact in fp32 when k_i v_j is (products of fp32 rounded once)
    assert rel_max(to_np(S), kv.numpy()) < 1e-6
    o_ref = torch.einsum("nhi,nhij->nhj", x["q"][0].double(), kv)
    assert rel_max(to_np(out), o_ref.numpy()) < 1e-5


def test_decode_in_place_on_a_view_of_a_state_pool(cuda_ok):
    """The state argument may be a contiguous slice of a larger pool (one page
    per sequence); pages outside it are untouched."""
    gla = _gla()
    x = _inputs(6, 2, 64, 64, "bf16", "scalar", steps=1)
    pool = torch.randn(10, 2, 64, 64, device="cuda")
    before = pool.clone()
    pool[2:8] = cuda(x["state"])
    gla.decode_step(cuda(x["q"][0]), cuda(x["k"][0]), cuda(x["v"][0]), cuda(x["g"][0]),
                    pool[2:8], scale=x["scale"])
    _, S_ref = oracle.decode_step(x["q"][0], x["k"][0], x["v"][0], x["g"][0], x["scale"],
                                  x["state"])
    torch.cuda.synchronize()
    assert torch.equal(pool[:2], before[:2]) and torch.equal(pool[8:], before[8:])
    assert rel_max(to_np(pool[2:8]), S_ref) <= TOL_STATE


def test_decode_full_size(cuda_ok):
    """N=1280, H=16, dk=dv=128, two consecutive steps: every output and every
    state page against the oracle."""
    gla = _gla()
    w = gla_inputs.WORKLOADS["decode"]
    x = gla_inputs.decode_inputs(w, steps=2)
    S = cuda(x["state"]).clone()
    outs, outs16 = [], []
    for t in range(2):
        args = (cuda(x["q"][t]), cuda(x["k"][t]), cuda(x["v"][t]), cuda(x["g"][t]))
        S16 = S.clone()
        outs16.append(gla.decode_step(*args, S16, scale=x["scale"]))
        outs.append(gla.decode_step(*args, S, scale=x["scale"], out_dtype=torch.float32))
        torch.cuda.synchronize()
        assert torch.equal(S16, S)
        check_bf16_rounding(outs16[t], outs[t])
    S_ref = to_np(x["state"])
    for t in range(2):
        o_ref, S_ref = oracle.decode_step(x["q"][t], x["k"][t], x["v"][t], x["g"][t],
                                          x["scale"], S_ref)
        e = rel_max(to_np(outs[t]), o_ref)
        e16 = rel_max(to_np(outs16[t]), o_ref)
        print(f"decode step {t}: output (fp32 result) {e:.3e}, output (bf16 tensor) {e16:.3e}")
        assert e <= out_tol(torch.bfloat16)
    e_s = rel_max(to_np(S), S_ref)
    print(f"decode state after 2 steps: {e_s:.3e}")
    assert e_s <= TOL_STATE


# ---------------------------------------------------------------------------
# Slot-indexed state pages and CUDA-graph decode buckets.
# ---------------------------------------------------------------------------
def test_decode_slots_match_dense_pages(cuda_ok):
    """Rows on pool pages slots[n] give the same outputs and states as the
    dense call on the gathered pages; pages no row names are untouched; a
    padding row (-1) neither writes its output nor touches any page."""
    gla = _gla()
    w = gla_inputs.WORKLOADS["decode"]
    d = gla_inputs.decode_inputs(w, steps=1, N=6, H=3)
    pool = torch.randn(10, 3, w.dk, w.dv, generator=torch.Generator().manual_seed(4)) * 0.1
    slots = torch.tensor([7, 2, -1, 9, 0, 4], dtype=torch.int32)
    live = slots >= 0
    pool_gpu = cuda(pool).contiguous()
    out = torch.full((6, 3, w.dv), 7.0, dtype=torch.float32, device="cuda")
    gla.decode_step(cuda(d["q"][0]), cuda(d["k"][0]), cuda(d["v"][0]), cuda(d["g"][0]),
                    pool_gpu, scale=d["scale"], out=out, slots=cuda(slots))
    gla.status_sync()
    dense = cuda(pool[slots[live].long()]).contiguous()
    ref = gla.decode_step(cuda(d["q"][0][live]), cuda(d["k"][0][live]), cuda(d["v"][0][live]),
                          cuda(d["g"][0][live]), dense, scale=d["scale"],
                          out_dtype=torch.float32)
    gla.status_sync()
    assert torch.equal(out[live], ref)
    assert (out[~live] == 7.0).all()
    assert torch.equal(pool_gpu[slots[live].long()], dense)
    untouched = [i for i in range(10) if i not in set(slots.tolist())]
    assert torch.equal(pool_gpu[untouched].cpu(), pool[untouched])


def test_decode_slot_out_of_range_is_reported(cuda_ok):
    gla = _gla()
    w = gla_inputs.WORKLOADS["decode"]
    d = gla_inputs.decode_inputs(w, steps=1, N=2, H=2)
    pool = torch.zeros(4, 2, w.dk, w.dv, device="cuda")
    with pytest.raises(gla.GlaError) as e:
        gla.decode_step(cuda(d["q"][0]), cuda(d["k"][0]), cuda(d["v"][0]), cuda(d["g"][0]),
                        pool, slots=cuda(torch.tensor([1, 4], dtype=torch.int32)))
        gla.status_sync()
    assert e.value.status == 1
    gla.status_sync()  # cleared


def test_decode_graph_buckets_replay_the_eager_step(cuda_ok):
    """Steps of varying width through the captured buckets equal the eager
    slot-indexed step on a copy of the pool, step after step."""
    gla = _gla()
    from gated_linear_attention_gla_gb300.serving import DecodeGraphs
    w = gla_inputs.WORKLOADS["decode"]
    H, S = 2, 12
    pool = (torch.randn(S, H, w.dk, w.dv, generator=torch.Generator().manual_seed(8)) * 0.1).cuda()
    pool_ref = pool.clone()
    graphs = DecodeGraphs(pool, max_width=8, out_dtype=torch.float32)
    assert graphs.buckets == [1, 2, 4, 8]
    rng = torch.Generator().manual_seed(21)
    for step, n in enumerate([3, 8, 1, 5, 5, 2]):
        d = gla_inputs.decode_inputs(w, steps=1, N=n, H=H, seed=100 + step)
        slots = torch.randperm(S, generator=rng)[:n].to(torch.int32)
        args = [cuda(d[x][0]) for x in ("q", "k", "v", "g")]
        if step % 2:
            got = graphs.step(*args, cuda(slots)).clone()
        else:
            buf = graphs.buffers(n)
            for name, t in zip(("q", "k", "v", "g", "slots"), (*args, cuda(slots))):
                buf[name].copy_(t)
            got = graphs.run(n).clone()
        ref = gla.decode_step(*args, pool_ref, scale=w.dk ** -0.5, slots=cuda(slots),
                              out_dtype=torch.float32)
        gla.status_sync()
        assert torch.equal(got, ref), step
        assert torch.equal(pool, pool_ref), step
