"""Pins of the fp64 oracle to things other than itself (CPU only).

Each check ties the oracle to what the "i14 Laplace 3B on AWS Trainium2" page
and plain mathematics fix: a textbook special case (g = 0 is causal linear
attention, a masked matmul), closed forms of the constant-decay recurrence,
the exact reset under g = -inf, the page's printed decay-schedule values,
the chunked form's re-association, prefill/decode equivalence, linearity in V,
continuation from a saved state, and packing.  The mutation tests at the end
plant plausible mistakes in a copy of the oracle's C source and show that
these pins catch them.
"""
import json
import os
import shutil
import subprocess
import tempfile

import numpy as np
import pytest

import gla_inputs
import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
RTOL = 1e-12


def rand_inputs(rng, B=2, T=9, H=2, dk=5, dv=7, vector=False, init=True, g_scale=0.3):
    q = rng.standard_normal((B, T, H, dk))
    k = rng.standard_normal((B, T, H, dk))
    v = rng.standard_normal((B, T, H, dv))
    gshape = (B, T, H, dk) if vector else (B, T, H)
    g = -g_scale * rng.random(gshape) - 0.01
    S0 = rng.standard_normal((B, H, dk, dv)) if init else None
    return q, k, v, g, S0


def rel(a, b):
    return np.max(np.abs(a - b)) / max(np.sqrt(np.mean(b * b)), 1e-300)


# --------------------------------------------------------------------------
# g = 0: the recurrence is causal (unnormalised) linear attention.
# --------------------------------------------------------------------------
def test_zero_gate_is_masked_matmul():
    rng = np.random.default_rng(1)
    q, k, v, g, S0 = rand_inputs(rng, T=11)
    g[:] = 0.0
    scale = 0.37
    out, fin = oracle.recurrent(q, k, v, g, scale, init_state=S0)
    for b in range(q.shape[0]):
        for h in range(q.shape[2]):
            Q, K, V = q[b, :, h], k[b, :, h], v[b, :, h]
            A = np.tril(Q @ K.T)  # causal mask, diagonal kept
            ref = scale * (A @ V + Q @ S0[b, h])
            assert rel(out[b, :, h], ref) < RTOL
            assert rel(fin[b, h], S0[b, h] + K.T @ V) < RTOL


def test_zero_gate_no_init_state():
    rng = np.random.default_rng(2)
    q, k, v, g, _ = rand_inputs(rng, init=False)
    g[:] = 0.0
    out, fin = oracle.recurrent(q, k, v, g, 1.0)
    for b in range(q.shape[0]):
        for h in range(q.shape[2]):
            Q, K, V = q[b, :, h], k[b, :, h], v[b, :, h]
            assert rel(out[b, :, h], np.tril(Q @ K.T) @ V) < RTOL
            assert rel(fin[b, h], K.T @ V) < RTOL


# --------------------------------------------------------------------------
# Closed forms of a constant decay.
# --------------------------------------------------------------------------
@pytest.mark.parametrize("lam", [0.5, 0.9, 0.99966])
def test_constant_decay_geometric_sum(lam):
    """q = k = e_1, v = 1, g = log(lam): o_t = scale * (1 - lam^(t+1)) / (1 - lam)."""
    T, dk, dv, scale = 40, 4, 3, 0.25
    q = np.zeros((1, T, 1, dk)); q[..., 0] = 1.0
    k = q.copy()
    v = np.ones((1, T, 1, dv))
    g = np.full((1, T, 1), np.log(lam))
    out, fin = oracle.recurrent(q, k, v, g, scale)
    t = np.arange(T)
    expect = scale * (1 - lam ** (t + 1)) / (1 - lam)
    for j in range(dv):
        np.testing.assert_allclose(out[0, :, 0, j], expect, rtol=1e-13)
    np.testing.assert_allclose(fin[0, 0, 0], (1 - lam ** T) / (1 - lam), rtol=1e-13)
    assert np.all(fin[0, 0, 1:] == 0.0)


def test_vector_gate_decays_key_rows():
    """Per-key-channel decays lam_i act on row i of S (the key channel).

    k = 1, v = e_0, g[i] = log(lam_i): S_t[i, 0] = (1 - lam_i^(t+1)) / (1 - lam_i),
    so q = e_i reads that row and q = 1 reads their sum.  Decaying columns
    instead (the transposed reading) gives a different answer.
    """
    T, dk, dv = 25, 4, 3
    lam = np.array([0.5, 0.8, 0.95, 0.999])
    k = np.ones((1, T, 1, dk))
    v = np.zeros((1, T, 1, dv)); v[..., 0] = 1.0
    g = np.broadcast_to(np.log(lam), (1, T, 1, dk)).copy()
    t = np.arange(T)[:, None]
    rows = (1 - lam[None, :] ** (t + 1)) / (1 - lam[None, :])  # [T, dk]
    for i in range(dk):
        q = np.zeros((1, T, 1, dk)); q[..., i] = 1.0
        out, _ = oracle.recurrent(q, k, v, g, 1.0)
        np.testing.assert_allclose(out[0, :, 0, 0], rows[:, i], rtol=1e-13)
        assert np.all(out[0, :, 0, 1:] == 0.0)
    out, fin = oracle.recurrent(np.ones((1, T, 1, dk)), k, v, g, 1.0)
    np.testing.assert_allclose(out[0, :, 0, 0], rows.sum(axis=1), rtol=1e-13)
    np.testing.assert_allclose(fin[0, 0, :, 0], rows[-1], rtol=1e-13)


def test_decay_schedule_printed_values():
    """The page prints lambda_0 = 0.5 and lambda_15 ~= 0.9997 for 16 heads, 1..2048."""
    with open(os.path.join(GOLDEN, "decay_schedule.json")) as f:
        gold = json.load(f)
    lam = oracle.decay_schedule(gold["heads"], gold["t_min"], gold["t_max"])
    assert lam.shape == (16,)
    assert lam[0] == pytest.approx(gold["lambda_0"], abs=1e-15)
    assert round(float(lam[15]), gold["lambda_15_printed_decimals"]) == gold["lambda_15_printed"]
    assert np.all(np.diff(lam) > 0)  # longer memory for later heads


def test_decay_schedule_half_lives_through_recurrence():
    """An impulse written at t=0 under head h's fixed decay halves after its half-life."""
    lam = oracle.decay_schedule(16, 1, 2048)
    half = np.array([2048 ** (h / 15) for h in range(16)])
    for h in (0, 5, 10):
        T = int(np.ceil(half[h])) + 2
        q = np.zeros((1, T, 1, 2)); q[..., 0] = 1
        k = np.zeros((1, T, 1, 2)); k[0, 0, 0, 0] = 1  # only token 0 writes
        v = np.ones((1, T, 1, 1))
        g = np.full((1, T, 1), np.log(lam[h]))
        out, _ = oracle.recurrent(q, k, v, g, 1.0)
        # o_t = lam^t; at t = half-life it is one half (interpolate for fractional)
        assert out[0, 0, 0, 0] == 1.0
        th = half[h]
        lo = int(np.floor(th))
        interp = out[0, lo, 0, 0] * lam[h] ** (th - lo)
        assert interp == pytest.approx(0.5, rel=1e-12)


# --------------------------------------------------------------------------
# g = -inf erases the state exactly.
# --------------------------------------------------------------------------
@pytest.mark.parametrize("vector", [False, True])
def test_minus_inf_resets_state(vector):
    rng = np.random.default_rng(3)
    q, k, v, g, S0 = rand_inputs(rng, B=1, T=12, vector=vector)
    t0 = 5
    g[:, t0] = -np.inf
    out, fin = oracle.recurrent(q, k, v, g, 0.5, init_state=S0)
    out2, fin2 = oracle.recurrent(q[:, t0:], k[:, t0:], v[:, t0:], g[:, t0:], 0.5)
    assert np.array_equal(out[:, t0:], out2)
    assert np.array_equal(fin, fin2)
    # the outputs before the reset do depend on the initial state
    out3, _ = oracle.recurrent(q, k, v, g, 0.5)
    assert not np.allclose(out[:, :t0], out3[:, :t0])


def test_minus_inf_on_one_key_channel_resets_that_row():
    rng = np.random.default_rng(4)
    q, k, v, g, S0 = rand_inputs(rng, B=1, T=8, vector=True)
    t0, i = 3, 2
    g[:, t0, :, i] = -np.inf
    _, fin = oracle.recurrent(q, k, v, g, 1.0, init_state=S0)
    # zero the history of row i before t0: same final row i
    k2 = k.copy(); k2[:, :t0, :, i] = 0.0
    S02 = S0.copy(); S02[:, :, i, :] = 123.0
    _, fin2 = oracle.recurrent(q, k2, v, g, 1.0, init_state=S02)
    np.testing.assert_array_equal(fin[:, :, i], fin2[:, :, i])
    # rows other than i never saw the change
    others = [r for r in range(q.shape[-1]) if r != i]
    np.testing.assert_array_equal(fin2[:, :, others], fin[:, :, others])
    # without the -inf, row i does remember its history
    g3 = g.copy(); g3[:, t0, :, i] = -0.1
    _, a = oracle.recurrent(q, k, v, g3, 1.0, init_state=S0)
    _, b = oracle.recurrent(q, k2, v, g3, 1.0, init_state=S02)
    assert not np.allclose(a[:, :, i], b[:, :, i])


# --------------------------------------------------------------------------
# The chunked form, the unrolled sum and the recurrence agree.
# --------------------------------------------------------------------------
@pytest.mark.parametrize("vector", [False, True])
def test_bruteforce_equals_recurrent(vector):
    rng = np.random.default_rng(5)
    q, k, v, g, S0 = rand_inputs(rng, T=10, vector=vector)
    a = oracle.recurrent(q, k, v, g, 0.3, init_state=S0)
    b = oracle.bruteforce(q, k, v, g, 0.3, init_state=S0)
    assert rel(a[0], b[0]) < 1e-12 and rel(a[1], b[1]) < 1e-12


@pytest.mark.parametrize("vector", [False, True])
def test_chunked_equals_recurrent_every_chunk_size(vector):
    rng = np.random.default_rng(6)
    T = 13
    q, k, v, g, S0 = rand_inputs(rng, T=T, vector=vector)
    ref_o, ref_s = oracle.recurrent(q, k, v, g, 0.7, init_state=S0)
    for chunk in range(1, T + 3):
        o, s = oracle.chunked(q, k, v, g, 0.7, chunk, init_state=S0)
        assert rel(o, ref_o) < 1e-12, chunk
        assert rel(s, ref_s) < 1e-12, chunk


def test_chunked_with_minus_inf_inside_a_chunk():
    rng = np.random.default_rng(7)
    q, k, v, g, S0 = rand_inputs(rng, T=16, vector=True)
    g[:, 6, :, 1] = -np.inf
    g[:, 9] = -np.inf
    ref = oracle.recurrent(q, k, v, g, 1.0, init_state=S0)
    got = oracle.chunked(q, k, v, g, 1.0, 8, init_state=S0)
    assert np.all(np.isfinite(got[0])) and np.all(np.isfinite(got[1]))
    assert rel(got[0], ref[0]) < 1e-12 and rel(got[1], ref[1]) < 1e-12


def test_chunked_packed_sequences():
    rng = np.random.default_rng(8)
    lens = [5, 1, 12, 0, 7]
    R = sum(lens)
    H, dk, dv = 2, 4, 3
    q = rng.standard_normal((1, R, H, dk)); k = rng.standard_normal((1, R, H, dk))
    v = rng.standard_normal((1, R, H, dv)); g = -0.2 * rng.random((1, R, H))
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    S0 = rng.standard_normal((len(lens), H, dk, dv))
    ref = oracle.recurrent(q, k, v, g, 1.0, init_state=S0, cu_seqlens=cu)
    for chunk in (1, 2, 4, 5, 64):
        got = oracle.chunked(q, k, v, g, 1.0, chunk, init_state=S0, cu_seqlens=cu)
        assert rel(got[0], ref[0]) < 1e-12 and rel(got[1], ref[1]) < 1e-12


# --------------------------------------------------------------------------
# Serving-form identities.
# --------------------------------------------------------------------------
@pytest.mark.parametrize("vector", [False, True])
def test_prefill_equals_decode_steps(vector):
    rng = np.random.default_rng(9)
    q, k, v, g, S0 = rand_inputs(rng, B=3, T=7, vector=vector)
    out, fin = oracle.recurrent(q, k, v, g, 0.5, init_state=S0)
    S = S0.copy()
    for t in range(q.shape[1]):
        o, S = oracle.decode_step(q[:, t], k[:, t], v[:, t], g[:, t], 0.5, S)
        assert rel(o, out[:, t]) < 1e-13
    assert rel(S, fin) < 1e-13


def test_decode_step_does_not_modify_input_state():
    rng = np.random.default_rng(10)
    S = rng.standard_normal((2, 2, 3, 4)); S_copy = S.copy()
    oracle.decode_step(rng.standard_normal((2, 2, 3)), rng.standard_normal((2, 2, 3)),
                       rng.standard_normal((2, 2, 4)), -rng.random((2, 2)), 1.0, S)
    assert np.array_equal(S, S_copy)


def test_continuation_from_saved_state():
    rng = np.random.default_rng(11)
    q, k, v, g, S0 = rand_inputs(rng, T=14, vector=True)
    t1 = 6
    full_o, full_s = oracle.recurrent(q, k, v, g, 0.9, init_state=S0)
    o1, s1 = oracle.recurrent(q[:, :t1], k[:, :t1], v[:, :t1], g[:, :t1], 0.9, init_state=S0)
    o2, s2 = oracle.chunked(q[:, t1:], k[:, t1:], v[:, t1:], g[:, t1:], 0.9, 3, init_state=s1)
    assert rel(np.concatenate([o1, o2], axis=1), full_o) < 1e-12
    assert rel(s2, full_s) < 1e-12


def test_linear_in_v_and_initial_state():
    rng = np.random.default_rng(12)
    q, k, v1, g, S1 = rand_inputs(rng, T=9)
    v2 = rng.standard_normal(v1.shape)
    S2 = rng.standard_normal(S1.shape)
    a = -1.75
    o1, f1 = oracle.recurrent(q, k, v1, g, 1.0, init_state=S1)
    o2, f2 = oracle.recurrent(q, k, v2, g, 1.0, init_state=S2)
    o3, f3 = oracle.recurrent(q, k, v1 + a * v2, g, 1.0, init_state=S1 + a * S2)
    assert rel(o3, o1 + a * o2) < 1e-12 and rel(f3, f1 + a * f2) < 1e-12
    # ... and with zero initial state, linear in V alone
    o4, _ = oracle.recurrent(q, k, v1, g, 1.0)
    o5, _ = oracle.recurrent(q, k, v2, g, 1.0)
    o6, _ = oracle.recurrent(q, k, v1 + a * v2, g, 1.0)
    assert rel(o6, o4 + a * o5) < 1e-12


def test_packing_equals_independent_runs():
    rng = np.random.default_rng(13)
    lens = [3, 8, 1, 6]
    H, dk, dv = 3, 4, 5
    seqs = [rand_inputs(rng, B=1, T=n, H=H, dk=dk, dv=dv, vector=True) for n in lens]
    q = np.concatenate([s[0] for s in seqs], axis=1)
    k = np.concatenate([s[1] for s in seqs], axis=1)
    v = np.concatenate([s[2] for s in seqs], axis=1)
    g = np.concatenate([s[3] for s in seqs], axis=1)
    S0 = np.concatenate([s[4] for s in seqs], axis=0)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    out, fin = oracle.recurrent(q, k, v, g, 0.4, init_state=S0, cu_seqlens=cu)
    for i, s in enumerate(seqs):
        o, f = oracle.recurrent(*s[:4], 0.4, init_state=s[4])
        assert np.array_equal(out[:, cu[i]:cu[i + 1]], o)
        assert np.array_equal(fin[i], f[0])


def test_empty_sequence_keeps_initial_state():
    rng = np.random.default_rng(14)
    H, dk, dv = 2, 3, 4
    q = np.zeros((1, 0, H, dk)); k = q.copy(); v = np.zeros((1, 0, H, dv))
    g = np.zeros((1, 0, H))
    S0 = rng.standard_normal((1, H, dk, dv))
    out, fin = oracle.recurrent(q, k, v, g, 1.0, init_state=S0)
    assert out.size == 0 and np.array_equal(fin, S0)
    out, fin = oracle.chunked(q, k, v, g, 1.0, 4, init_state=S0)
    assert out.size == 0 and np.array_equal(fin, S0)


def test_rejects_bad_cu_seqlens():
    q = np.zeros((1, 4, 1, 2)); v = np.zeros((1, 4, 1, 2)); g = np.zeros((1, 4, 1))
    with pytest.raises(ValueError):
        oracle.recurrent(q, q, v, g, 1.0, cu_seqlens=np.array([0, 3, 2, 4], np.int32))


# --------------------------------------------------------------------------
# Mutation tests: a copy of the oracle with a planted mistake fails the pins.
# --------------------------------------------------------------------------
MUTANTS = {
    # readout before the update (token t would not see its own key/value)
    "readout_before_update": (
        "            /* S <- diag(exp g_t) S + k_t^T v_t */",
        "            for (int j = 0; j < dv; ++j) { double acc = 0.0;\n"
        "                for (int i = 0; i < dk; ++i) acc += qt[i] * S[(size_t)i * dv + j];\n"
        "                ot[j] = scale * acc; }\n"
        "            if (0)"),
    # decay applied to value columns instead of key rows
    "gate_on_columns": (
        "decay_factor(g, vector_gate, row, H, h, dk, i);\n                for (int j = 0; j < dv; ++j)\n"
        "                    S[(size_t)i * dv + j] = a * S",
        "decay_factor(g, vector_gate, row, H, h, dk, i); (void)a;\n                for (int j = 0; j < dv; ++j)\n"
        "                    S[(size_t)i * dv + j] = decay_factor(g, vector_gate, row, H, h, dk, j % dk) * S"),
    # sign error on the log-decay
    "decay_sign": ("return exp(g[(size_t)row * H + h]);", "return exp(-g[(size_t)row * H + h]);"),
    # scale applied twice
    "double_scale": ("ot[j] = scale * acc;\n            }\n        }\n        if (final_state)",
                     "ot[j] = scale * scale * acc;\n            }\n        }\n        if (final_state)"),
    # outer product transposed (k_j for index j)
    "outer_transposed": ("+ kt[i] * vt[j];\n            }\n            /* o_t",
                         "+ kt[j % dk] * vt[i % dv];\n            }\n            /* o_t"),
}


def _build_mutant(name, tmp):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "gla_oracle.c")).read()
    old, new = MUTANTS[name]
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    src = src.replace(old, new, 1)
    c = os.path.join(tmp, f"{name}.c")
    so = os.path.join(tmp, f"lib{name}.so")
    with open(c, "w") as f:
        f.write(src)
    subprocess.run(["gcc", "-O1", "-fopenmp", "-fPIC", "-shared", "-o", so, c, "-lm"], check=True)
    return so


def _pins_pass(run):
    """A compact selection of the pins above, run against ``run(q,k,v,g,scale,S0)``."""
    rng = np.random.default_rng(99)
    ok = True
    # g = 0 masked matmul
    q, k, v, g, S0 = rand_inputs(rng, B=1, T=6, dk=4, dv=4)
    g0 = np.zeros_like(g)
    o, _ = run(q, k, v, g0, 0.5, S0)
    Q, K, V = q[0, :, 0], k[0, :, 0], v[0, :, 0]
    ok &= rel(o[0, :, 0], 0.5 * (np.tril(Q @ K.T) @ V + Q @ S0[0, 0])) < 1e-12
    # constant-decay closed form
    T = 10
    qq = np.zeros((1, T, 1, 4)); qq[..., 0] = 1
    o, _ = run(qq, qq.copy(), np.ones((1, T, 1, 4)), np.full((1, T, 1), np.log(0.5)), 1.0, None)
    ok &= np.allclose(o[0, :, 0, 0], (1 - 0.5 ** (np.arange(T) + 1)) / 0.5, rtol=1e-13)
    # vector gate on key rows
    lam = np.array([0.5, 0.8, 0.95, 0.999])
    kk = np.ones((1, T, 1, 4)); vv = np.zeros((1, T, 1, 4)); vv[..., 0] = 1
    gg = np.broadcast_to(np.log(lam), (1, T, 1, 4)).copy()
    o, _ = run(np.ones((1, T, 1, 4)), kk, vv, gg, 1.0, None)
    rows = (1 - lam[None] ** (np.arange(T)[:, None] + 1)) / (1 - lam[None])
    ok &= np.allclose(o[0, :, 0, 0], rows.sum(1), rtol=1e-13)
    return bool(ok)


def _ctypes_runner(so):
    import ctypes
    lib = ctypes.CDLL(so)
    dp = ctypes.POINTER(ctypes.c_double)
    lib.gla_oracle_recurrent_f64.argtypes = [dp, dp, dp, dp, ctypes.c_int, ctypes.c_double,
                                             dp, dp, dp, ctypes.c_void_p] + [ctypes.c_int] * 6
    lib.gla_oracle_recurrent_f64.restype = ctypes.c_int

    def run(q, k, v, g, scale, S0):
        q, k, v, g = (np.ascontiguousarray(x, dtype=np.float64) for x in (q, k, v, g))
        B, T, H, dk = q.shape
        dv = v.shape[-1]
        out = np.zeros(v.shape)
        fin = np.zeros((B, H, dk, dv))
        S = None if S0 is None else np.ascontiguousarray(S0, dtype=np.float64)
        p = lambda a: None if a is None else a.ctypes.data_as(dp)  # noqa: E731
        rc = lib.gla_oracle_recurrent_f64(p(q), p(k), p(v), p(g), int(g.ndim == 4), scale,
                                          p(S), p(out), p(fin), None, B, H, T, dk, dv, 1)
        assert rc == 0
        return out, fin
    return run


def test_unmutated_oracle_passes_compact_pins():
    assert _pins_pass(lambda q, k, v, g, s, S0: oracle.recurrent(q, k, v, g, s, init_state=S0))


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name):
    with tempfile.TemporaryDirectory() as tmp:
        run = _ctypes_runner(_build_mutant(name, tmp))
        assert not _pins_pass(run), f"mutant {name} slipped through the pins"


def test_laplace_workload_gate_is_the_decay_schedule():
    """The laplace input recipe writes g = log(lambda_h) for every token; its
    per-head values agree with the oracle's decay schedule (itself pinned to
    the page's printed lambda_0 and lambda_15), an independent restatement."""
    x = gla_inputs.prefill_inputs(gla_inputs.WORKLOADS["laplace"], B=1, T=3)
    lam = oracle.decay_schedule(16, 1.0, 2048.0)
    g = x["g"].double().numpy()
    assert g.shape == (1, 3, 16)
    np.testing.assert_allclose(np.exp(g[0]), np.broadcast_to(lam, (3, 16)), rtol=1e-6)


# ---------------------------------------------------------------------------
# The mixer epilogue (self-augmentation, head RMSNorm, SiLU gate).
# ---------------------------------------------------------------------------
def _epi_inputs(seed=0, n=5, H=3, dk=8, dv=6):
    r = np.random.default_rng(seed)
    return (r.normal(size=(n, H, dv)), r.normal(size=(n, H, dk)), r.normal(size=(n, H, dk)),
            r.normal(size=(n, H, dv)))


def test_epilogue_augmentation_at_zero_balance_adds_half_the_value():
    """The page: at initialisation (aug = 0) the augmentation is a
    half-strength skip of the value."""
    o, q, k, v = _epi_inputs()
    got = oracle.mixer_epilogue(o, q, k, v, aug=np.zeros((3, 8)))
    np.testing.assert_allclose(got, o + 0.5 * v, rtol=0, atol=1e-15)


def test_epilogue_augmentation_gate_limits():
    """A large positive (negative) q . (aug * k) passes all (none) of v; the
    gate is the logistic function of that one number per token and head."""
    o, q, k, v = _epi_inputs(1)
    big = 1e3 * np.ones((3, 8))
    s = np.sum(q * big * k, axis=-1, keepdims=True)
    got = oracle.mixer_epilogue(o, q, k, v, aug=big)
    np.testing.assert_allclose(got, o + np.where(s > 0, v, 0.0), atol=1e-12)
    a = np.linspace(-1, 1, 8)[None, :].repeat(3, 0)
    t = np.einsum("nhd,hd,nhd->nh", q, a, k)[..., None]
    np.testing.assert_allclose(oracle.mixer_epilogue(o, q, k, v, aug=a) - o,
                               v * (1 / (1 + np.exp(-t))), rtol=1e-13)


def test_epilogue_rmsnorm_gives_unit_rms_and_ignores_the_row_scale():
    o, q, k, v = _epi_inputs(2)
    w = np.ones((3, 6))
    y = oracle.mixer_epilogue(o, q, k, v, norm_w=w, eps=0.0)
    np.testing.assert_allclose(np.sqrt(np.mean(y * y, axis=-1)), 1.0, rtol=1e-13)
    y2 = oracle.mixer_epilogue(o * np.array([3.0, 0.25, 7.0])[None, :, None], q, k, v,
                               norm_w=w, eps=0.0)
    np.testing.assert_allclose(y2, y, rtol=1e-12)
    # the weight multiplies channel by channel, after the normalisation
    wv = np.arange(1, 7)[None, :].repeat(3, 0) * 1.0
    np.testing.assert_allclose(oracle.mixer_epilogue(o, q, k, v, norm_w=wv, eps=0.0), y * wv,
                               rtol=1e-13)
    # eps bounds the gain of a zero row
    assert np.all(oracle.mixer_epilogue(np.zeros_like(o), q, k, v, norm_w=w, eps=1e-6) == 0)


def test_epilogue_silu_gate():
    o, q, k, v = _epi_inputs(3)
    zero = oracle.mixer_epilogue(o, q, k, v, z=np.zeros_like(o))
    assert np.all(zero == 0)
    big = oracle.mixer_epilogue(o, q, k, v, z=np.full_like(o, 40.0))
    np.testing.assert_allclose(big, 40.0 * o, rtol=1e-15)
    # silu(-x) = silu(x) - x
    zz = np.random.default_rng(4).normal(size=o.shape)
    np.testing.assert_allclose(oracle.mixer_epilogue(o, q, k, v, z=-zz),
                               oracle.mixer_epilogue(o, q, k, v, z=zz) - zz * o, atol=1e-13)


def test_epilogue_order_augment_then_normalise_then_gate():
    o, q, k, v = _epi_inputs(5)
    a, w, zz = np.zeros((3, 8)), np.ones((3, 6)), np.full_like(o, 40.0)
    y = oracle.mixer_epilogue(o, q, k, v, aug=a, norm_w=w, eps=0.0, z=zz)
    x = o + 0.5 * v
    ref = 40.0 * x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True))
    np.testing.assert_allclose(y, ref, rtol=1e-13)
