"""Pins of the oracle's gradient (``oracle.backward``) to things other than
itself (CPU only).

The gradient is tied to central finite differences of the oracle's forward
recurrence (``oracle.recurrent``, a separate code path), to closed forms of
the undecayed case (g = 0, causal linear attention as matrix products) and of
a one-channel constant decay, to the chain rule between the two gate shapes,
and to packing.  The mutation tests plant plausible mistakes in a copy of the
C source's backward and show that the finite-difference pin catches each.
"""
import ctypes
import os
import shutil
import subprocess
import tempfile

import numpy as np
import pytest

import oracle


def rand_problem(rng, B=2, T=70, H=2, dk=3, dv=4, vector=False, g_scale=1.0):
    q = rng.standard_normal((B, T, H, dk))
    k = rng.standard_normal((B, T, H, dk))
    v = rng.standard_normal((B, T, H, dv))
    g = -g_scale * rng.random((B, T, H, dk) if vector else (B, T, H)) - 0.01
    S0 = rng.standard_normal((B, H, dk, dv))
    do = rng.standard_normal((B, T, H, dv))
    dF = rng.standard_normal((B, H, dk, dv))
    return q, k, v, g, S0, do, dF


def loss(q, k, v, g, scale, S0, do, dF, cu=None):
    out, fin = oracle.recurrent(q, k, v, g, scale, init_state=S0, cu_seqlens=cu)
    return float(np.sum(out * do) + np.sum(fin * dF))


def fd_errors(rng, args, grads, scale, do, dF, cu=None, samples=12, eps=1e-5):
    """Largest |central difference - gradient| over random coordinates of each input."""
    errs = []
    for ai, (a, gr) in enumerate(zip(args, grads)):
        worst = 0.0
        for _ in range(samples):
            idx = tuple(int(rng.integers(0, n)) for n in a.shape)
            plus = [x.copy() for x in args]
            minus = [x.copy() for x in args]
            plus[ai][idx] += eps
            minus[ai][idx] -= eps
            fd = (loss(*plus[:4], scale, plus[4], do, dF, cu) -
                  loss(*minus[:4], scale, minus[4], do, dF, cu)) / (2 * eps)
            worst = max(worst, abs(fd - gr[idx]) / max(1.0, abs(fd)))
        errs.append(worst)
    return errs


@pytest.mark.parametrize("vector", [False, True])
def test_gradient_matches_central_differences(vector):
    # T = 70 crosses the oracle's 64-token checkpoint segment
    rng = np.random.default_rng(3 + vector)
    q, k, v, g, S0, do, dF = rand_problem(rng, vector=vector)
    scale = 0.7
    grads = oracle.backward(q, k, v, g, scale, do, init_state=S0, d_final=dF)
    errs = fd_errors(rng, [q, k, v, g, S0], grads, scale, do, dF)
    assert max(errs) < 1e-7, errs


def test_gradient_packed_matches_central_differences():
    rng = np.random.default_rng(11)
    cu = np.array([0, 5, 5, 71, 80], dtype=np.int32)  # one empty sequence
    R, H, dk, dv = int(cu[-1]), 2, 3, 4
    q, k, v, g, S0, do, dF = rand_problem(rng, B=1, T=R, H=H, dk=dk, dv=dv, vector=True)
    S0 = rng.standard_normal((4, H, dk, dv))
    dF = rng.standard_normal((4, H, dk, dv))
    grads = oracle.backward(q, k, v, g, 0.5, do, init_state=S0, d_final=dF, cu_seqlens=cu)
    errs = fd_errors(rng, [q, k, v, g, S0], grads, 0.5, do, dF, cu=cu)
    assert max(errs) < 1e-7, errs
    # the empty sequence passes d_final straight through to d_init
    assert np.array_equal(grads[4][1], dF[1])


def test_zero_gate_closed_form():
    """g = 0: o = scale (tril(Q K^T) V + Q S0), final = S0 + K^T V, so every
    gradient is a product of whole matrices."""
    rng = np.random.default_rng(5)
    q, k, v, g, S0, do, dF = rand_problem(rng, B=1, T=13, H=1, dk=4, dv=5)
    g[:] = 0.0
    scale = 0.45
    dq, dk_, dv_, dg, d0 = oracle.backward(q, k, v, g, scale, do, init_state=S0, d_final=dF)
    Q, K, V, dO = q[0, :, 0], k[0, :, 0], v[0, :, 0], do[0, :, 0]
    S, F = S0[0, 0], dF[0, 0]
    M = np.tril(dO @ V.T)                        # M[t, u] = do_t . v_u for u <= t
    np.testing.assert_allclose(dq[0, :, 0], scale * (M @ K + dO @ S.T), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dk_[0, :, 0], scale * (M.T @ Q) + V @ F.T, rtol=1e-12, atol=1e-12)
    A = np.tril(Q @ K.T)
    np.testing.assert_allclose(dv_[0, :, 0], scale * (A.T @ dO) + K @ F, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(d0[0, 0], scale * Q.T @ dO + F, rtol=1e-12, atol=1e-12)
    # dg_t = <S_{t-1}, Sbar_t> with the states as prefix / suffix sums of outer products
    T = Q.shape[0]
    for t in range(T):
        before = S + K[:t].T @ V[:t]
        after = F + scale * Q[t:].T @ dO[t:]
        assert abs(dg[0, t, 0] - np.sum(before * after)) < 1e-11


def test_constant_decay_closed_form():
    """One channel, q = k = v = 1, g = log(lam) at every token: o_t = sum_{u<=t}
    lam^(t-u), and the summed gate gradient is d/d log(lam) of sum_t o_t."""
    T, lam = 20, 0.8
    ones = np.ones((1, T, 1, 1))
    g = np.full((1, T, 1), np.log(lam))
    _, _, _, dg, _ = oracle.backward(ones, ones, ones, g, 1.0, ones)
    t = np.arange(T)
    # sum_t (1 - lam^(t+1)) / (1 - lam), differentiated in lam, times lam
    f = lambda x: np.sum((1 - x ** (t + 1)) / (1 - x))            # noqa: E731
    df = lambda x: np.sum((-(t + 1) * x ** t * (1 - x) + (1 - x ** (t + 1))) / (1 - x) ** 2)  # noqa
    assert abs(np.sum(dg) - lam * df(lam)) < 1e-10 * abs(lam * df(lam))
    assert f(lam) > 0


def test_head_gate_is_the_channel_sum_of_the_vector_gate():
    """Chain rule: a per-head gate equals a per-channel gate with equal entries,
    so its gradient is the sum of the per-channel gradients."""
    rng = np.random.default_rng(8)
    q, k, v, g, S0, do, dF = rand_problem(rng, T=40)
    gv = np.repeat(g[..., None], q.shape[-1], axis=-1)
    s_grads = oracle.backward(q, k, v, g, 0.3, do, init_state=S0, d_final=dF)
    v_grads = oracle.backward(q, k, v, gv, 0.3, do, init_state=S0, d_final=dF)
    np.testing.assert_allclose(s_grads[3], v_grads[3].sum(-1), rtol=1e-11, atol=1e-11)
    for a, b in zip(s_grads[:3] + s_grads[4:], v_grads[:3] + v_grads[4:]):
        np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-12)


def test_empty_and_missing_gradients():
    rng = np.random.default_rng(2)
    q, k, v, g, S0, do, dF = rand_problem(rng, B=1, T=0)
    dq, dk_, dv_, dg, d0 = oracle.backward(q, k, v, g, 1.0, do, init_state=S0, d_final=dF)
    assert dq.shape == q.shape and np.array_equal(d0, dF)
    q, k, v, g, S0, do, dF = rand_problem(rng, B=1, T=6)
    *_, d0 = oracle.backward(q, k, v, g, 1.0, np.zeros_like(do), init_state=S0)
    assert not d0.any()


# --------------------------------------------------------------------------
# Mutation tests on the backward
# --------------------------------------------------------------------------
BWD_MUTANTS = {
    # the gate gradient without the token's own decay factor
    "dg_missing_decay": ("dg[((size_t)row * H + h) * dk + i] = a * acc;",
                         "dg[((size_t)row * H + h) * dk + i] = acc;"),
    # readout gradient added after the decay (token t's own readout decayed)
    "readout_grad_decayed": ("Sbar[(size_t)i * dv + j] *= a;",
                             "Sbar[(size_t)i * dv + j] *= a * a;"),
    # scale dropped from the readout's contribution to Sbar
    "missing_scale": ("Sbar[(size_t)i * dv + j] += scale * qt[i] * dot[j];",
                      "Sbar[(size_t)i * dv + j] += qt[i] * dot[j];"),
    # dk against the key instead of the value
    "dk_wrong_operand": ("acc += Sbar[(size_t)i * dv + j] * vt[j];",
                         "acc += Sbar[(size_t)i * dv + j] * vt[j % dv] * kt[i];"),
    # dq from the state before the token's own update
    "dq_before_update": ("acc += S[(size_t)i * dv + j] * dot[j];",
                         "acc += (S[(size_t)i * dv + j] - kt[i] * vt[j]) * dot[j];"),
}


def _build_bwd_mutant(name, tmp):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "gla_oracle.c")).read()
    old, new = BWD_MUTANTS[name]
    assert src.count(old) == 1, f"mutation site for {name} not unique"
    src = src.replace(old, new)
    c = os.path.join(tmp, f"{name}.c")
    so = os.path.join(tmp, f"lib{name}.so")
    with open(c, "w") as f:
        f.write(src)
    subprocess.run(["gcc", "-O1", "-fopenmp", "-fPIC", "-shared", "-o", so, c, "-lm"], check=True)
    return so


def _bwd_runner(so):
    lib = ctypes.CDLL(so)
    dp = ctypes.POINTER(ctypes.c_double)
    lib.gla_oracle_backward_f64.argtypes = ([dp] * 4 + [ctypes.c_int, ctypes.c_double] +
                                            [dp] * 8 + [ctypes.c_void_p] + [ctypes.c_int] * 6)
    lib.gla_oracle_backward_f64.restype = ctypes.c_int

    def run(q, k, v, g, scale, do, S0, dF):
        c = lambda a: np.ascontiguousarray(a, dtype=np.float64)  # noqa: E731
        q, k, v, g, do, S0, dF = map(c, (q, k, v, g, do, S0, dF))
        B, T, H, dk = q.shape
        dv = v.shape[-1]
        outs = [np.zeros(q.shape), np.zeros(k.shape), np.zeros(v.shape), np.zeros(g.shape),
                np.zeros(S0.shape)]
        p = lambda a: a.ctypes.data_as(dp)  # noqa: E731
        rc = lib.gla_oracle_backward_f64(p(q), p(k), p(v), p(g), int(g.ndim == 4), scale, p(S0),
                                         p(do), p(dF), *[p(o) for o in outs], None, B, H, T, dk,
                                         dv, 1)
        assert rc == 0
        return outs
    return run


def _fd_pin_passes(backward):
    rng = np.random.default_rng(21)
    q, k, v, g, S0, do, dF = rand_problem(rng, B=1, T=9, H=1, dk=3, dv=2, vector=True)
    grads = backward(q, k, v, g, 0.6, do, S0, dF)
    return max(fd_errors(rng, [q, k, v, g, S0], grads, 0.6, do, dF, samples=20)) < 1e-7


def test_unmutated_backward_passes_the_fd_pin():
    assert _fd_pin_passes(lambda q, k, v, g, s, do, S0, dF: oracle.backward(
        q, k, v, g, s, do, init_state=S0, d_final=dF))


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
@pytest.mark.parametrize("name", sorted(BWD_MUTANTS))
def test_planted_backward_mistake_is_caught(name):
    with tempfile.TemporaryDirectory() as tmp:
        assert not _fd_pin_passes(_bwd_runner(_build_bwd_mutant(name, tmp))), name
