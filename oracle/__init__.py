"""fp64 CPU oracle for gated linear attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It shares no code with the CUDA library
in ``gated_linear_attention_gla_gb300`` and never imports it.

Source of the method: the "i14 Laplace 3B on AWS Trainium2" blog page,
section "i14 and the Laplace 3B architecture" (paragraphs "GLA mixer" and
"Decay schedule"), and section "Challenge 1: Using native PyTorch on Trainium
for GLA" (the chunked form, Figure 3).  The page's equations were images and
did not survive; the definitions below follow its prose:

* state update  ``S_t = diag(exp g_t) S_{t-1} + k_t^T v_t``  -- the state
  shrinks by the decay and gains the token's key/value pair as a rank-one term;
* readout       ``o_t = scale * q_t S_t`` -- the query reads the state after
  the update (so token t sees its own key/value);
* chunked form  -- inside each chunk a causal attention with decay weights,
  plus what the carried-in state contributes; then the state advances once
  with the chunk's total decay; chunks are independent except for that
  state hand-off.

``g`` is a log-decay: shape ``[..., H]`` (one per token and head: the page's
Simple GLA) or ``[..., H, dk]`` (one per key channel: row i of S decays by
``exp(g[i])``).

Functions
---------
recurrent     token-by-token recurrence in C (the definition; OpenMP over
              (sequence, head))
chunked       the chunked form in C, any chunk size
decode_step   one recurrent step over N independent states, in C
backward      the gradient of the recurrence (reverse mode, token by token), in C
bruteforce    the unrolled recurrence as one O(T^2) sum per token, numpy, tiny
              inputs only
decay_schedule  the page's fixed geometric per-head decay (paragraph "Decay
              schedule's reach")
mixer_epilogue  what follows the readout in the page's mixer (paragraph "GLA
              mixer", after the readout): self-augmentation, head RMSNorm,
              SiLU output gate; numpy, fp64

Every pin of these functions lives in ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gla_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libgla_oracle.so")
_lock = threading.Lock()
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)
_ip = ctypes.POINTER(ctypes.c_int32)


def build(force: bool = False) -> str:
    """Compile ``gla_oracle.c`` into ``libgla_oracle.so`` next to it (gcc, OpenMP).

    No fast-math and no floating-point contraction, so x86 and Arm hosts
    round alike.
    """
    if force or not os.path.exists(_LIB_PATH) or (
        os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
    ):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = [
            "gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fPIC",
            "-shared", "-o", tmp, _SRC, "-lm",
        ]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            common = [_dp, _dp, _dp, _dp, ctypes.c_int, ctypes.c_double, _dp, _dp, _dp, _ip,
                      ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int]
            lib.gla_oracle_recurrent_f64.argtypes = common + [ctypes.c_int]
            lib.gla_oracle_recurrent_f64.restype = ctypes.c_int
            lib.gla_oracle_chunked_f64.argtypes = common + [ctypes.c_int, ctypes.c_int]
            lib.gla_oracle_chunked_f64.restype = ctypes.c_int
            lib.gla_oracle_decode_step_f64.argtypes = [
                _dp, _dp, _dp, _dp, ctypes.c_int, ctypes.c_double, _dp, _dp,
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int]
            lib.gla_oracle_decode_step_f64.restype = ctypes.c_int
            lib.gla_oracle_backward_f64.argtypes = [
                _dp, _dp, _dp, _dp, ctypes.c_int, ctypes.c_double, _dp, _dp, _dp, _dp, _dp,
                _dp, _dp, _dp, _ip, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_int, ctypes.c_int]
            lib.gla_oracle_backward_f64.restype = ctypes.c_int
            lib.gla_oracle_max_threads.argtypes = []
            lib.gla_oracle_max_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def max_threads() -> int:
    """Threads the oracle's OpenMP loops use by default on this host."""
    return int(_load().gla_oracle_max_threads())


def _f64(x):
    """Exact widening of a float/bfloat16 array (numpy or torch CPU) to fp64."""
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor: bf16 has no numpy dtype
        x = x.detach().cpu().double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(_dp)


def _shapes(q, v, g, cu_seqlens):
    """Return (B, T, H, dk, dv, rows, vector_gate) for dense or packed inputs."""
    H, dk = q.shape[-2], q.shape[-1]
    dv = v.shape[-1]
    rows = int(np.prod(q.shape[:-2]))
    if cu_seqlens is not None:
        B, T = len(cu_seqlens) - 1, 0
        if int(cu_seqlens[-1]) != rows:
            raise ValueError("cu_seqlens[-1] must equal the number of token rows")
    else:
        if q.ndim != 4:
            raise ValueError("dense inputs are [B, T, H, d]")
        B, T = q.shape[0], q.shape[1]
    if g.shape == q.shape[:-1]:
        vector_gate = 0
    elif g.shape == q.shape:
        vector_gate = 1
    else:
        raise ValueError(f"g shape {g.shape} matches neither [..., H] nor [..., H, dk]")
    return B, T, H, dk, dv, rows, vector_gate


def _run(kind, q, k, v, g, scale, init_state, cu_seqlens, chunk, nthreads):
    q, k, v, g = _f64(q), _f64(k), _f64(v), _f64(g)
    init = _f64(init_state)
    cu = None
    if cu_seqlens is not None:
        cu = np.ascontiguousarray(np.asarray(
            cu_seqlens.cpu().numpy() if hasattr(cu_seqlens, "cpu") else cu_seqlens,
            dtype=np.int32))
    B, T, H, dk, dv, rows, vg = _shapes(q, v, g, cu)
    out = np.zeros(v.shape, dtype=np.float64)
    final = np.zeros((B, H, dk, dv), dtype=np.float64)
    if init is not None and init.shape != final.shape:
        raise ValueError(f"init_state must be {final.shape}")
    cu_p = None if cu is None else cu.ctypes.data_as(_ip)
    lib = _load()
    args = [_ptr(q), _ptr(k), _ptr(v), _ptr(g), vg, float(scale), _ptr(init), _ptr(out),
            _ptr(final), cu_p, B, H, T, dk, dv]
    if kind == "recurrent":
        rc = lib.gla_oracle_recurrent_f64(*args, int(nthreads))
    else:
        rc = lib.gla_oracle_chunked_f64(*args, int(chunk), int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle {kind} rejected its arguments")
    return out, final


def recurrent(q, k, v, g, scale, init_state=None, cu_seqlens=None, nthreads=0):
    """Token-by-token recurrence.  Returns ``(out, final_state)`` in fp64.

    Dense inputs are ``[B, T, H, d]``; packed inputs are ``[1, R, H, d]`` (or
    ``[R, H, d]``) with ``cu_seqlens`` of length B+1.  ``init_state`` is
    ``[B, H, dk, dv]`` or None (zero).
    """
    return _run("recurrent", q, k, v, g, scale, init_state, cu_seqlens, 0, nthreads)


def chunked(q, k, v, g, scale, chunk, init_state=None, cu_seqlens=None, nthreads=0):
    """The chunked form with chunk size ``chunk``.  Returns ``(out, final_state)``."""
    return _run("chunked", q, k, v, g, scale, init_state, cu_seqlens, chunk, nthreads)


def decode_step(q, k, v, g, scale, state, nthreads=0):
    """One recurrent step over N sequences.

    ``q, k [N, H, dk]``, ``v [N, H, dv]``, ``g [N, H]`` or ``[N, H, dk]``,
    ``state [N, H, dk, dv]``.  Returns ``(out, new_state)``; the input state is
    not modified.
    """
    q, k, v, g = _f64(q), _f64(k), _f64(v), _f64(g)
    S = _f64(state).copy()
    N, H, dk = q.shape
    dv = v.shape[-1]
    if g.shape == (N, H):
        vg = 0
    elif g.shape == (N, H, dk):
        vg = 1
    else:
        raise ValueError("g must be [N, H] or [N, H, dk]")
    out = np.zeros((N, H, dv), dtype=np.float64)
    rc = _load().gla_oracle_decode_step_f64(_ptr(q), _ptr(k), _ptr(v), _ptr(g), vg,
                                             float(scale), _ptr(S), _ptr(out), N, H, dk,
                                             dv, int(nthreads))
    if rc != 0:
        raise ValueError("oracle decode_step rejected its arguments")
    return out, S


def backward(q, k, v, g, scale, d_out, init_state=None, d_final=None, cu_seqlens=None,
             nthreads=0):
    """The gradient of ``recurrent`` by reverse mode, one token at a time (in C).

    For a loss with ``dL/d out = d_out`` and ``dL/d final_state = d_final``
    (zero when None), returns ``(dq, dk, dv, dg, d_init)`` in fp64, shaped like
    q, k, v, g and the state ``[B, H, dk, dv]``.  The reverse sweep carries
    ``Sbar_t = dL/dS_t`` backwards:
    ``Sbar_t = scale q_t^T do_t + diag(exp g_{t+1}) Sbar_{t+1}``, and
    ``dq_t = scale S_t do_t^T``, ``dk_t = Sbar_t v_t^T``, ``dv_t = k_t Sbar_t``,
    ``dg_t[i] = exp(g_t[i]) sum_j S_{t-1}[i, j] Sbar_t[i, j]`` (summed over i
    for the per-head gate), ``d_init = diag(exp g_0) Sbar_0``.
    """
    q, k, v, g, do = _f64(q), _f64(k), _f64(v), _f64(g), _f64(d_out)
    init, dfin = _f64(init_state), _f64(d_final)
    cu = None
    if cu_seqlens is not None:
        cu = np.ascontiguousarray(np.asarray(
            cu_seqlens.cpu().numpy() if hasattr(cu_seqlens, "cpu") else cu_seqlens,
            dtype=np.int32))
    B, T, H, dk, dv, rows, vg = _shapes(q, v, g, cu)
    if do.shape != v.shape:
        raise ValueError("d_out must have the shape of v")
    st = (B, H, dk, dv)
    for name, x in (("init_state", init), ("d_final", dfin)):
        if x is not None and x.shape != st:
            raise ValueError(f"{name} must be {st}")
    dq, dkk = np.zeros(q.shape), np.zeros(k.shape)
    dvv, dg = np.zeros(v.shape), np.zeros(g.shape)
    d_init = np.zeros(st)
    cu_p = None if cu is None else cu.ctypes.data_as(_ip)
    rc = _load().gla_oracle_backward_f64(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), vg, float(scale), _ptr(init), _ptr(do), _ptr(dfin),
        _ptr(dq), _ptr(dkk), _ptr(dvv), _ptr(dg), _ptr(d_init), cu_p, B, H, T, dk, dv,
        int(nthreads))
    if rc != 0:
        raise ValueError("oracle backward rejected its arguments")
    return dq, dkk, dvv, dg, d_init


def bruteforce(q, k, v, g, scale, init_state=None):
    """The recurrence unrolled into one sum per token (dense inputs, tiny sizes).

    Solving the linear recurrence gives
    ``S_t = sum_{j<=t} diag(P(j,t)) k_j^T v_j + diag(P(-1,t)) S_0`` with
    ``P(j,t) = exp(sum_{u=j+1..t} g_u)``, so
    ``o_t = scale * (sum_{j<=t} (q_t . (k_j * P(j,t))) v_j + (q_t * P(-1,t)) S_0)``.
    Evaluated directly in numpy with an explicit causal loop.
    """
    q, k, v, g = _f64(q), _f64(k), _f64(v), _f64(g)
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    vec = g.shape == q.shape
    gg = g if vec else np.broadcast_to(g[..., None], q.shape)
    out = np.zeros((B, T, H, dv))
    final = np.zeros((B, H, dk, dv))
    S0 = np.zeros((B, H, dk, dv)) if init_state is None else _f64(init_state)
    for b in range(B):
        for h in range(H):
            G = gg[b, :, h, :]  # [T, dk]
            for t in range(T):
                acc = np.zeros(dv)
                for j in range(t + 1):
                    P = np.exp(G[j + 1:t + 1].sum(axis=0))
                    acc += np.dot(q[b, t, h] * P, k[b, j, h]) * v[b, j, h]
                P0 = np.exp(G[:t + 1].sum(axis=0))
                acc += (q[b, t, h] * P0) @ S0[b, h]
                out[b, t, h] = scale * acc
            S = np.exp(G.sum(axis=0))[:, None] * S0[b, h]
            for j in range(T):
                P = np.exp(G[j + 1:].sum(axis=0))
                S += np.outer(k[b, j, h] * P, v[b, j, h])
            final[b, h] = S
    return out, final


def decay_schedule(H: int = 16, t_min: float = 1.0, t_max: float = 2048.0):
    """Fixed per-head decays lambda_h of the page's "Decay schedule" paragraph.

    The half-lives are spread geometrically from ``t_min`` to ``t_max`` tokens
    over the H heads, and lambda_h is the per-token decay with that half-life:
    ``T_h = t_min * (t_max / t_min) ** (h / (H - 1))``, ``lambda_h = 2 ** (-1 / T_h)``.
    (The page prints lambda_0 = 0.5 and lambda_15 ~= 0.9997 for 16 heads,
    T_min = 1, T_max = 2048.)  Returns a float64 array; log(lambda_h) is the
    per-token log-decay g of head h.
    """
    h = np.arange(H, dtype=np.float64)
    half_life = t_min * (t_max / t_min) ** (h / (H - 1))
    return 2.0 ** (-1.0 / half_life)


def mixer_epilogue(o, q, k, v, aug=None, norm_w=None, eps=1e-6, z=None):
    """The steps after the readout, per token and head, in fp64 (numpy):

    * self-augmentation (when ``aug`` is given): ``o += sigmoid(q . (aug * k)) * v``
      -- the page adds the value, gated by the query dotted with a learned
      per-key-channel rescaling ``aug`` of the key (``aug = 0`` gives half of v);
    * head RMSNorm (when ``norm_w`` is given): ``o = o / sqrt(mean_j o_j^2 + eps)
      * norm_w[h]`` over the head's dv channels (heads of one decay tier share a
      weight row: the caller lays the rows out per head);
    * output gate (when ``z`` is given): ``o *= silu(z)`` with ``silu(x) = x *
      sigmoid(x)``.

    Shapes: ``o, v [.., H, dv]``, ``q, k [.., H, dk]``, ``aug [H, dk]``,
    ``norm_w [H, dv]``, ``z [.., H, dv]``.  Returns a new fp64 array.
    """
    def sigmoid(x):  # 1 / (1 + exp(-x)), written with tanh so that no exp overflows
        return 0.5 * (1.0 + np.tanh(0.5 * x))

    o = _f64(o).copy()
    if aug is not None:
        q, k, v, a = _f64(q), _f64(k), _f64(v), _f64(aug)
        s = np.sum(q * a * k, axis=-1, keepdims=True)
        o = o + sigmoid(s) * v
    if norm_w is not None:
        w = _f64(norm_w)
        o = o / np.sqrt(np.mean(o * o, axis=-1, keepdims=True) + eps) * w
    if z is not None:
        zz = _f64(z)
        o = o * (zz * sigmoid(zz))
    return o
