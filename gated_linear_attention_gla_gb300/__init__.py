"""Gated linear attention (GLA) on one NVIDIA GB300 (sm_103a).

Python face of ``libgla.so`` (C ABI in ``include/gla.h``).  PyTorch supplies
device memory and streams only; every step of the computation runs in the
library's CUDA kernels, and a missing library is an error, never a fallback.

    out, final = chunk_fwd(q, k, v, g, init_state=S0)          # prefill
    out = decode_step(q, k, v, g, state)                         # one token, in place
    dq, dk, dv, dg, d_init = chunk_bwd(q, k, v, g, d_out, init_state=S0)   # training

The recurrence (the "i14 Laplace 3B on AWS Trainium2" page, paragraph "GLA
mixer"): ``S_t = diag(exp g_t) S_{t-1} + k_t^T v_t``, ``o_t = scale q_t S_t``.
"""
from __future__ import annotations

from typing import Optional

import torch

from . import _binding
from ._binding import (GLA_FLAG_FP32_IO, GLA_FLAG_FP32_OUT, GLA_FLAG_VECTOR_GATE,  # noqa: F401
                       GlaError, lib, status_string, version)

__all__ = ["chunk_fwd", "chunk_bwd", "decode_step", "status_sync", "set_wait_limit_ns", "GlaError",
           "lib", "version",
           "GLA_FLAG_FP32_IO", "GLA_FLAG_FP32_OUT", "GLA_FLAG_VECTOR_GATE"]


def _ptr(t: Optional[torch.Tensor]) -> int:
    return 0 if t is None else t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check(cond: bool, msg: str):
    if not cond:
        raise ValueError(msg)


def _out_dtype(q: torch.Tensor, out, out_dtype):
    if out is not None:
        out_dtype = out.dtype
    if out_dtype is None:
        out_dtype = q.dtype
    _check(out_dtype == q.dtype or (q.dtype == torch.bfloat16 and out_dtype == torch.float32),
           "out is q's dtype, or fp32 for bf16 inputs")
    return out_dtype


def _mixer_args(mixer, q, H, dk, dv, lead):
    """Check the mixer epilogue options {aug [H, dk], norm_w [H, dv] (fp32),
    eps, z [*lead, H, dv] (q's dtype)}; returns (aug, norm_w, eps, z)."""
    if mixer is None:
        return None, None, 0.0, None
    unknown = set(mixer) - {"aug", "norm_w", "eps", "z"}
    _check(not unknown, f"unknown mixer options {sorted(unknown)}")
    aug, norm_w, z = mixer.get("aug"), mixer.get("norm_w"), mixer.get("z")
    eps = float(mixer.get("eps", 1e-6))
    for name, t, shape, dt in (("aug", aug, (H, dk), torch.float32),
                               ("norm_w", norm_w, (H, dv), torch.float32),
                               ("z", z, (*lead, H, dv), q.dtype)):
        if t is not None:
            _check(t.is_cuda and t.is_contiguous() and t.dtype == dt and tuple(t.shape) == shape,
                   f"mixer {name} must be a contiguous {dt} CUDA tensor {shape}")
    return aug, norm_w, eps, z


def _io_flags(q: torch.Tensor, g: torch.Tensor, gate_shape_scalar, gate_shape_vector,
              out_dtype) -> int:
    _check(q.dtype in (torch.bfloat16, torch.float32), "q/k/v must be bf16 or fp32")
    flags = GLA_FLAG_FP32_IO if q.dtype == torch.float32 else 0
    if q.dtype == torch.bfloat16 and out_dtype == torch.float32:
        flags |= GLA_FLAG_FP32_OUT
    _check(g.dtype == torch.float32, "g must be fp32")
    if tuple(g.shape) == tuple(gate_shape_vector):
        flags |= GLA_FLAG_VECTOR_GATE
    else:
        _check(tuple(g.shape) == tuple(gate_shape_scalar),
               f"g must be {tuple(gate_shape_scalar)} or {tuple(gate_shape_vector)}")
    return flags


def chunk_fwd(q, k, v, g, scale: Optional[float] = None, init_state=None, cu_seqlens=None,
              chunk: int = 128, out=None, final_state=None, output_final_state: bool = True,
              stream=None, out_dtype=None, mixer=None):
    """Chunked GLA prefill; returns ``(out, final_state)``.

    Dense: ``q, k [B, T, H, dk]``, ``v [B, T, H, dv]``, ``g [B, T, H]`` or
    ``[B, T, H, dk]`` (fp32).  Packed: ``q, k [1, R, H, dk]`` (or ``[R, H, dk]``)
    with ``cu_seqlens`` int32 ``[B+1]`` on the device.  ``init_state`` and the
    returned ``final_state`` are fp32 ``[B, H, dk, dv]``.  ``out`` has q's dtype,
    or fp32 (``out_dtype=torch.float32``) for bf16 inputs.

    ``mixer`` (optional dict): the steps after the readout (gla_chunk_fwd_mixer:
    the prefill, then a pass over out) -- ``aug`` fp32 [H, dk] (self-augmentation),
    ``norm_w`` fp32 [H, dv] and ``eps`` (head RMSNorm), ``z`` [.., H, dv] in
    q's dtype (SiLU output gate); absent keys skip their step.
    """
    for name, t in (("q", q), ("k", k), ("v", v), ("g", g)):
        _check(t.is_cuda and t.is_contiguous(), f"{name} must be a contiguous CUDA tensor")
    _check(k.shape == q.shape and k.dtype == q.dtype and v.dtype == q.dtype,
           "k must match q; v must have q's dtype")
    H, dk, dv = q.shape[-2], q.shape[-1], v.shape[-1]
    _check(v.shape[:-1] == q.shape[:-1], "v must be [..., H, dv] with q's leading dims")
    if cu_seqlens is not None:
        _check(cu_seqlens.is_cuda and cu_seqlens.dtype == torch.int32,
               "cu_seqlens must be int32 on the GPU")
        B = cu_seqlens.numel() - 1
        T = q.numel() // (H * dk)
        _check(q.dim() == 3 or (q.dim() == 4 and q.shape[0] == 1),
               "packed inputs are [1, R, H, d] or [R, H, d]")
    else:
        _check(q.dim() == 4, "dense inputs are [B, T, H, d]")
        B, T = q.shape[0], q.shape[1]
    out_dtype = _out_dtype(q, out, out_dtype)
    flags = _io_flags(q, g, q.shape[:-1], q.shape, out_dtype)
    if scale is None:
        scale = dk ** -0.5
    if init_state is not None:
        _check(init_state.is_cuda and init_state.dtype == torch.float32 and
               init_state.is_contiguous() and tuple(init_state.shape) == (B, H, dk, dv),
               f"init_state must be contiguous fp32 [{B}, {H}, {dk}, {dv}]")
    if out is None:
        out = torch.empty(v.shape, dtype=out_dtype, device=q.device)
    if final_state is None and output_final_state:
        final_state = torch.empty((B, H, dk, dv), dtype=torch.float32, device=q.device)
    aug, norm_w, eps, z = _mixer_args(mixer, q, H, dk, dv, q.shape[:-2])
    if mixer is None:
        rc = _binding.gla_chunk_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), scale, _ptr(init_state),
                                    _ptr(out), _ptr(final_state), _ptr(cu_seqlens), B, H, T,
                                    dk, dv, chunk, _stream(stream), flags)
        name = "gla_chunk_fwd"
    else:
        rc = _binding.gla_chunk_fwd_mixer(_ptr(q), _ptr(k), _ptr(v), _ptr(g), scale,
                                          _ptr(init_state), _ptr(out), _ptr(final_state),
                                          _ptr(cu_seqlens), B, H, T, dk, dv, chunk, _ptr(aug),
                                          _ptr(norm_w), eps, _ptr(z), _stream(stream), flags)
        name = "gla_chunk_fwd_mixer"
    if rc != 0:
        raise GlaError(rc, name)
    return out, final_state


def chunk_bwd(q, k, v, g, d_out, scale: Optional[float] = None, init_state=None,
              d_final_state=None, cu_seqlens=None, grad_dtype=None, need_dg: bool = True,
              need_d_init: bool = True, tensor_cores: bool = True, workspace=None,
              fixed_workspace: bool = False, stream=None):
    """Gradient of ``chunk_fwd`` (gla_chunk_bwd); returns ``(dq, dk, dv, dg, d_init)``.

    ``q, k, v, g, scale, init_state, cu_seqlens`` as given to ``chunk_fwd``;
    ``d_out`` (q's dtype, v's shape) and ``d_final_state`` (fp32 state, or
    None for zero) are the gradients of the loss with respect to the forward's
    outputs.  ``dq, dk, dv`` come in q's dtype, or fp32 with
    ``grad_dtype=torch.float32`` for bf16 inputs; ``dg`` (fp32, g's shape) and
    ``d_init`` (fp32 state) are None when not requested.

    ``tensor_cores``: use the tensor-core path where it covers the call (bf16;
    per-head gate with dk, dv each 64 or 128, every gradient; per-key-channel
    gate with dk = dv = 128, dv only), with ``workspace`` (a CUDA uint8 tensor of at
    least ``gla_chunk_bwd_workspace_size`` bytes) or a fresh allocation; False
    runs the fp32 CUDA-core kernels.  ``fixed_workspace``: call
    gla_chunk_bwd_fixed_workspace instead, whose workspace is the library's own
    fixed device buffer (nothing is allocated; ``workspace`` is ignored); a
    call whose workspace need exceeds that buffer raises GlaError
    (GLA_ERR_UNSUPPORTED).
    """
    for name, t in (("q", q), ("k", k), ("v", v), ("g", g), ("d_out", d_out)):
        _check(t.is_cuda and t.is_contiguous(), f"{name} must be a contiguous CUDA tensor")
    _check(k.shape == q.shape and k.dtype == q.dtype and v.dtype == q.dtype,
           "k must match q; v must have q's dtype")
    _check(d_out.shape == v.shape and d_out.dtype == q.dtype, "d_out must match v")
    H, dk, dv = q.shape[-2], q.shape[-1], v.shape[-1]
    _check(v.shape[:-1] == q.shape[:-1], "v must be [..., H, dv] with q's leading dims")
    if cu_seqlens is not None:
        _check(cu_seqlens.is_cuda and cu_seqlens.dtype == torch.int32,
               "cu_seqlens must be int32 on the GPU")
        B = cu_seqlens.numel() - 1
        T = q.numel() // (H * dk)
    else:
        _check(q.dim() == 4, "dense inputs are [B, T, H, d]")
        B, T = q.shape[0], q.shape[1]
    grad_dtype = _out_dtype(q, None, grad_dtype)
    flags = _io_flags(q, g, q.shape[:-1], q.shape, grad_dtype)
    if scale is None:
        scale = dk ** -0.5
    st = (B, H, dk, dv)
    for name, t in (("init_state", init_state), ("d_final_state", d_final_state)):
        if t is not None:
            _check(t.is_cuda and t.dtype == torch.float32 and t.is_contiguous() and
                   tuple(t.shape) == st, f"{name} must be contiguous fp32 {list(st)}")
    dq = torch.empty(q.shape, dtype=grad_dtype, device=q.device)
    dk_ = torch.empty(k.shape, dtype=grad_dtype, device=q.device)
    dv_ = torch.empty(v.shape, dtype=grad_dtype, device=q.device)
    dg = torch.empty(g.shape, dtype=torch.float32, device=q.device) if need_dg else None
    d_init = torch.empty(st, dtype=torch.float32, device=q.device) if need_d_init else None
    if fixed_workspace:
        rc = _binding.gla_chunk_bwd_fixed_workspace(
            _ptr(q), _ptr(k), _ptr(v), _ptr(g), scale, _ptr(init_state), _ptr(d_out),
            _ptr(d_final_state), _ptr(dq), _ptr(dk_), _ptr(dv_), _ptr(dg), _ptr(d_init),
            _ptr(cu_seqlens), B, H, T, dk, dv, _stream(stream), flags)
        if rc != 0:
            raise GlaError(rc, "gla_chunk_bwd_fixed_workspace")
        return dq, dk_, dv_, dg, d_init
    ws_bytes = 0
    if tensor_cores:
        ws_bytes = _binding.chunk_bwd_workspace_size(B, H, T, dk, dv, cu_seqlens is not None,
                                                     flags)
        if workspace is not None:
            _check(workspace.is_cuda and workspace.device == q.device and
                   workspace.dtype == torch.uint8 and workspace.is_contiguous() and
                   workspace.data_ptr() % 256 == 0,
                   "workspace must be a contiguous, 256-byte aligned uint8 tensor on q's GPU")
        if ws_bytes and (workspace is None or workspace.numel() < ws_bytes):
            workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    else:
        workspace = None
    rc = _binding.gla_chunk_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), scale, _ptr(init_state),
                                _ptr(d_out), _ptr(d_final_state), _ptr(dq), _ptr(dk_),
                                _ptr(dv_), _ptr(dg), _ptr(d_init), _ptr(cu_seqlens), B, H, T,
                                dk, dv, _ptr(workspace) if ws_bytes else 0, ws_bytes,
                                _stream(stream), flags)
    if rc != 0:
        raise GlaError(rc, "gla_chunk_bwd")
    return dq, dk_, dv_, dg, d_init


def decode_step(q, k, v, g, state, scale: Optional[float] = None, out=None, stream=None,
                out_dtype=None, slots=None, mixer=None):
    """One recurrent step for N sequences; ``state [N, H, dk, dv]`` (fp32) is
    updated in place.  ``q, k [N, H, dk]``, ``v [N, H, dv]``, ``g [N, H]`` or
    ``[N, H, dk]``.  Returns ``out [N, H, dv]`` in q's dtype (or fp32).

    With ``slots`` (int32 [N] on the GPU) ``state`` is a pool
    ``[num_slots, H, dk, dv]`` and row n uses page ``slots[n]`` (-1: a padding
    row that does nothing; see gla_decode_step_slots).  ``mixer``: the steps
    after the readout, fused into the step (as for ``chunk_fwd``; ``z`` is
    [N, H, dv])."""
    for name, t in (("q", q), ("k", k), ("v", v), ("g", g), ("state", state)):
        _check(t.is_cuda and t.is_contiguous(), f"{name} must be a contiguous CUDA tensor")
    _check(q.dim() == 3 and k.shape == q.shape and v.shape[:-1] == q.shape[:-1],
           "q, k are [N, H, dk] and v is [N, H, dv]")
    _check(k.dtype == q.dtype and v.dtype == q.dtype, "q, k, v share one dtype")
    N, H, dk = q.shape
    dv = v.shape[-1]
    if slots is None:
        _check(state.dtype == torch.float32 and tuple(state.shape) == (N, H, dk, dv),
               f"state must be fp32 [{N}, {H}, {dk}, {dv}]")
    else:
        _check(slots.is_cuda and slots.dtype == torch.int32 and slots.is_contiguous() and
               tuple(slots.shape) == (N,), f"slots must be contiguous int32 [{N}] on the GPU")
        _check(state.dtype == torch.float32 and state.dim() == 4 and
               tuple(state.shape[1:]) == (H, dk, dv),
               f"the state pool must be fp32 [num_slots, {H}, {dk}, {dv}]")
    out_dtype = _out_dtype(q, out, out_dtype)
    flags = _io_flags(q, g, (N, H), (N, H, dk), out_dtype)
    if scale is None:
        scale = dk ** -0.5
    if out is None:
        out = torch.empty((N, H, dv), dtype=out_dtype, device=q.device)
    if mixer is not None:
        aug, norm_w, eps, z = _mixer_args(mixer, q, H, dk, dv, (N,))
        rc = _binding.gla_decode_step_mixer(
            _ptr(q), _ptr(k), _ptr(v), _ptr(g), scale, _ptr(state),
            0 if slots is None else state.shape[0], _ptr(slots), _ptr(out), N, H, dk, dv,
            _ptr(aug), _ptr(norm_w), eps, _ptr(z), _stream(stream), flags)
        name = "gla_decode_step_mixer"
    elif slots is None:
        rc = _binding.gla_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(g), scale, _ptr(state),
                                      _ptr(out), N, H, dk, dv, _stream(stream), flags)
        name = "gla_decode_step"
    else:
        rc = _binding.gla_decode_step_slots(_ptr(q), _ptr(k), _ptr(v), _ptr(g), scale,
                                            _ptr(state), state.shape[0], _ptr(slots), _ptr(out),
                                            N, H, dk, dv, _stream(stream), flags)
        name = "gla_decode_step_slots"
    if rc != 0:
        raise GlaError(rc, name)
    return out


def set_wait_limit_ns(nanoseconds: int) -> int:
    """Wall-time limit of the tensor-core prefill kernels' hand-off waits
    (process-wide; 0 restores the default, 2 s).  Returns the previous setting.
    A wait that runs out ends the kernel early: the next status_sync() raises
    GlaError with GLA_ERR_TIMEOUT (5) and the call's outputs are undefined."""
    return _binding.gla_set_wait_limit_ns(nanoseconds)


def status_sync(stream=None) -> int:
    """Synchronise ``stream`` and return (and clear) the device status; raises on error."""
    rc = _binding.gla_status_sync(_stream(stream))
    if rc != 0:
        raise GlaError(rc, "gla_status_sync")
    return rc
