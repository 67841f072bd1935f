"""ctypes binding of libgla.so -- argument marshalling only.

Every call goes straight to the C ABI declared in ``include/gla.h``; all
arithmetic runs in the library's CUDA kernels.  If the library is missing the
first call raises: there is no fallback of any kind.
"""
from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libgla.so")

GLA_OK = 0
GLA_ERR_INVALID_ARG = 1
GLA_ERR_UNSUPPORTED = 2
GLA_ERR_MISALIGNED = 3
GLA_ERR_CUDA = 4
GLA_ERR_TIMEOUT = 5

GLA_FLAG_FP32_IO = 1 << 0
GLA_FLAG_VECTOR_GATE = 1 << 1
GLA_FLAG_FP32_OUT = 1 << 2

_lock = threading.Lock()
_lib = None

_vp = ctypes.c_void_p
_i = ctypes.c_int


class GlaError(RuntimeError):
    """A libgla call returned a non-OK status."""

    def __init__(self, status: int, where: str):
        self.status = status
        msg = f"{where}: {status_string(status)} (status {status})"
        if status == GLA_ERR_CUDA:
            msg += f": {lib().gla_last_error_string().decode()}"
        super().__init__(msg)


def lib() -> ctypes.CDLL:
    """Load libgla.so (once).  Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it with "
                    "`python -m gated_linear_attention_gla_gb300.build` "
                    "(or __graft_entry__.build()); there is no CPU fallback")
            L = ctypes.CDLL(LIB_PATH)
            L.gla_chunk_fwd.argtypes = [_vp, _vp, _vp, _vp, ctypes.c_float, _vp, _vp, _vp, _vp,
                                        _i, _i, _i, _i, _i, _i, _vp, ctypes.c_uint]
            L.gla_chunk_fwd.restype = _i
            L.gla_chunk_fwd_mixer.argtypes = [_vp, _vp, _vp, _vp, ctypes.c_float, _vp, _vp,
                                              _vp, _vp, _i, _i, _i, _i, _i, _i, _vp, _vp,
                                              ctypes.c_float, _vp, _vp, ctypes.c_uint]
            L.gla_chunk_fwd_mixer.restype = _i
            L.gla_decode_step.argtypes = [_vp, _vp, _vp, _vp, ctypes.c_float, _vp, _vp,
                                          _i, _i, _i, _i, _vp, ctypes.c_uint]
            L.gla_decode_step.restype = _i
            L.gla_decode_step_slots.argtypes = [_vp, _vp, _vp, _vp, ctypes.c_float, _vp, _i, _vp,
                                                _vp, _i, _i, _i, _i, _vp, ctypes.c_uint]
            L.gla_decode_step_slots.restype = _i
            L.gla_decode_step_mixer.argtypes = [_vp, _vp, _vp, _vp, ctypes.c_float, _vp, _i, _vp,
                                                _vp, _i, _i, _i, _i, _vp, _vp, ctypes.c_float,
                                                _vp, _vp, ctypes.c_uint]
            L.gla_decode_step_mixer.restype = _i
            L.gla_mixer_epilogue.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_float, _vp,
                                             _i, _i, _i, _i, _vp, ctypes.c_uint]
            L.gla_mixer_epilogue.restype = _i
            L.gla_chunk_bwd.argtypes = [_vp, _vp, _vp, _vp, ctypes.c_float, _vp, _vp, _vp,
                                        _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp,
                                        ctypes.c_size_t, _vp, ctypes.c_uint]
            L.gla_chunk_bwd.restype = _i
            L.gla_chunk_bwd_fixed_workspace.argtypes = [
                _vp, _vp, _vp, _vp, ctypes.c_float, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                _i, _i, _i, _i, _i, _vp, ctypes.c_uint]
            L.gla_chunk_bwd_fixed_workspace.restype = _i
            L.gla_chunk_bwd_workspace_size.argtypes = [_i, _i, _i, _i, _i, _i, ctypes.c_uint]
            L.gla_chunk_bwd_workspace_size.restype = ctypes.c_size_t
            L.gla_status_string.argtypes = [_i]
            L.gla_status_string.restype = ctypes.c_char_p
            L.gla_status_sync.argtypes = [_vp]
            L.gla_status_sync.restype = _i
            L.gla_version.argtypes = []
            L.gla_version.restype = ctypes.c_char_p
            L.gla_chunk_fwd_kernel.argtypes = [_i, _i, _i, ctypes.c_uint]
            L.gla_chunk_fwd_kernel.restype = ctypes.c_char_p
            L.gla_last_error_string.argtypes = []
            L.gla_last_error_string.restype = ctypes.c_char_p
            L.gla_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
            L.gla_set_wait_limit_ns.restype = ctypes.c_uint64
            _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().gla_status_string(int(status)).decode()


def version() -> str:
    return lib().gla_version().decode()


def gla_chunk_fwd(q, k, v, g, scale, init_state, out, final_state, cu_seqlens, B, H, T, dk,
                  dv, chunk, stream, flags) -> int:
    """Raw call: pointers are ints (0 = NULL), ``stream`` an int handle."""
    return lib().gla_chunk_fwd(q or None, k or None, v or None, g or None, float(scale),
                               init_state or None, out or None, final_state or None,
                               cu_seqlens or None, B, H, T, dk, dv, chunk, stream or None,
                               flags)


def gla_chunk_fwd_mixer(q, k, v, g, scale, init_state, out, final_state, cu_seqlens, B, H, T,
                        dk, dv, chunk, aug, norm_w, eps, z, stream, flags) -> int:
    """Raw call: pointers are ints (0 = NULL), ``stream`` an int handle."""
    n = lambda p: p or None  # noqa: E731
    return lib().gla_chunk_fwd_mixer(n(q), n(k), n(v), n(g), float(scale), n(init_state),
                                     n(out), n(final_state), n(cu_seqlens), B, H, T, dk, dv,
                                     chunk, n(aug), n(norm_w), float(eps), n(z), n(stream),
                                     flags)


def gla_decode_step(q, k, v, g, scale, state_inout, out, N, H, dk, dv, stream, flags) -> int:
    """Raw call: pointers are ints, ``stream`` an int handle."""
    return lib().gla_decode_step(q or None, k or None, v or None, g or None, float(scale),
                                 state_inout or None, out or None, N, H, dk, dv,
                                 stream or None, flags)


def gla_decode_step_slots(q, k, v, g, scale, state_pool, num_slots, slots, out, N, H, dk, dv,
                          stream, flags) -> int:
    """Raw call: pointers are ints, ``stream`` an int handle."""
    return lib().gla_decode_step_slots(q or None, k or None, v or None, g or None, float(scale),
                                       state_pool or None, num_slots, slots or None,
                                       out or None, N, H, dk, dv, stream or None, flags)


def gla_decode_step_mixer(q, k, v, g, scale, state, num_slots, slots, out, N, H, dk, dv, aug,
                          norm_w, eps, z, stream, flags) -> int:
    """Raw call: pointers are ints, ``stream`` an int handle."""
    return lib().gla_decode_step_mixer(q or None, k or None, v or None, g or None, float(scale),
                                       state or None, num_slots, slots or None, out or None, N,
                                       H, dk, dv, aug or None, norm_w or None, float(eps),
                                       z or None, stream or None, flags)


def gla_mixer_epilogue(out, q, k, v, aug, norm_w, eps, z, rows, H, dk, dv, stream, flags) -> int:
    """Raw call: pointers are ints, ``stream`` an int handle."""
    return lib().gla_mixer_epilogue(out or None, q or None, k or None, v or None, aug or None,
                                    norm_w or None, float(eps), z or None, rows, H, dk, dv,
                                    stream or None, flags)


def gla_chunk_bwd(q, k, v, g, scale, init_state, d_out, d_final, dq, dk_out, dv_out, dg,
                  d_init, cu_seqlens, B, H, T, dk, dv, workspace, workspace_bytes, stream,
                  flags) -> int:
    """Raw call: pointers are ints (0 = NULL), ``stream`` an int handle."""
    n = lambda p: p or None  # noqa: E731
    return lib().gla_chunk_bwd(n(q), n(k), n(v), n(g), float(scale), n(init_state), n(d_out),
                               n(d_final), n(dq), n(dk_out), n(dv_out), n(dg), n(d_init),
                               n(cu_seqlens), B, H, T, dk, dv, n(workspace),
                               int(workspace_bytes), n(stream), flags)


def gla_chunk_bwd_fixed_workspace(q, k, v, g, scale, init_state, d_out, d_final, dq, dk_out,
                                  dv_out, dg, d_init, cu_seqlens, B, H, T, dk, dv, stream,
                                  flags) -> int:
    """Raw call: pointers are ints (0 = NULL), ``stream`` an int handle."""
    n = lambda p: p or None  # noqa: E731
    return lib().gla_chunk_bwd_fixed_workspace(
        n(q), n(k), n(v), n(g), float(scale), n(init_state), n(d_out), n(d_final), n(dq),
        n(dk_out), n(dv_out), n(dg), n(d_init), n(cu_seqlens), B, H, T, dk, dv, n(stream), flags)


def chunk_bwd_workspace_size(B, H, T, dk, dv, packed, flags) -> int:
    """Workspace bytes for gla_chunk_bwd's tensor-core path (0: not covered)."""
    return int(lib().gla_chunk_bwd_workspace_size(B, H, T, dk, dv, int(bool(packed)), flags))


def chunk_fwd_kernel(dk, dv, chunk, flags):
    """Name of the kernel gla_chunk_fwd would run ("tensor_core" / "cuda_core"), or None."""
    r = lib().gla_chunk_fwd_kernel(dk, dv, chunk, flags)
    return None if r is None else r.decode()


def gla_status_sync(stream) -> int:
    return lib().gla_status_sync(stream or None)


def gla_set_wait_limit_ns(nanoseconds) -> int:
    """Set the tensor-core kernels' hand-off wait limit (0: default); returns the previous one."""
    return int(lib().gla_set_wait_limit_ns(int(nanoseconds)))
