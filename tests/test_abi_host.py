"""The C ABI library on the host: it builds, loads, exports every declared
symbol, and rejects bad arguments before touching the GPU (CPU only)."""
import ctypes
import os
import re

import pytest

from gated_linear_attention_gla_gb300 import _binding, build as glabuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gla.h")

A = 1 << 20  # a 16-byte-aligned fake device address; never dereferenced here
FAKE = [A * (i + 1) for i in range(12)]


@pytest.fixture(scope="module")
def L():
    glabuild.build()
    return _binding.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gla_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("gla_chunk_fwd", "gla_chunk_bwd", "gla_decode_step", "gla_decode_step_slots",
              "gla_status_string", "gla_status_sync"):
        assert n in names


def test_every_declared_symbol_is_exported(L):
    for name in declared_functions():
        assert hasattr(L, name), f"{name} declared in gla.h but not exported"


def test_no_torch_in_the_library(L):
    # the boundary is a plain C library: it must not need libtorch/libc10
    import subprocess
    out = subprocess.run(["ldd", _binding.LIB_PATH], capture_output=True, text=True).stdout
    libs = [line.split()[0] for line in out.splitlines() if line.strip()]
    assert not [x for x in libs if re.match(r"lib(torch|c10)", os.path.basename(x))]


def test_status_strings(L):
    for s in range(6):
        assert _binding.status_string(s)
    assert _binding.status_string(99) == "unknown status"
    assert re.match(r"^\d+\.\d+\.\d+$", _binding.version())


def chunk(q=FAKE[0], k=FAKE[1], v=FAKE[2], g=FAKE[3], scale=0.1, init=FAKE[4], out=FAKE[5],
          final=FAKE[6], cu=0, B=2, H=4, T=256, dk=128, dv=128, chunk=128, flags=0):
    return _binding.gla_chunk_fwd(q, k, v, g, scale, init, out, final, cu, B, H, T, dk, dv,
                                  chunk, 0, flags)


def decode(q=FAKE[0], k=FAKE[1], v=FAKE[2], g=FAKE[3], scale=0.1, state=FAKE[4], out=FAKE[5],
           N=8, H=4, dk=128, dv=128, flags=0):
    return _binding.gla_decode_step(q, k, v, g, scale, state, out, N, H, dk, dv, 0, flags)


E = _binding


@pytest.mark.parametrize("kw,status", [
    (dict(flags=1 << 5), E.GLA_ERR_INVALID_ARG),
    (dict(B=-1), E.GLA_ERR_INVALID_ARG),
    (dict(H=-3), E.GLA_ERR_INVALID_ARG),
    (dict(T=-1), E.GLA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), E.GLA_ERR_INVALID_ARG),
    (dict(scale=float("inf")), E.GLA_ERR_INVALID_ARG),
    (dict(dk=80), E.GLA_ERR_UNSUPPORTED),
    (dict(dk=192), E.GLA_ERR_UNSUPPORTED),
    (dict(dv=256), E.GLA_ERR_UNSUPPORTED),
    (dict(chunk=100), E.GLA_ERR_UNSUPPORTED),
    (dict(chunk=256), E.GLA_ERR_UNSUPPORTED),
    (dict(q=0), E.GLA_ERR_INVALID_ARG),
    (dict(g=0), E.GLA_ERR_INVALID_ARG),
    (dict(out=0), E.GLA_ERR_INVALID_ARG),
    (dict(q=FAKE[0] + 8), E.GLA_ERR_MISALIGNED),
    (dict(out=FAKE[5] + 2), E.GLA_ERR_MISALIGNED),
    (dict(init=FAKE[4] + 4), E.GLA_ERR_MISALIGNED),
    (dict(g=FAKE[3] + 2), E.GLA_ERR_MISALIGNED),
    (dict(g=FAKE[3] + 4, flags=E.GLA_FLAG_VECTOR_GATE), E.GLA_ERR_MISALIGNED),
    (dict(cu=FAKE[7] + 2), E.GLA_ERR_MISALIGNED),
    (dict(out=FAKE[0]), E.GLA_ERR_INVALID_ARG),          # out aliases q
    (dict(out=FAKE[2] + 64), E.GLA_ERR_INVALID_ARG),     # out overlaps v
    (dict(final=FAKE[4] + 16), E.GLA_ERR_INVALID_ARG),   # final partially overlaps init
    (dict(final=FAKE[1]), E.GLA_ERR_INVALID_ARG),        # final overlaps k
    (dict(B=1 << 20, T=1 << 20), E.GLA_ERR_INVALID_ARG),  # size overflow
])
def test_chunk_fwd_rejects_before_launch(L, kw, status):
    assert chunk(**kw) == status


def test_chunk_fwd_empty_problems_are_no_ops(L):
    # nothing to compute and nothing to write: returns before any CUDA call
    assert chunk(B=0) == E.GLA_OK
    assert chunk(H=0) == E.GLA_OK
    assert chunk(T=0, final=0, q=0, k=0, v=0, g=0, out=0) == E.GLA_OK


@pytest.mark.parametrize("kw,status", [
    (dict(flags=1 << 7), E.GLA_ERR_INVALID_ARG),
    (dict(N=-1), E.GLA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), E.GLA_ERR_INVALID_ARG),
    (dict(dk=32), E.GLA_ERR_UNSUPPORTED),
    (dict(dv=96), E.GLA_ERR_UNSUPPORTED),
    (dict(dv=256), E.GLA_ERR_UNSUPPORTED),
    (dict(state=0), E.GLA_ERR_INVALID_ARG),
    (dict(k=0), E.GLA_ERR_INVALID_ARG),
    (dict(v=FAKE[2] + 4), E.GLA_ERR_MISALIGNED),
    (dict(state=FAKE[4] + 8), E.GLA_ERR_MISALIGNED),
    (dict(g=FAKE[3] + 1), E.GLA_ERR_MISALIGNED),
    (dict(out=FAKE[4]), E.GLA_ERR_INVALID_ARG),          # out inside the state
    (dict(state=FAKE[0]), E.GLA_ERR_INVALID_ARG),        # state overlaps q
    (dict(N=1 << 20, H=1 << 12), E.GLA_ERR_INVALID_ARG),  # too many units
])
def test_decode_step_rejects_before_launch(L, kw, status):
    assert decode(**kw) == status


def decode_slots(q=FAKE[0], k=FAKE[1], v=FAKE[2], g=FAKE[3], scale=0.1, pool=FAKE[4],
                 num_slots=16, slots=FAKE[6], out=FAKE[5], N=8, H=4, dk=128, dv=128, flags=0):
    return _binding.gla_decode_step_slots(q, k, v, g, scale, pool, num_slots, slots, out, N, H,
                                          dk, dv, 0, flags)


@pytest.mark.parametrize("kw,status", [
    (dict(slots=0), E.GLA_ERR_INVALID_ARG),
    (dict(num_slots=-1), E.GLA_ERR_INVALID_ARG),
    (dict(slots=FAKE[6] + 2), E.GLA_ERR_MISALIGNED),
    (dict(dv=96), E.GLA_ERR_UNSUPPORTED),
    (dict(out=FAKE[4]), E.GLA_ERR_INVALID_ARG),        # out inside the pool
    (dict(slots=FAKE[4] + 64), E.GLA_ERR_INVALID_ARG),  # slots inside the pool
    (dict(num_slots=1 << 20, H=1 << 12), E.GLA_ERR_INVALID_ARG),  # pool too large
])
def test_decode_slots_rejects_before_launch(L, kw, status):
    assert decode_slots(**kw) == status


def test_decode_slots_empty_is_no_op(L):
    assert decode_slots(N=0) == E.GLA_OK
    assert decode_slots(H=0) == E.GLA_OK


def test_decode_step_empty_is_no_op(L):
    assert decode(N=0) == E.GLA_OK
    assert decode(H=0) == E.GLA_OK


def test_ctypes_signatures_match_header(L):
    """The binding's argument counts equal the header's parameter counts."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    for name in ("gla_chunk_fwd", "gla_chunk_fwd_mixer", "gla_chunk_bwd",
                 "gla_chunk_bwd_fixed_workspace",
                 "gla_chunk_bwd_workspace_size", "gla_decode_step", "gla_decode_step_slots",
                 "gla_decode_step_mixer", "gla_mixer_epilogue", "gla_status_sync",
                 "gla_status_string"):
        m = re.search(name + r"\s*\(([^)]*)\)", text)
        nparams = len([p for p in m.group(1).split(",") if p.strip() and p.strip() != "void"])
        assert len(getattr(L, name).argtypes) == nparams, name


def epilogue(out=FAKE[5], q=FAKE[0], k=FAKE[1], v=FAKE[2], aug=FAKE[7], norm_w=FAKE[8], eps=1e-6,
             z=FAKE[9], rows=16, H=4, dk=128, dv=128, flags=0):
    return _binding.gla_mixer_epilogue(out, q, k, v, aug, norm_w, eps, z, rows, H, dk, dv, 0,
                                       flags)


@pytest.mark.parametrize("kw,status", [
    (dict(flags=E.GLA_FLAG_VECTOR_GATE), E.GLA_ERR_INVALID_ARG),   # not an epilogue flag
    (dict(eps=-1.0), E.GLA_ERR_INVALID_ARG),
    (dict(eps=float("inf")), E.GLA_ERR_INVALID_ARG),
    (dict(rows=-1), E.GLA_ERR_INVALID_ARG),
    (dict(out=0), E.GLA_ERR_INVALID_ARG),
    (dict(q=0), E.GLA_ERR_INVALID_ARG),              # aug needs q, k, v
    (dict(dk=80), E.GLA_ERR_UNSUPPORTED),
    (dict(out=FAKE[5] + 1), E.GLA_ERR_MISALIGNED),
    (dict(aug=FAKE[7] + 2), E.GLA_ERR_MISALIGNED),
    (dict(z=FAKE[5] + 64), E.GLA_ERR_INVALID_ARG),   # z inside out
])
def test_mixer_epilogue_rejects_before_launch(L, kw, status):
    assert epilogue(**kw) == status


def test_mixer_epilogue_trivial_calls_are_no_ops(L):
    assert epilogue(rows=0) == E.GLA_OK
    assert epilogue(H=0) == E.GLA_OK
    assert epilogue(aug=0, norm_w=0, z=0) == E.GLA_OK            # nothing to apply
    assert epilogue(aug=0, norm_w=0, z=0, q=0, k=0, v=0) == E.GLA_OK


def test_decode_mixer_rejects_before_launch(L):
    call = lambda **kw: _binding.gla_decode_step_mixer(
        *[kw.get(n, d) for n, d in (("q", FAKE[0]), ("k", FAKE[1]), ("v", FAKE[2]),
                                     ("g", FAKE[3]))], 0.1, FAKE[4], kw.get("num_slots", 0),
        kw.get("slots", 0), FAKE[5], 8, 4, 128, 128, FAKE[7], FAKE[8], kw.get("eps", 1e-6),
        FAKE[9], 0, 0)
    assert call(num_slots=3) == E.GLA_ERR_INVALID_ARG      # a pool size without slots
    assert call(eps=-0.5) == E.GLA_ERR_INVALID_ARG
    assert call(q=0) == E.GLA_ERR_INVALID_ARG


WS = 1 << 32  # a fake 256-byte-aligned workspace far from the other fake tensors


def bwd(q=FAKE[0], k=FAKE[1], v=FAKE[2], g=FAKE[3], scale=0.1, init=FAKE[4], d_out=FAKE[5],
        d_final=FAKE[6], dq=FAKE[7], dk_out=FAKE[8], dv_out=FAKE[9], dg=FAKE[10],
        d_init=FAKE[11], cu=0, B=2, H=4, T=256, dk=128, dv=128, ws=0, ws_bytes=0, flags=0):
    return _binding.gla_chunk_bwd(q, k, v, g, scale, init, d_out, d_final, dq, dk_out, dv_out,
                                  dg, d_init, cu, B, H, T, dk, dv, ws, ws_bytes, 0, flags)


@pytest.mark.parametrize("kw,status", [
    (dict(flags=1 << 5), E.GLA_ERR_INVALID_ARG),
    (dict(B=-1), E.GLA_ERR_INVALID_ARG),
    (dict(T=-2), E.GLA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), E.GLA_ERR_INVALID_ARG),
    (dict(dk=80), E.GLA_ERR_UNSUPPORTED),
    (dict(dv=96), E.GLA_ERR_UNSUPPORTED),
    (dict(d_out=0), E.GLA_ERR_INVALID_ARG),
    (dict(dq=0), E.GLA_ERR_INVALID_ARG),
    (dict(dv_out=0), E.GLA_ERR_INVALID_ARG),
    (dict(dq=FAKE[7] + 8), E.GLA_ERR_MISALIGNED),
    (dict(dg=FAKE[10] + 4), E.GLA_ERR_MISALIGNED),
    (dict(d_init=FAKE[11] + 4), E.GLA_ERR_MISALIGNED),
    (dict(g=FAKE[3] + 4, flags=E.GLA_FLAG_VECTOR_GATE), E.GLA_ERR_MISALIGNED),
    (dict(dq=FAKE[0]), E.GLA_ERR_INVALID_ARG),             # dq overlaps q
    (dict(dk_out=FAKE[7] + 64), E.GLA_ERR_INVALID_ARG),    # dk overlaps dq
    (dict(d_init=FAKE[6]), E.GLA_ERR_INVALID_ARG),         # d_init overlaps d_final
    (dict(dg=FAKE[5] + 256), E.GLA_ERR_INVALID_ARG),       # dg inside d_out
    (dict(B=1 << 20, T=1 << 20), E.GLA_ERR_INVALID_ARG),   # size overflow
    (dict(ws=WS + 16, ws_bytes=1 << 30), E.GLA_ERR_MISALIGNED),
    (dict(ws=FAKE[7], ws_bytes=1 << 30), E.GLA_ERR_INVALID_ARG),  # workspace over dq and more
])
def test_chunk_bwd_rejects_before_launch(L, kw, status):
    assert bwd(**kw) == status


def test_chunk_bwd_empty_problems_are_no_ops(L):
    assert bwd(B=0) == E.GLA_OK
    assert bwd(H=0) == E.GLA_OK
    assert bwd(T=0, d_init=0, q=0, k=0, v=0, g=0, d_out=0, dq=0, dk_out=0, dv_out=0,
               dg=0) == E.GLA_OK


def test_chunk_bwd_workspace_size(L):
    ws = _binding.chunk_bwd_workspace_size
    n = ws(2, 4, 256, 128, 128, 0, 0)
    assert n > 0 and n % 256 == 0
    # reversed q, k, v, do (bf16), the shifted gate and four states (the prefill
    # runs store the gradients in the caller's buffers directly)
    tok = 2 * 256 * 4
    states = 4 * 2 * 4 * 128 * 128 * 4
    assert n == tok * 128 * 4 * 2 + tok * 4 + states
    assert ws(2, 4, 512, 128, 128, 1, 0) == n          # packed: T counts the rows
    assert ws(2, 4, 256, 128, 128, 0, E.GLA_FLAG_FP32_IO) == 0
    # per-key-channel gate: reversed q, k, do (bf16), the gate rows, a state
    nv = ws(2, 4, 256, 128, 128, 0, E.GLA_FLAG_VECTOR_GATE)
    assert nv >= tok * 128 * (3 * 2 + 4) + 2 * 4 * 128 * 128 * 4
    assert nv < tok * 128 * (3 * 2 + 4 + 4) + 2 * 4 * 128 * 128 * 4
    assert ws(2, 4, 256, 96, 192, 0, 0) == 0
    assert ws(2, 4, 256, 128, 192, 0, 0) == 0
    assert ws(2, 4, 256, 64, 64, 0, E.GLA_FLAG_VECTOR_GATE) == 0
    # per-head gate, head sizes 64 and 128 in any pair: the same sections at their widths
    for dk, dv in ((64, 64), (64, 128), (128, 64)):
        assert ws(2, 4, 256, dk, dv, 0, 0) == tok * (2 * dk + 2 * dv) * 2 + tok * 4 + \
            4 * 2 * 4 * dk * dv * 4
    assert ws(0, 4, 256, 128, 128, 0, 0) == 0


def test_chunk_bwd_fixed_workspace_rejects_before_launch(L):
    call = lambda **kw: _binding.gla_chunk_bwd_fixed_workspace(  # noqa: E731
        *[kw.get(n, d) for n, d in (("q", FAKE[0]), ("k", FAKE[1]), ("v", FAKE[2]),
                                     ("g", FAKE[3]))], kw.get("scale", 0.1), FAKE[4], FAKE[5],
        FAKE[6], kw.get("dq", FAKE[7]), FAKE[8], FAKE[9], FAKE[10], FAKE[11], 0, 2, 4,
        kw.get("T", 256), kw.get("dk", 128), 128, 0, kw.get("flags", 0))
    assert call(flags=1 << 5) == E.GLA_ERR_INVALID_ARG
    assert call(dk=80) == E.GLA_ERR_UNSUPPORTED
    assert call(dq=0) == E.GLA_ERR_INVALID_ARG
    assert call(dq=FAKE[0]) == E.GLA_ERR_INVALID_ARG       # dq overlaps q
    assert call(scale=float("nan")) == E.GLA_ERR_INVALID_ARG
    assert call(T=-1) == E.GLA_ERR_INVALID_ARG


def test_chunk_bwd_fixed_workspace_rejects_oversize_on_the_host(L):
    """A call whose workspace need exceeds the fixed 384 MiB buffer is rejected
    on the host, before any CUDA call (there is no GPU here, so a CUDA call
    would have failed with GLA_ERR_CUDA instead), and the message names the
    need and the limit."""
    big = [(i + 1) << 32 for i in range(12)]  # fake device addresses 4 GiB apart
    B, H, T = 16, 16, 2048
    need = _binding.chunk_bwd_workspace_size(B, H, T, 128, 128, False, 0)
    assert need > 384 << 20
    rc = _binding.gla_chunk_bwd_fixed_workspace(*big[:4], 0.1, big[4], big[5], big[6],
                                                *big[7:12], 0, B, H, T, 128, 128, 0, 0)
    assert rc == E.GLA_ERR_UNSUPPORTED
    msg = L.gla_last_error_string().decode()
    assert str(need) in msg and str(384 << 20) in msg, msg
    # a smaller call with the same pointers gets past this check and fails only
    # where it needs the GPU
    rc = _binding.gla_chunk_bwd_fixed_workspace(*big[:4], 0.1, big[4], big[5], big[6],
                                                *big[7:12], 0, 2, H, T, 128, 128, 0, 0)
    assert rc == E.GLA_ERR_CUDA


def test_chunk_fwd_mixer_rejects_before_launch(L):
    def call(**kw):
        a = dict(q=FAKE[0], k=FAKE[1], v=FAKE[2], g=FAKE[3], init=FAKE[4], out=FAKE[5],
                 final=FAKE[6], aug=FAKE[7], norm_w=FAKE[8], eps=1e-6, z=FAKE[9], flags=0)
        a.update(kw)
        return _binding.gla_chunk_fwd_mixer(a["q"], a["k"], a["v"], a["g"], 0.1, a["init"],
                                            a["out"], a["final"], 0, 2, 4, 256, 128, 128, 128,
                                            a["aug"], a["norm_w"], a["eps"], a["z"], 0,
                                            a["flags"])
    assert call(eps=-1.0) == E.GLA_ERR_INVALID_ARG
    assert call(eps=float("nan")) == E.GLA_ERR_INVALID_ARG
    assert call(aug=FAKE[7] + 4) == E.GLA_ERR_MISALIGNED
    assert call(z=FAKE[5] + 64) == E.GLA_ERR_INVALID_ARG     # z inside out
    assert call(aug=FAKE[5]) == E.GLA_ERR_INVALID_ARG        # aug inside out
    assert call(q=FAKE[0] + 8) == E.GLA_ERR_MISALIGNED       # the prefill's own checks
    assert call(out=FAKE[0]) == E.GLA_ERR_INVALID_ARG


def test_wait_limit_setting_round_trips(L):
    """gla_set_wait_limit_ns is host-only: it returns the previous setting."""
    L.gla_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
    L.gla_set_wait_limit_ns.restype = ctypes.c_uint64
    old = L.gla_set_wait_limit_ns(12345)
    try:
        assert L.gla_set_wait_limit_ns(777) == 12345
    finally:
        assert L.gla_set_wait_limit_ns(old) == 777
