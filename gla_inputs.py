"""Seeded synthetic inputs for gated linear attention (shared by tests and bench).

This module holds input recipes only -- shapes, distributions and seeds -- and
none of the method's arithmetic.  Both the CUDA path and the CPU oracle are
fed from it; it imports neither of them.

Every tensor is drawn on the CPU from ``torch.Generator`` seeded with
``1000 + workload index`` and rounded once to the I/O dtype, so both sides
read bit-identical values.  Recipes (the five workloads the method is served
and measured on):

==========  ===============================================================
tiny        B=1, H=2, T=256, dk=dv=64, chunk 64, fp32 I/O, zero initial state
prefill     B=4, H=16, T=2048 (16 chunks of 128), dk=dv=128, bf16 I/O,
            initial state N(0, 0.02)
decode      N=1280 sequences, H=16, dk=dv=128, bf16 I/O, fp32 state
            N(0, 0.1) updated in place, 64 distinct steps
varlen      16 sequences, lengths uniform in [512, 16384] packed with
            cu_seqlens, H=32, dk=dv=128, chunk 128, initial state N(0, 0.05)
vector      B=8, H=16, T=4096, dk=dv=128, chunk 128, per-key-channel gate,
            zero initial state
laplace     B=8, H=16, T=2048, dk=96, dv=192 (the Laplace 3B head), chunk 128,
            the fixed geometric per-head decay (half-lives 1 .. 2048 tokens),
            initial state N(0, 0.02)
==========  ===============================================================

Common distributions: q, k, v ~ N(0, 1) (standard deviation 1); k is
L2-normalised per (token, head) in fp32 before rounding; the gate is
``g = logsigmoid(x) / g_div`` with ``x ~ N(g_mu, 1)`` (g_mu 3, except 4 for
varlen and 2 with g_div 4 for the vector gate), except for the laplace
workload, whose gate is the page's fixed per-head decay: head h has the
half-life T_h = 2048 ** (h / 15) tokens and g = -ln 2 / T_h for every token;
``scale = dk ** -0.5``.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch
import torch.nn.functional as F


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    index: int
    H: int
    dk: int
    dv: int
    io: str = "bf16"            # "bf16" or "fp32": dtype of q, k, v and out
    gate: str = "scalar"        # "scalar" ([.., H]) or "vector" ([.., H, dk])
    decay: str = "random"       # "random" (logsigmoid of a normal) or "schedule" (fixed per head)
    g_mu: float = 3.0
    g_div: float = 1.0
    B: int = 0                  # dense prefill batch
    T: int = 0                  # dense prefill length
    chunk: int = 128
    init_std: float = 0.0       # 0 -> no initial state (zeros)
    nseq: int = 0               # packed prefill: number of sequences
    len_lo: int = 0
    len_hi: int = 0
    N: int = 0                  # decode: concurrent sequences
    steps: int = 0              # decode: distinct steps
    state_std: float = 0.0      # decode: state distribution

    @property
    def seed(self) -> int:
        return 1000 + self.index

    @property
    def torch_dtype(self):
        return torch.float32 if self.io == "fp32" else torch.bfloat16


WORKLOADS = {
    "tiny": Workload("tiny", 0, H=2, dk=64, dv=64, io="fp32", B=1, T=256, chunk=64),
    "prefill": Workload("prefill", 1, H=16, dk=128, dv=128, B=4, T=2048, chunk=128,
                        init_std=0.02),
    "decode": Workload("decode", 2, H=16, dk=128, dv=128, N=1280, steps=64, state_std=0.1),
    "varlen": Workload("varlen", 3, H=32, dk=128, dv=128, g_mu=4.0, chunk=128,
                       init_std=0.05, nseq=16, len_lo=512, len_hi=16384),
    "vector": Workload("vector", 4, H=16, dk=128, dv=128, gate="vector", g_mu=2.0,
                       g_div=4.0, B=8, T=4096, chunk=128),
    "laplace": Workload("laplace", 5, H=16, dk=96, dv=192, decay="schedule", B=8, T=2048,
                        chunk=128, init_std=0.02),
}


def _normal(gen, shape, std=1.0):
    x = torch.randn(*shape, generator=gen, dtype=torch.float32)
    return x if std == 1.0 else x * std


def _gate(gen, shape, w: Workload):
    if w.decay == "schedule":
        # fixed per-head log-decay: half-lives spread geometrically over 1 .. 2048
        # tokens across the heads, the same value for every token
        h = torch.arange(w.H, dtype=torch.float64)
        half_life = 2048.0 ** (h / max(w.H - 1, 1))
        g_h = (-torch.log(torch.tensor(2.0, dtype=torch.float64)) / half_life).float()
        shape_h = [1] * (len(shape) - 1) + [w.H] if w.gate == "scalar" else \
            [1] * (len(shape) - 2) + [w.H, 1]
        return g_h.reshape(shape_h).expand(shape).contiguous()
    x = _normal(gen, shape) + w.g_mu
    return (F.logsigmoid(x) / w.g_div).contiguous()


def _qkv(gen, lead, w: Workload):
    q = _normal(gen, (*lead, w.H, w.dk))
    k = _normal(gen, (*lead, w.H, w.dk))
    k = k / k.norm(dim=-1, keepdim=True)
    v = _normal(gen, (*lead, w.H, w.dv))
    dt = w.torch_dtype
    return q.to(dt).contiguous(), k.to(dt).contiguous(), v.to(dt).contiguous()


def prefill_inputs(w: Workload, seed: Optional[int] = None, **override):
    """Dense or packed prefill inputs for workload ``w`` (sizes may be overridden).

    Returns a dict with ``q, k, v`` ([B, T, H, d], or [1, R, H, d] when packed),
    ``g`` (fp32, [.., H] or [.., H, dk]), ``init_state`` (fp32 [B, H, dk, dv] or
    None), ``cu_seqlens`` (int32 [B+1] or None), ``scale`` and ``chunk``.
    Override keys: any Workload field, plus ``lengths`` (explicit packed
    sequence lengths).
    """
    lengths = override.pop("lengths", None)
    if override:
        w = dataclasses.replace(w, **override)
    gen = torch.Generator().manual_seed(w.seed if seed is None else seed)
    packed = lengths is not None or w.nseq > 0
    if packed:
        if lengths is None:
            lengths = torch.randint(w.len_lo, w.len_hi + 1, (w.nseq,), generator=gen)
        lengths = torch.as_tensor(lengths, dtype=torch.int64)
        cu = torch.zeros(len(lengths) + 1, dtype=torch.int64)
        cu[1:] = torch.cumsum(lengths, 0)
        cu_seqlens = cu.to(torch.int32)
        B, lead = len(lengths), (1, int(cu[-1]))
    else:
        cu_seqlens = None
        B, lead = w.B, (w.B, w.T)
    q, k, v = _qkv(gen, lead, w)
    gshape = (*lead, w.H) if w.gate == "scalar" else (*lead, w.H, w.dk)
    g = _gate(gen, gshape, w)
    init = _normal(gen, (B, w.H, w.dk, w.dv), w.init_std) if w.init_std > 0 else None
    return dict(q=q, k=k, v=v, g=g, init_state=init, cu_seqlens=cu_seqlens,
                scale=w.dk ** -0.5, chunk=w.chunk, workload=w)


def mixer_inputs(w: Workload, lead, seed: Optional[int] = None, tiers: int = 4, **override):
    """Synthetic weights and gate stream for the mixer's steps after the readout:
    ``aug`` fp32 [H, dk] ~ N(0, 0.5) (the self-augmentation balance), ``norm_w``
    fp32 [H, dv] ~ 1 + N(0, 0.1) with the heads split into ``tiers`` equal runs
    that share one row (the head RMSNorm per decay tier), ``z`` [*lead, H, dv]
    ~ N(0, 1) in the I/O dtype (the output gate stream), ``eps`` 1e-6."""
    if override:
        w = dataclasses.replace(w, **override)
    gen = torch.Generator().manual_seed((w.seed if seed is None else seed) + 7)
    aug = _normal(gen, (w.H, w.dk), 0.5)
    per = -(-w.H // tiers)
    rows = 1.0 + _normal(gen, (tiers, w.dv), 0.1)
    norm_w = rows[torch.arange(w.H) // per].contiguous()
    z = _normal(gen, (*lead, w.H, w.dv)).to(w.torch_dtype).contiguous()
    return dict(aug=aug, norm_w=norm_w, eps=1e-6, z=z)


def grad_inputs(x, seed: Optional[int] = None, d_final_std: float = 0.1):
    """Upstream gradients for a backward call on prefill inputs ``x`` (a dict
    from ``prefill_inputs``): ``d_out`` ~ N(0, 1) shaped like v in the I/O
    dtype, and ``d_final_state`` ~ N(0, d_final_std) fp32 [B, H, dk, dv]
    (None when ``d_final_std`` is 0)."""
    w = x["workload"]
    gen = torch.Generator().manual_seed((w.seed if seed is None else seed) + 13)
    d_out = _normal(gen, tuple(x["v"].shape)).to(x["v"].dtype).contiguous()
    B = x["init_state"].shape[0] if x["init_state"] is not None else (
        len(x["cu_seqlens"]) - 1 if x["cu_seqlens"] is not None else x["q"].shape[0])
    H, dk, dv = x["q"].shape[-2], x["q"].shape[-1], x["v"].shape[-1]
    d_final = _normal(gen, (B, H, dk, dv), d_final_std) if d_final_std > 0 else None
    return dict(d_out=d_out, d_final_state=d_final)


def decode_inputs(w: Workload, seed: Optional[int] = None, **override):
    """Decode inputs: ``state [N, H, dk, dv]`` fp32 and per-step lists of
    ``q, k [N, H, dk]``, ``v [N, H, dv]`` (I/O dtype) and ``g`` ([N, H] or
    [N, H, dk], fp32), stacked along a leading step axis."""
    if override:
        w = dataclasses.replace(w, **override)
    gen = torch.Generator().manual_seed(w.seed if seed is None else seed)
    state = _normal(gen, (w.N, w.H, w.dk, w.dv), w.state_std).contiguous()
    q, k, v = _qkv(gen, (w.steps, w.N), w)
    gshape = (w.steps, w.N, w.H) if w.gate == "scalar" else (w.steps, w.N, w.H, w.dk)
    g = _gate(gen, gshape, w)
    return dict(state=state, q=q, k=k, v=v, g=g, scale=w.dk ** -0.5, workload=w)
