"""Decode-width buckets: CUDA graphs of the slot-indexed decode step.

Serving decodes one token for every live sequence at each step, and the number
of live sequences changes as requests arrive and finish.  Launching the decode
kernel through Python costs microseconds per step; a CUDA graph replays it for
almost nothing, but a graph is fixed to its buffers and sizes.  So the step is
captured once per bucket width W (by default the powers of two up to the
largest width), over static buffers, with the states kept in a pool of pages
addressed by slot (``gla_decode_step_slots``): a batch of n <= W live rows is
copied into the first n rows of the static buffers, the remaining W - n rows
get slot -1 (rows the kernel skips), and the graph of width W is replayed.
Rows past the widest batch since the last clean-up already hold -1, so the
padding costs a fill launch only on a step whose batch is narrower than the
previous one.

The state pool, the dtypes and the head sizes are fixed at construction.  The
fast path is ``buffers(n)`` (views of the static inputs, for the producer of
q, k, v, g and slots to write into) followed by ``run(n)``; ``step`` copies
given tensors in first (five extra copies per step).  The output is a view of
the static output buffer, valid until the next step.
"""
from __future__ import annotations

from typing import Optional, Sequence

import torch

from . import decode_step


def default_buckets(max_width: int):
    """Powers of two up to ``max_width``, plus ``max_width`` itself."""
    if max_width < 1:
        raise ValueError("max_width must be >= 1")
    out, w = [], 1
    while w < max_width:
        out.append(w)
        w *= 2
    out.append(max_width)
    return out


def pick_bucket(buckets: Sequence[int], n: int) -> int:
    """The smallest bucket width that holds ``n`` rows."""
    for w in sorted(buckets):
        if w >= n:
            return w
    raise ValueError(f"{n} rows exceed the widest bucket ({max(buckets)})")


class DecodeGraphs:
    """One captured decode step per bucket width over a fixed state pool.

    ``state_pool``: fp32 [num_slots, H, dk, dv] on the GPU (updated in place).
    ``dtype``: dtype of q, k, v (bf16 or fp32); ``vector_gate``: g is
    [n, H, dk] instead of [n, H]; ``out_dtype``: as for ``decode_step``.
    """

    def __init__(self, state_pool: torch.Tensor, max_width: int,
                 buckets: Optional[Sequence[int]] = None, dtype=torch.bfloat16,
                 vector_gate: bool = False, scale: Optional[float] = None, out_dtype=None):
        if not (state_pool.is_cuda and state_pool.dtype == torch.float32 and
                state_pool.dim() == 4 and state_pool.is_contiguous()):
            raise ValueError("state_pool must be a contiguous fp32 CUDA tensor "
                             "[num_slots, H, dk, dv]")
        self.pool = state_pool
        _, H, dk, dv = state_pool.shape
        self.buckets = sorted(set(buckets or default_buckets(max_width)))
        if self.buckets[0] < 1:
            raise ValueError("bucket widths must be >= 1")
        W = self.buckets[-1]
        dev = state_pool.device
        self.scale = dk ** -0.5 if scale is None else scale
        self.q = torch.zeros(W, H, dk, dtype=dtype, device=dev)
        self.k = torch.zeros_like(self.q)
        self.v = torch.zeros(W, H, dv, dtype=dtype, device=dev)
        self.g = torch.zeros((W, H, dk) if vector_gate else (W, H), dtype=torch.float32,
                             device=dev)
        self.slots = torch.full((W,), -1, dtype=torch.int32, device=dev)
        self._dirty = 0  # slots rows at or past this index hold -1
        self.out = torch.zeros(W, H, dv, dtype=out_dtype or dtype, device=dev)
        self.graphs = {}
        side = torch.cuda.Stream(device=dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):
            # one eager call first (every slot -1: nothing changes) so that the
            # library's one-time setup happens outside the capture
            for w in self.buckets:
                self._launch(w)
        torch.cuda.current_stream(dev).wait_stream(side)
        torch.cuda.synchronize(dev)
        for w in self.buckets:
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=side):
                self._launch(w)
            self.graphs[w] = graph
        torch.cuda.synchronize(dev)

    def _launch(self, w: int):
        decode_step(self.q[:w], self.k[:w], self.v[:w], self.g[:w], self.pool,
                    scale=self.scale, out=self.out[:w], slots=self.slots[:w])

    def buffers(self, n: int):
        """Views of the first ``n`` rows of the static inputs (q, k, v, g, slots)
        for the next ``run(n)``."""
        pick_bucket(self.buckets, n)
        self._dirty = max(self._dirty, n)  # the caller writes slots rows [0, n)
        return {"q": self.q[:n], "k": self.k[:n], "v": self.v[:n], "g": self.g[:n],
                "slots": self.slots[:n]}

    def run(self, n: int):
        """Decode one token for the ``n`` rows already in ``buffers(n)`` (their
        slots distinct pool pages): pad to the bucket with slot -1 rows and
        replay its graph.  Returns out [n, H, dv]."""
        w = pick_bucket(self.buckets, n)
        if self._dirty > n:  # a wider batch ran before: its extra rows back to -1
            self.slots[n:self._dirty].fill_(-1)
        self._dirty = n
        self.graphs[w].replay()
        return self.out[:n]

    def step(self, q, k, v, g, slots):
        """``run`` after copying q, k, v, g and slots (int32 [n]) into the
        static buffers."""
        n = q.shape[0]
        b = self.buffers(n)
        for name, t in (("q", q), ("k", k), ("v", v), ("g", g), ("slots", slots)):
            b[name].copy_(t, non_blocking=True)
        return self.run(n)
