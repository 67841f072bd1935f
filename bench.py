#!/usr/bin/env python
"""Throughput of the GLA hot path on GB300: chunked prefill and decode.

One bench step is one pass of the serving hot path over synthetic inputs:

* four ``gla_chunk_fwd`` calls over the prefill workload -- B=4 sequences of
  T=2048 tokens, H=16, dk=dv=128, chunk 128, bf16 I/O, fp32 initial and final
  states, one call per input set -- replayed from one CUDA graph, whose
  tokens/s is the headline ``value`` (the same calls launched one by one from
  Python are timed too: ``prefill.ms_per_call_eager_median``);
* 64 consecutive ``gla_decode_step`` calls over the decode workload -- N=1280
  concurrent sequences, H=16, dk=dv=128, fp32 states updated in place --
  reported as ``decode`` (sequence-steps/s).

Prefill and decode are timed separately with CUDA events on the stream that
launches them.  Four prefill input sets (572 MB together, L2 is 129 MB) are
rotated so no step reads its inputs from L2; the decode state alone is 1.34 GB.
``roofline`` is the dominant kernel's (the decode step: 64 launches per
step against 4 prefill calls) achieved HBM bandwidth against the measured copy bandwidth;
``prefill.roofline`` is the prefill kernel's.

After the step (outside its time), side measurements are added to the line:
the other prefill workloads, decode-width graph buckets, the mixer epilogue,
and ``backward`` -- the chunked backward (gla_chunk_bwd) on the prefill
workload's sizes, with its roofline against the CUDA cores' fp32 FMA peak.

``--impl reference`` times the fp64 CPU oracle (the reference for parity, a
deliberately plain program) on the same prefill workload, whole (about 0.2 s
per step on 16 host cores, so K steps end within seconds).

Multi-GPU (torchrun): every rank runs its own replica (the (sequence, head)
units are independent, so there is no data-path collective); the process
group is used only for the barrier and the max-over-ranks time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import gla_inputs  # noqa: E402

METRIC = "GLA prefill tokens/s & decode seq-steps/s on 1 GB300; % of tensor/HBM roofline"
N_SETS = 4
DECODE_STEPS = 64
PROFILE_DIR = os.path.join(ROOT, "profiles")


# ----------------------------------------------------------------- workloads
def prefill_bytes(w, B, T, rows=None) -> int:
    """Algorithmic HBM bytes of one prefill call over B sequences (B * T token
    rows, or ``rows`` when packed): read q, k, v (bf16) and g (fp32, one per
    head or per key channel), the initial state (fp32, when the workload has
    one); write out (bf16) and the final state (fp32)."""
    rows = B * T if rows is None else rows
    g_per_head = w.dk if w.gate == "vector" else 1
    io = 2 * rows * w.H * (2 * w.dk + w.dv) + 4 * rows * w.H * g_per_head + 2 * rows * w.H * w.dv
    n_states = 2 if (w.init_std > 0 or w.name == "prefill") else 1
    states = n_states * 4 * B * w.H * w.dk * w.dv
    return io + states


def prefill_flops(w, B, T, rows=None) -> int:
    """Tensor-core flops of the chunked form as computed (full C x C tiles):
    per token and head 2 * (C * (dk + dv) + 2 * dk * dv)."""
    rows = B * T if rows is None else rows
    return 2 * (w.chunk * (w.dk + w.dv) + 2 * w.dk * w.dv) * rows * w.H


def prefill_config(world: int) -> dict:
    """The ``config`` of both arms' JSON lines: the prefill workload the
    headline value is measured on."""
    wp = gla_inputs.WORKLOADS["prefill"]
    pb = prefill_bytes(wp, wp.B, wp.T)
    return {
        "workload": f"simple-GLA chunked prefill B={wp.B} H={wp.H} T={wp.T} dk=dv={wp.dk} "
                    f"chunk={wp.chunk} bf16 I/O, fp32 states",
        "global_batch": wp.B * world, "seq_len": wp.T, "heads": wp.H, "dk": wp.dk,
        "dv": wp.dv, "chunk": wp.chunk, "parallelism": f"replicas x{world}",
        "l2": f"{N_SETS} rotating prefill input sets "
              f"({N_SETS * pb / 1e6:.0f} MB > 129 MB L2); decode state 1.34 GB",
    }


# fp32 FMA peak of the CUDA cores: 152 SMs x 128 fp32 lanes x 2 flops per FMA at
# the maximum SM clock (2070 MHz); the backward is bound by these units.
FP32_LANES = 152 * 128
SM_MAX_MHZ = 2070.0


def fp32_peak_tflops(sm_mhz: float = SM_MAX_MHZ) -> float:
    return FP32_LANES * 2 * sm_mhz * 1e6 / 1e12


BWD_CHUNK = 64


def backward_flops(w, B, T, chunk=BWD_CHUNK) -> int:
    """Algorithmic flops of the chunked backward (the causal triangles counted
    as halves): per token and head, the five C x C x d products dO V^T, P K,
    P^T Q, Q K^T, M^T dO at C/2 MACs per output column each -- (C/2)(2 dv + 3 dk)
    -- plus the three inter-chunk readouts (dq, dk, dv) and the two state steps
    (S forward, the carried gradient backward), dk dv MACs each: 2 flops per
    MAC.  Chunks of 64 on the CUDA cores, 128 on the tensor cores."""
    macs = (chunk // 2) * (2 * w.dv + 3 * w.dk) + 5 * w.dk * w.dv
    return 2 * macs * B * T * w.H


def backward_bytes(w, B, T) -> int:
    """Algorithmic HBM bytes of one backward call: read q, k, v, d_out (bf16)
    and g (fp32), the initial state and the final state's gradient (fp32);
    write dq, dk, dv (bf16), dg (fp32) and the initial state's gradient."""
    tok = B * T * w.H
    g_per = w.dk if w.gate == "vector" else 1
    io = tok * (2 * (2 * w.dk + 2 * w.dv) + 4 * g_per + 2 * (2 * w.dk + w.dv) + 4 * g_per)
    return io + 3 * 4 * B * w.H * w.dk * w.dv


def decode_bytes(w) -> int:
    """Algorithmic HBM bytes of one decode step: fp32 state read + write, q, k,
    v (bf16), g (fp32) read, out (bf16) write."""
    units = w.N * w.H
    return units * (8 * w.dk * w.dv + 2 * (2 * w.dk + w.dv) + 4 + 2 * w.dv)


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d["hbm_gbs"], d["bf16_tflops"], d.get("bf16_tflops_sustained"), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


def kernel_source_hash(name: str) -> str:
    path = os.path.join(ROOT, "gated_linear_attention_gla_gb300", "csrc", name)
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def profiled_traffic(summary: str, source: str):
    """DRAM bytes per launch recorded beside a committed ncu summary (the
    ``.json`` of the same name: ``traffic_bytes_per_launch`` and the kernel
    source's hash), or None when it is missing or the kernel source changed
    since the capture."""
    path = os.path.join(PROFILE_DIR, os.path.splitext(summary)[0] + ".json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    if rec.get("kernel_source_sha256_16") != kernel_source_hash(source):
        return None
    return float(rec["traffic_bytes_per_launch"])


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 100 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,utilization.gpu,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.gpu_index), "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        time.sleep(0.2)
        self.proc.terminate()
        self.proc.wait(timeout=10)
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append(dict(sm=float(parts[1]), smmax=float(parts[2]),
                                 power=float(parts[3]), util=float(parts[4]),
                                 reasons=[n for n, v in zip(
                                     ("hw_slowdown", "hw_thermal_slowdown",
                                      "sw_thermal_slowdown", "sw_power_cap"), parts[5:9])
                                     if v.lower().startswith("active")]))
            except ValueError:
                continue
        os.unlink(self.path)
        loaded = [r for r in rows if r["util"] > 0] or rows
        if not loaded:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        reasons = sorted({x for r in loaded for x in r["reasons"]})
        return {"sm_mhz": statistics.median(r["sm"] for r in loaded),
                "sm_max_mhz": max(r["smmax"] for r in loaded), "reasons": reasons,
                "samples": len(loaded), "power_w_max": max(r["power"] for r in loaded)}


# --------------------------------------------------------------- distributed
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def dist_init(world, local, backend="nccl"):
    if world > 1:
        import torch.distributed as dist
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    backend = dist.get_backend()
    dev = torch.device("cuda", torch.cuda.current_device()) if backend == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    backend = dist.get_backend()
    dev = torch.device("cuda", torch.cuda.current_device()) if backend == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ------------------------------------------------------------- CPU baseline
def cpu_baseline(budget_s: float = 10.0):
    """The fp64 oracle on this host's cores, as it stands: the whole prefill
    workload repeated until ``budget_s`` has passed (at least once), and one
    decode step over all 1280 sequences repeated likewise."""
    import oracle
    wp = gla_inputs.WORKLOADS["prefill"]
    x = gla_inputs.prefill_inputs(wp)
    cores = oracle.max_threads()
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle.recurrent(x["q"], x["k"], x["v"], x["g"], x["scale"], init_state=x["init_state"])
        reps += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    prefill = dict(value=wp.B * wp.T * reps / dt, unit="tokens/s", cores=cores, kind="oracle",
                   sample=f"full prefill workload (B={wp.B}, T={wp.T}, H={wp.H}, d={wp.dk}) "
                          f"x {reps}, fp64 token-by-token recurrence, {dt:.1f} s")
    # the same program on one core: the first sequence of the workload (all heads)
    one = {n: x[n][:1].contiguous() for n in ("q", "k", "v", "g", "init_state")}
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle.recurrent(one["q"], one["k"], one["v"], one["g"], x["scale"],
                         init_state=one["init_state"], nthreads=1)
        reps += 1
        if time.perf_counter() - t0 >= budget_s / 3:
            break
    dt1 = time.perf_counter() - t0
    prefill["one_core"] = dict(value=wp.T * reps / dt1, unit="tokens/s", cores=1,
                               sample=f"one sequence (T={wp.T}, H={wp.H}) x {reps}, "
                                      f"{dt1:.1f} s")
    wd = gla_inputs.WORKLOADS["decode"]
    d = gla_inputs.decode_inputs(wd, steps=1)
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle.decode_step(d["q"][0], d["k"][0], d["v"][0], d["g"][0], d["scale"], d["state"])
        reps += 1
        if time.perf_counter() - t0 >= budget_s / 2:
            break
    dt = time.perf_counter() - t0
    decode = dict(value=wd.N * reps / dt, unit="seq*steps/s", cores=cores, kind="oracle",
                  sample=f"one decode step over N={wd.N}, H={wd.H} x {reps}, fp64, {dt:.1f} s")
    return prefill, decode


# ------------------------------------------------------------------ GPU arm
# the other prefill workloads: their kernel and the profile that records its traffic
SIDE_WORKLOADS = {
    "vector": ("chunk_tc_vec_kernel", "chunk_tc_vec_kernel.vector_b8_h16_t4096.md",
               "gla_chunk_tc_vec.cu"),
    "varlen": ("chunk_tc_kernel", None, "gla_chunk_tc.cu"),
    "laplace": ("chunk_tc_kernel", "chunk_tc_kernel.laplace_b8_h16_t2048.md", "gla_chunk_tc.cu"),
}


def time_side_workloads(gla, dev, hbm, peak_kind, reps=10, warmup=3):
    """The vector-gate and packed varlen prefill workloads, each timed alone
    (CUDA events around `reps` calls after `warmup`), with their HBM roofline."""
    out = {}
    stream = torch.cuda.current_stream()
    for name, (kernel, profile, source) in SIDE_WORKLOADS.items():
        w = gla_inputs.WORKLOADS[name]
        x = gla_inputs.prefill_inputs(w)
        q, k, v, g = (x[n].to(dev) for n in ("q", "k", "v", "g"))
        s0 = x["init_state"].to(dev) if x["init_state"] is not None else None
        cu = x["cu_seqlens"].to(dev) if x["cu_seqlens"] is not None else None
        nseq = (len(x["cu_seqlens"]) - 1) if cu is not None else w.B
        rows = q.numel() // (w.H * w.dk)
        o = torch.empty(v.shape, dtype=torch.bfloat16, device=dev)
        fin = torch.empty(nseq, w.H, w.dk, w.dv, dtype=torch.float32, device=dev)

        def call():
            gla.chunk_fwd(q, k, v, g, scale=x["scale"], init_state=s0, cu_seqlens=cu,
                          chunk=w.chunk, out=o, final_state=fin)
        for _ in range(warmup):
            call()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            call()
        b.record(stream)
        torch.cuda.synchronize()
        gla.status_sync()
        sec = a.elapsed_time(b) / 1e3 / reps
        nbytes = prefill_bytes(w, nseq, 0, rows=rows)
        gbs = nbytes / sec / 1e9
        desc = (f"{nseq} packed sequences ({rows} tokens), " if cu is not None else
                f"B={w.B} T={w.T} ") + (f"H={w.H} dk={w.dk} dv={w.dv} chunk={w.chunk} "
                                        f"{w.gate} gate ({w.decay} decay), bf16 I/O")
        out[name] = {
            "workload": desc, "ms_per_call": sec * 1e3, "tokens_per_call": rows,
            "value": rows / sec, "unit": "tokens/s", "calls": reps,
            "roofline": {"kernel": kernel, "bound": "hbm", "achieved": gbs, "peak": hbm,
                         "unit": "GB/s", "frac": gbs / hbm, "peak_kind": peak_kind,
                         "traffic": profiled_traffic(profile, source) if profile else None,
                         "algorithmic_bytes_per_launch": nbytes}}
        del q, k, v, g, s0, cu, o, fin
        torch.cuda.empty_cache()
    return out


def time_decode_graphs(gla, dev, width=64, steps=200):
    """A small decode batch (`width` sequences, the decode workload's heads and
    head sizes, states in a pool addressed by slot): `steps` consecutive steps
    launched one by one from Python, then replayed from the captured CUDA graph
    of that width (inputs in the graph's buffers).  At this size launch
    overhead, not HBM, sets the step time (the 67 MB pool stays in L2)."""
    from gated_linear_attention_gla_gb300.serving import DecodeGraphs
    w = gla_inputs.WORKLOADS["decode"]
    d = gla_inputs.decode_inputs(w, steps=1, N=width)
    q, k, v, g = (d[n][0].to(dev) for n in ("q", "k", "v", "g"))
    pool = d["state"].to(dev).contiguous()
    slots = torch.arange(width, dtype=torch.int32, device=dev)
    out = torch.empty(width, w.H, w.dv, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def timed(fn):
        for _ in range(5):
            fn()
        torch.cuda.synchronize()
        a.record(stream)
        for _ in range(steps):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) * 1e3 / steps
    eager = timed(lambda: gla.decode_step(q, k, v, g, pool, scale=d["scale"], out=out,
                                          slots=slots))
    graphs = DecodeGraphs(pool, max_width=width)
    buf = graphs.buffers(width)  # the inputs written once, where a producer would write them
    for name, t in (("q", q), ("k", k), ("v", v), ("g", g), ("slots", slots)):
        buf[name].copy_(t)
    graph = timed(lambda: graphs.run(width))
    gla.status_sync()
    nbytes = width * w.H * (8 * w.dk * w.dv + 2 * (2 * w.dk + w.dv) + 4 + 2 * w.dv)
    return {"workload": f"decode step N={width} H={w.H} dk=dv={w.dk}, states in a slot pool",
            "steps": steps, "eager_us_per_step": eager, "graph_us_per_step": graph,
            "algorithmic_bytes_per_step": nbytes, "graph_gbs": nbytes / graph / 1e3}


def time_mixer(gla, dev, hbm, reps=20, warmup=3):
    """The mixer's steps after the readout: the prefill workload with and without
    the epilogue pass (gla_mixer_epilogue over its output), the per-key-channel
    workload with and without the steps (fused into its kernel), and the decode
    workload's step with and without the fused epilogue; each timed alone."""
    stream = torch.cuda.current_stream()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def timed(fn):
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        a.record(stream)
        for _ in range(reps):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / reps
    res = {}
    w = gla_inputs.WORKLOADS["prefill"]
    x = gla_inputs.prefill_inputs(w)
    q, k, v, g, s0 = (x[n].to(dev) for n in ("q", "k", "v", "g", "init_state"))
    m = gla_inputs.mixer_inputs(w, q.shape[:-2])
    mix = {n: (t.to(dev) if torch.is_tensor(t) else t) for n, t in m.items()}
    out = torch.empty(v.shape, dtype=torch.bfloat16, device=dev)
    fin = torch.empty_like(s0)
    kw = dict(scale=x["scale"], init_state=s0, chunk=w.chunk, out=out, final_state=fin)
    plain = timed(lambda: gla.chunk_fwd(q, k, v, g, **kw))
    fused = timed(lambda: gla.chunk_fwd(q, k, v, g, mixer=mix, **kw))
    units = w.B * w.T * w.H
    # epilogue bytes: read o, q, k, v, z (bf16), the weights; write o
    epi_bytes = units * 2 * (w.dv + 2 * w.dk + w.dv + w.dv + w.dv)
    res["prefill"] = {"workload": f"prefill B={w.B} T={w.T} H={w.H} d={w.dk}, epilogue pass "
                                  f"over the bf16 output",
                      "ms_plain": plain, "ms_with_epilogue": fused, "ratio": fused / plain,
                      "epilogue_ms": fused - plain, "epilogue_bytes": epi_bytes,
                      "epilogue_frac_of_hbm": epi_bytes / ((fused - plain) / 1e3) / 1e9 / hbm}
    # the per-key-channel workload: the kernel applies the steps itself
    wv = gla_inputs.WORKLOADS["vector"]
    xv = gla_inputs.prefill_inputs(wv)
    qv, kv, vv, gv = (xv[n].to(dev) for n in ("q", "k", "v", "g"))
    mv = gla_inputs.mixer_inputs(wv, qv.shape[:-2])
    mixv = {n: (t.to(dev) if torch.is_tensor(t) else t) for n, t in mv.items()}
    outv = torch.empty(vv.shape, dtype=torch.bfloat16, device=dev)
    kwv = dict(scale=xv["scale"], chunk=wv.chunk, out=outv, output_final_state=False)
    plain_v = timed(lambda: gla.chunk_fwd(qv, kv, vv, gv, **kwv))
    fused_v = timed(lambda: gla.chunk_fwd(qv, kv, vv, gv, mixer=mixv, **kwv))
    res["prefill_vector"] = {
        "workload": f"per-key-channel prefill B={wv.B} T={wv.T} H={wv.H} d={wv.dk}, the "
                    f"steps fused into the kernel (augmentation through P', RMSNorm and gate "
                    f"before the store)",
        "ms_plain": plain_v, "ms_fused": fused_v, "ratio": fused_v / plain_v}
    del qv, kv, vv, gv, outv
    wd = gla_inputs.WORKLOADS["decode"]
    d = gla_inputs.decode_inputs(wd, steps=1)
    dq, dk_, dv_, dg = (d[n][0].to(dev) for n in ("q", "k", "v", "g"))
    st = d["state"].to(dev)
    md = gla_inputs.mixer_inputs(wd, (wd.N,))
    dmix = {n: (t.to(dev) if torch.is_tensor(t) else t) for n, t in md.items()}
    dout = torch.empty(wd.N, wd.H, wd.dv, dtype=torch.bfloat16, device=dev)
    p_ms = timed(lambda: gla.decode_step(dq, dk_, dv_, dg, st, scale=d["scale"], out=dout))
    f_ms = timed(lambda: gla.decode_step(dq, dk_, dv_, dg, st, scale=d["scale"], out=dout,
                                         mixer=dmix))
    res["decode"] = {"workload": f"decode step N={wd.N} H={wd.H} d={wd.dk}, fused epilogue",
                     "ms_plain": p_ms, "ms_fused": f_ms,
                     "fused_overhead": f_ms / p_ms - 1.0}
    gla.status_sync()
    return res


def time_backward(gla, dev, reps=5, warmup=3):
    """The chunked backward (gla_chunk_bwd: dq, dk, dv, dg, d_init) on the
    prefill workload's sizes, for the per-head gate and for the per-key-channel
    gate; timed alone with CUDA events on the launching stream."""
    stream = torch.cuda.current_stream()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    res = []
    w0 = gla_inputs.WORKLOADS["prefill"]
    hbm, bf16_peak, _, kind = peaks()
    from gated_linear_attention_gla_gb300 import _binding
    vec = dict(gate="vector", g_mu=2.0, g_div=4.0)
    for gate, over, tc in (("per-head", {}, True), ("per-head", {}, False),
                           ("per-key-channel", vec, True), ("per-key-channel", vec, False)):
        w = gla_inputs.dataclasses.replace(w0, **over)
        x = gla_inputs.prefill_inputs(w)
        gr = gla_inputs.grad_inputs(x)
        args = [x[n].to(dev) for n in ("q", "k", "v", "g")] + [gr["d_out"].to(dev)]
        ws = None
        if tc:
            flags = _binding.GLA_FLAG_VECTOR_GATE if w.gate == "vector" else 0
            n = _binding.chunk_bwd_workspace_size(w.B, w.H, w.T, w.dk, w.dv, False, flags)
            ws = torch.empty(n, dtype=torch.uint8, device=dev)
        kw = dict(scale=x["scale"], init_state=x["init_state"].to(dev),
                  d_final_state=gr["d_final_state"].to(dev), tensor_cores=tc, workspace=ws)
        for _ in range(warmup):
            gla.chunk_bwd(*args, **kw)
        torch.cuda.synchronize()
        a.record(stream)
        for _ in range(reps):
            gla.chunk_bwd(*args, **kw)
        b.record(stream)
        torch.cuda.synchronize()
        gla.status_sync()
        ms = a.elapsed_time(b) / reps
        sec = ms / 1e3
        entry = {
            "workload": f"chunked backward, {gate} gate, B={w.B} T={w.T} H={w.H} "
                        f"dk=dv={w.dk}, bf16 q/k/v/d_out, bf16 gradients, fp32 dg and d_init",
            "path": ("CUDA cores (fp32)" if not tc else
                     "tensor cores (3 prefill runs)" if w.gate != "vector" else
                     "dv on the tensor cores (reversed prefill), dq and dk on the CUDA cores"),
            "ms": ms, "tokens_per_s": w.B * w.T / sec}
        if tc and w.gate != "vector":
            nbytes = backward_bytes(w, w.B, w.T)
            flops = backward_flops(w, w.B, w.T, chunk=128)
            entry["roofline"] = {
                "bound": "hbm", "achieved": nbytes / sec / 1e9, "peak": hbm, "unit": "GB/s",
                "frac": nbytes / sec / 1e9 / hbm, "peak_kind": kind,
                "algorithmic_bytes": nbytes,
                "tensor": {"achieved_tflops": flops / sec / 1e12, "peak_tflops": bf16_peak,
                           "frac": flops / sec / 1e12 / bf16_peak, "algorithmic_flops": flops},
                "workspace_bytes": ws.numel()}
            entry["launches"] = 5  # prepare, 3 x prefill, tail (after a driver memset of dg)
        elif tc:
            # mostly the CUDA-core dq and dk kernels: their fp32 roofline
            flops = backward_flops(w, w.B, w.T)
            peak = fp32_peak_tflops()
            entry["roofline"] = {
                "bound": "alu", "achieved": flops / sec / 1e12, "peak": peak,
                "unit": "TFLOP/s", "frac": flops / sec / 1e12 / peak,
                "peak_source": "fp32 FMA lanes x 2 x max SM clock (derived)",
                "algorithmic_flops": flops, "workspace_bytes": ws.numel()}
            entry["launches"] = 4  # prepare, per-key-channel prefill, dq, dk
        else:
            flops = backward_flops(w, w.B, w.T)
            peak = fp32_peak_tflops()
            entry["roofline"] = {
                "bound": "alu", "achieved": flops / sec / 1e12, "peak": peak,
                "unit": "TFLOP/s", "frac": flops / sec / 1e12 / peak,
                "peak_source": "fp32 FMA lanes x 2 x max SM clock (derived)",
                "algorithmic_flops": flops}
            # dq, dk, dv (+ the dg scan for the per-head gate, after a driver memset
            # of dg that is not counted)
            entry["launches"] = 3 if gate == "per-key-channel" else 4
        res.append(entry)
    return res


def run_gla(args, world, rank, local):
    import gated_linear_attention_gla_gb300 as gla
    from gated_linear_attention_gla_gb300 import build as glabuild

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    glabuild.build()
    gla.lib()  # loud failure if the library is missing

    wp, wd = gla_inputs.WORKLOADS["prefill"], gla_inputs.WORKLOADS["decode"]
    B, T, H = wp.B, wp.T, wp.H
    sets = []
    for i in range(N_SETS):
        x = gla_inputs.prefill_inputs(wp, seed=wp.seed + 7919 * i + 104729 * rank)
        sets.append({n: (x[n].to(dev) if x[n] is not None else None)
                     for n in ("q", "k", "v", "g", "init_state")})
    scale = wp.dk ** -0.5
    outs = [torch.empty(B, T, H, wp.dv, dtype=torch.bfloat16, device=dev) for _ in range(N_SETS)]
    finals = [torch.empty(B, H, wp.dk, wp.dv, dtype=torch.float32, device=dev)
              for _ in range(N_SETS)]
    d = gla_inputs.decode_inputs(wd, steps=DECODE_STEPS, seed=wd.seed + 104729 * rank)
    d_state = d["state"].to(dev)
    d_q, d_k, d_v, d_g = (d[n].to(dev) for n in ("q", "k", "v", "g"))
    d_out = torch.empty(DECODE_STEPS, wd.N, wd.H, wd.dv, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream()

    def prefill(i):
        s = sets[i % N_SETS]
        gla.chunk_fwd(s["q"], s["k"], s["v"], s["g"], scale=scale, init_state=s["init_state"],
                      chunk=wp.chunk, out=outs[i % N_SETS], final_state=finals[i % N_SETS])

    def decode64():
        for t in range(DECODE_STEPS):
            gla.decode_step(d_q[t], d_k[t], d_v[t], d_g[t], d_state, scale=wd.dk ** -0.5,
                            out=d_out[t])

    for i in range(args.warmup):
        prefill(i)
        decode64()
    gla.status_sync()
    # The step's prefill is the N_SETS rotating calls, replayed from one CUDA
    # graph: the same launches and the same work, without the host's per-call
    # launch gaps (the eager per-call time is reported beside it).
    g_pre = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream(device=dev)
    cap.wait_stream(stream)
    with torch.cuda.stream(cap):
        for i in range(N_SETS):
            prefill(i)
    cap.synchronize()
    with torch.cuda.graph(g_pre, stream=cap):
        for i in range(N_SETS):
            prefill(i)
    torch.cuda.synchronize()
    for _ in range(2):
        g_pre.replay()
    torch.cuda.synchronize()

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    sampler = ClockSampler(local if world > 1 else dev.index)
    sampler.start()
    barrier(world)
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    for i in range(args.steps):
        e0, e1, e2 = ev[i]
        e0.record(stream)
        g_pre.replay()
        e1.record(stream)
        decode64()
        e2.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    wall = time.perf_counter() - wall0
    clocks = sampler.stop()
    gla.status_sync()

    # per prefill call (each step replays N_SETS calls)
    pre_ms = [ev[i][0].elapsed_time(ev[i][1]) / N_SETS for i in range(args.steps)]
    # the same calls launched one by one from Python, events around each
    eager_ms = []
    for i in range(max(8, args.steps)):
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        prefill(i)
        a1.record(stream)
        torch.cuda.synchronize()
        eager_ms.append(a0.elapsed_time(a1))
    dec_ms = [ev[i][1].elapsed_time(ev[i][2]) for i in range(args.steps)]
    pre_s = max_over_ranks(sum(pre_ms) * N_SETS / 1e3, world)
    dec_s = max_over_ranks(sum(dec_ms) / 1e3, world)
    step_s = max_over_ranks(wall / args.steps, world)
    tokens = sum_over_ranks(B * T * N_SETS * args.steps, world)
    seq_steps = sum_over_ranks(wd.N * DECODE_STEPS * args.steps, world)

    # ---------------------------------------------------------------- e2e
    # Host buffers in, host buffers out: each step copies its inputs from
    # pinned host memory, runs, and copies its outputs back.  Two buffer slots
    # pipeline the steps as a server would: step i's input copies (one stream)
    # overlap step i-1's compute and result copies (another stream), and a slot
    # is refilled only once the step that last used it has been read and
    # copied out.
    host = {n: x[n].pin_memory() if x[n] is not None else None
            for n in ("q", "k", "v", "g", "init_state")}
    h_out = torch.empty(B, T, H, wp.dv, dtype=torch.bfloat16).pin_memory()
    h_fin = torch.empty(B, H, wp.dk, wp.dv, dtype=torch.float32).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host.values() if t is not None)
    d2h = h_out.numel() * 2 + h_fin.numel() * 4
    e2e_steps = max(3, min(args.steps, 20))
    copy_in = torch.cuda.Stream(device=dev)
    copy_out = torch.cuda.Stream(device=dev)

    def pipelined(n_steps, h2d_fn, compute_fn, d2h_fn):
        copy_in.wait_stream(stream)
        copy_out.wait_stream(stream)
        read_done, out_free = [None, None], [None, None]
        for i in range(n_steps):
            j = i % 2
            if read_done[j] is not None:
                copy_in.wait_event(read_done[j])
            with torch.cuda.stream(copy_in):
                h2d_fn(j)
            e_in = torch.cuda.Event()
            e_in.record(copy_in)
            stream.wait_event(e_in)
            if out_free[j] is not None:
                stream.wait_event(out_free[j])
            compute_fn(j)
            e_c = torch.cuda.Event()
            e_c.record(stream)
            read_done[j] = e_c
            copy_out.wait_event(e_c)
            with torch.cuda.stream(copy_out):
                d2h_fn(j)
            e_o = torch.cuda.Event()
            e_o.record(copy_out)
            out_free[j] = e_o
        stream.wait_stream(copy_in)
        stream.wait_stream(copy_out)

    pslot = (N_SETS - 1, N_SETS - 2)  # the device input sets and outputs of the two slots

    def pre_h2d(j):
        for n, t in host.items():
            if t is not None:
                sets[pslot[j]][n].copy_(t, non_blocking=True)

    def pre_d2h(j):
        h_out.copy_(outs[pslot[j]], non_blocking=True)
        h_fin.copy_(finals[pslot[j]], non_blocking=True)

    def e2e_prefill(n):
        pipelined(n, pre_h2d, lambda j: prefill(pslot[j]), pre_d2h)

    hd = {n: d[n][0].pin_memory() for n in ("q", "k", "v", "g")}
    hd_out = torch.empty(wd.N, wd.H, wd.dv, dtype=torch.bfloat16).pin_memory()
    d_h2d = sum(t.numel() * t.element_size() for t in hd.values())
    d_d2h = hd_out.numel() * 2

    def dec_h2d(j):
        for n, dst in (("q", d_q), ("k", d_k), ("v", d_v), ("g", d_g)):
            dst[j].copy_(hd[n], non_blocking=True)

    def dec_compute(j):
        gla.decode_step(d_q[j], d_k[j], d_v[j], d_g[j], d_state, scale=wd.dk ** -0.5,
                        out=d_out[j])

    def dec_d2h(j):
        hd_out.copy_(d_out[j], non_blocking=True)

    def e2e_decode(n):
        pipelined(n, dec_h2d, dec_compute, dec_d2h)

    e2e_prefill(2)
    e2e_decode(2)
    torch.cuda.synchronize()
    barrier(world)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    e2e_prefill(e2e_steps)
    b.record(stream)
    torch.cuda.synchronize()
    e2e_pre_s = max_over_ranks(a.elapsed_time(b) / 1e3, world)
    a.record(stream)
    e2e_decode(e2e_steps)
    b.record(stream)
    torch.cuda.synchronize()
    e2e_dec_s = max_over_ranks(a.elapsed_time(b) / 1e3, world)
    barrier(world)
    gla.status_sync()

    if rank != 0:
        return None

    hbm, tf_burst, tf_sust, peak_kind = peaks()
    pb = prefill_bytes(wp, B, T)
    pf = prefill_flops(wp, B, T)
    pre_launch_s = statistics.mean(pre_ms) / 1e3
    pre_gbs = pb / pre_launch_s / 1e9
    db = decode_bytes(wd)
    dec_launch_s = statistics.mean(dec_ms) / 1e3 / DECODE_STEPS
    dec_gbs = db / dec_launch_s / 1e9

    dec_roof = {"kernel": "decode_kernel", "bound": "hbm", "achieved": dec_gbs, "peak": hbm,
                "unit": "GB/s", "frac": dec_gbs / hbm, "peak_kind": peak_kind,
                "traffic": profiled_traffic("decode_kernel.decode_n1280_h16.md", "gla_decode.cu"),
                "algorithmic_bytes_per_launch": db,
                "time_share_of_step": DECODE_STEPS * dec_launch_s /
                (DECODE_STEPS * dec_launch_s + N_SETS * pre_launch_s)}
    line = {
        "metric": METRIC,
        "value": tokens / pre_s,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": step_s * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded normal q, k, v; logsigmoid gates; no dataset)",
        "config": prefill_config(world),
        "prefill": {
            "ms_per_call": statistics.mean(pre_ms),
            "ms_per_call_median": statistics.median(pre_ms), "tokens_per_call": B * T,
            "calls": args.steps * N_SETS,
            "launch": f"{N_SETS} rotating calls per step replayed from one CUDA graph",
            "ms_per_call_eager_median": statistics.median(eager_ms),
            "roofline": {
                "kernel": "chunk_tc_kernel", "bound": "hbm", "achieved": pre_gbs, "peak": hbm,
                "unit": "GB/s", "frac": pre_gbs / hbm, "peak_kind": peak_kind,
                "traffic": profiled_traffic("chunk_tc_kernel.prefill_b4_h16_t2048.md",
                                            "gla_chunk_tc.cu"),
                "algorithmic_bytes_per_launch": pb,
                "tensor": {"achieved_tflops": pf / pre_launch_s / 1e12, "peak_tflops": tf_burst,
                           "frac": pf / pre_launch_s / 1e12 / tf_burst,
                           "flops_per_launch": pf}},
        },
        # the kernel that takes most of each step (64 decode launches per prefill)
        "roofline": dec_roof,
        "decode": {
            "value": seq_steps / dec_s, "unit": "seq*steps/s",
            "workload": f"decode step N={wd.N} H={wd.H} dk=dv={wd.dk}, fp32 state in place, "
                        f"{DECODE_STEPS} consecutive steps per timing",
            "ms_per_step": dec_launch_s * 1e3,
            "ms_per_step_median": statistics.median(dec_ms) / DECODE_STEPS,
            "roofline": dec_roof,
        },
        "e2e": {"value": B * T * e2e_steps * world / e2e_pre_s, "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "decode": {"value": wd.N * e2e_steps * world / e2e_dec_s,
                           "unit": "seq*steps/s", "h2d_bytes_per_step": d_h2d,
                           "d2h_bytes_per_step": d_d2h}},
        "gpu_launches": args.steps * (N_SETS + DECODE_STEPS),
        "clocks": clocks,
    }
    if not args.no_side_workloads:
        # timed after the step (outside ms_per_step and gpu_launches)
        line["prefill_workloads"] = time_side_workloads(gla, dev, hbm, peak_kind)
        line["decode_graphs"] = [time_decode_graphs(gla, dev, width=n) for n in (8, 64)]
        line["mixer"] = time_mixer(gla, dev, hbm)
        line["backward"] = time_backward(gla, dev)
    if world == 1 and not args.no_cpu_baseline:
        pre_cpu, dec_cpu = cpu_baseline(args.cpu_budget)
        line["cpu_baseline"] = pre_cpu
        line["decode"]["cpu_baseline"] = dec_cpu
    return line


# ------------------------------------------------------------- profile cases
def run_profile_case(args):
    """One kernel alone, for Nsight Compute captures: W warm-up launches, then K
    timed launches of the prefill or the decode kernel.  Prints one JSON line."""
    import gated_linear_attention_gla_gb300 as gla
    from gated_linear_attention_gla_gb300 import build as glabuild
    glabuild.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    if args.profile in ("backward", "backward-tc"):
        w = gla_inputs.WORKLOADS["prefill"]
        x = gla_inputs.prefill_inputs(w)
        gr = gla_inputs.grad_inputs(x)
        bargs = [x[n].to(dev) for n in ("q", "k", "v", "g")] + [gr["d_out"].to(dev)]
        bkw = dict(scale=x["scale"], init_state=x["init_state"].to(dev),
                   d_final_state=gr["d_final_state"].to(dev),
                   tensor_cores=args.profile == "backward-tc")

        def call():
            gla.chunk_bwd(*bargs, **bkw)
        nbytes = 0
    elif args.profile in ("prefill", "vector", "varlen", "laplace", "fp32", "mixer"):
        # fp32: the prefill workload with fp32 q, k, v, out (the CUDA-core kernel);
        # mixer: the prefill workload with the mixer's steps after the readout
        w = gla_inputs.WORKLOADS[args.profile if args.profile not in ("fp32", "mixer")
                                 else "prefill"]
        x = gla_inputs.prefill_inputs(w)
        q, k, v, g = (x[n].to(dev) for n in ("q", "k", "v", "g"))
        if args.profile == "fp32":
            q, k, v = q.float(), k.float(), v.float()
        s0 = x["init_state"].to(dev) if x["init_state"] is not None else None
        cu = x["cu_seqlens"].to(dev) if x["cu_seqlens"] is not None else None
        kw = dict(scale=x["scale"], init_state=s0, cu_seqlens=cu, chunk=w.chunk)
        if args.profile == "mixer":
            m = gla_inputs.mixer_inputs(w, q.shape[:-2])
            kw["mixer"] = {n: (t.to(dev) if torch.is_tensor(t) else t) for n, t in m.items()}

        def call():
            gla.chunk_fwd(q, k, v, g, **kw)
        nseq = (len(x["cu_seqlens"]) - 1) if cu is not None else w.B
        rows = q.numel() // (w.H * w.dk)
        nbytes = prefill_bytes(w, nseq, 0, rows=rows)
        if args.profile == "fp32":  # q, k, v and out in fp32: twice their bf16 bytes
            nbytes += 2 * rows * w.H * (2 * w.dk + w.dv) + 2 * rows * w.H * w.dv
    else:
        w = gla_inputs.WORKLOADS["decode"]
        d = gla_inputs.decode_inputs(w, steps=1, N=args.decode_n)
        q, k, v, g = (d[n][0].to(dev) for n in ("q", "k", "v", "g"))
        st = d["state"].to(dev)
        w = gla_inputs.dataclasses.replace(w, N=args.decode_n)

        def call():
            gla.decode_step(q, k, v, g, st, scale=d["scale"])
        nbytes = decode_bytes(w)
    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(args.steps):
        call()
    b.record()
    torch.cuda.synchronize()
    gla.status_sync()
    ms = a.elapsed_time(b) / args.steps
    print(json.dumps({"profile": args.profile, "ms_per_launch": ms,
                      "algorithmic_bytes": nbytes, "gbs": nbytes / ms / 1e6}), flush=True)


# ------------------------------------------------------------ reference arm
def run_reference(args, world, rank):
    """The fp64 CPU oracle as the reference arm (rank 0 only)."""
    if rank != 0:
        return None
    import oracle
    wp = gla_inputs.WORKLOADS["prefill"]
    x = gla_inputs.prefill_inputs(wp)
    cores = oracle.max_threads()
    for _ in range(args.warmup):
        oracle.recurrent(x["q"][:1, :256], x["k"][:1, :256], x["v"][:1, :256],
                         x["g"][:1, :256], x["scale"], init_state=x["init_state"][:1])
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.recurrent(x["q"], x["k"], x["v"], x["g"], x["scale"], init_state=x["init_state"])
        times.append(time.perf_counter() - t0)
    total = sum(times)
    value = wp.B * wp.T * args.steps / total
    sample = (f"full prefill workload (B={wp.B}, T={wp.T}, H={wp.H}, d={wp.dk}) per step, "
              f"fp64 token-by-token recurrence")
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": total / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded normal q, k, v; logsigmoid gates; no dataset)",
        "config": prefill_config(world),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["gla", "reference"], default="gla")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=10.0,
                    help="seconds of oracle time for the cpu_baseline sample")
    ap.add_argument("--no-side-workloads", action="store_true",
                    help="skip timing the vector-gate and varlen prefill workloads")
    ap.add_argument("--profile", choices=["prefill", "vector", "varlen", "laplace", "fp32",
                                          "mixer", "decode", "backward", "backward-tc"],
                    default=None,
                    help="run one kernel alone (for ncu captures) instead of the bench")
    ap.add_argument("--decode-n", type=int, default=1280,
                    help="sequences for --profile decode")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.profile:
        run_profile_case(args)
        return
    world, rank, local = dist_env()
    if args.impl == "reference":
        line = run_reference(args, world, rank)
    else:
        dist_init(world, local)
        line = run_gla(args, world, rank, local)
    if line is not None:
        print(json.dumps(line), flush=True)
    if world > 1 and args.impl != "reference":
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
