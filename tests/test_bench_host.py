"""bench.py host logic on the CPU: algorithmic byte counts, the profile
summaries it reads, the reference arm's JSON line, and the multi-rank timing
reduction over a world-size-2 gloo process group."""
import json
import os
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import gla_inputs  # noqa: E402


def test_algorithmic_bytes_match_the_stated_figures():
    w = gla_inputs.WORKLOADS["prefill"]
    # per (token, head): 3 * 2 * 128 + 4 + 2 * 128 = 1028, plus 2 fp32 states per (b, h)
    assert bench.prefill_bytes(w, w.B, w.T) == 1028 * w.B * w.T * w.H + 2 * 4 * w.B * w.H * 128 * 128
    assert bench.prefill_bytes(w, w.B, w.T) == 143_130_624
    assert bench.prefill_flops(w, w.B, w.T) == 131_072 * w.B * w.T * w.H
    d = gla_inputs.WORKLOADS["decode"]
    assert bench.decode_bytes(d) == 132_100 * d.N * d.H == 2_705_408_000


def test_profiled_traffic_follows_the_kernel_source():
    t = bench.profiled_traffic("chunk_tc_kernel.prefill_b4_h16_t2048.md", "gla_chunk_tc.cu")
    text = open(os.path.join(ROOT, "profiles", "chunk_tc_kernel.prefill_b4_h16_t2048.md")).read()
    recorded = text.split("kernel_source_sha256_16:")[1].split()[0]
    if recorded == bench.kernel_source_hash("gla_chunk_tc.cu"):
        assert t is not None and t > 0
    else:
        assert t is None  # the kernel changed since the counters were taken
    assert bench.profiled_traffic("no_such_profile.md", "gla_chunk_tc.cu") is None


def test_reference_arm_prints_one_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], capture_output=True, text=True,
                       timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["value"] > 0
    assert d["unit"] == "tokens/s" and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]


def test_reference_arm_other_ranks_are_silent():
    env = dict(os.environ, WORLD_SIZE="2", RANK="1", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], capture_output=True, text=True,
                       timeout=300, cwd=ROOT, env=env)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_warmup_below_three_is_refused():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--warmup", "2"],
                       capture_output=True, text=True, timeout=120, cwd=ROOT)
    assert r.returncode != 0


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        mx = bench.max_over_ranks(float(rank + 1) * 1.5, world)
        sm = bench.sum_over_ranks(float(rank + 1), world)
        q.put((rank, mx, sm))
    finally:
        dist.destroy_process_group()


def test_timing_reduction_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(2))
    for rank, mx, sm in got:
        assert mx == pytest.approx(3.0)   # max over ranks of (rank + 1) * 1.5
        assert sm == pytest.approx(3.0)   # 1 + 2


def test_clock_sampler_parses_nvidia_smi_rows(tmp_path, monkeypatch):
    s = bench.ClockSampler(0)
    s.path = str(tmp_path / "c.csv")
    with open(s.path, "w") as f:
        f.write("0, 1995, 2070, 600.5, 97, Not Active, Not Active, Not Active, Active\n")
        f.write("0, 2070, 2070, 650.0, 100, Not Active, Not Active, Not Active, Not Active\n")
        f.write("0, 345, 2070, 100.0, 0, Not Active, Not Active, Not Active, Not Active\n")

    class P:
        def terminate(self):
            pass

        def wait(self, timeout=None):
            return 0
    s.proc = P()
    monkeypatch.setattr(bench.time, "sleep", lambda *_: None)
    c = s.stop()
    assert c["samples"] == 2 and c["sm_max_mhz"] == 2070.0
    assert c["sm_mhz"] == pytest.approx((1995 + 2070) / 2)
    assert c["reasons"] == ["sw_power_cap"]


def test_decode_bucket_choice():
    from gated_linear_attention_gla_gb300.serving import default_buckets, pick_bucket
    assert default_buckets(1) == [1]
    assert default_buckets(8) == [1, 2, 4, 8]
    assert default_buckets(12) == [1, 2, 4, 8, 12]
    b = default_buckets(12)
    assert [pick_bucket(b, n) for n in (1, 2, 3, 5, 8, 9, 12)] == [1, 2, 4, 8, 8, 12, 12]
    with pytest.raises(ValueError):
        pick_bucket(b, 13)
    with pytest.raises(ValueError):
        default_buckets(0)


def test_backward_flops_and_fp32_peak():
    import bench
    w = gla_inputs.WORKLOADS["prefill"]
    # per token and head: 32 * (2 * 128 + 3 * 128) + 5 * 128 * 128 MACs
    per = 32 * 640 + 5 * 16384
    assert bench.backward_flops(w, w.B, w.T) == 2 * per * w.B * w.T * w.H
    assert abs(bench.fp32_peak_tflops() - 152 * 128 * 2 * 2.07e9 / 1e12) < 1e-9
