"""Which kernel serves which call (GPU): the tensor-core prefill for bf16 I/O
with chunk 128, the fp32 CUDA-core prefill otherwise, the decode kernel for
decode.  Kernel names come from the CUDA profiler (CUPTI) via torch.profiler."""
import pytest
import torch

import gla_inputs
from parity import cuda

pytestmark = pytest.mark.gpu


def kernels_launched(fn):
    from torch.profiler import ProfilerActivity, profile
    torch.cuda.synchronize()
    with profile(activities=[ProfilerActivity.CUDA]) as prof:
        fn()
        torch.cuda.synchronize()
    return {e.name for e in prof.events() if e.device_type == torch.autograd.DeviceType.CUDA}


def _prefill(chunk, io="bf16", gate="scalar", dk=128):
    import gated_linear_attention_gla_gb300 as gla
    x = gla_inputs.prefill_inputs(gla_inputs.WORKLOADS["prefill"], B=1, T=300, H=2, io=io,
                                  gate=gate, dk=dk, chunk=chunk)
    args = [cuda(x[n]) for n in ("q", "k", "v", "g")]
    return lambda: gla.chunk_fwd(*args, init_state=cuda(x["init_state"]), chunk=chunk)


def test_bf16_chunk128_runs_the_tensor_core_kernel(cuda_ok):
    names = kernels_launched(_prefill(128))
    assert any("chunk_tc_kernel" in n for n in names), names
    assert not any("chunk_simt_kernel" in n for n in names), names


@pytest.mark.parametrize("kw", [dict(chunk=64), dict(chunk=128, io="fp32")])
def test_other_prefill_calls_run_the_cuda_core_kernel(cuda_ok, kw):
    names = kernels_launched(_prefill(**kw))
    assert any("chunk_simt_kernel" in n for n in names), names


def test_decode_runs_the_decode_kernel(cuda_ok):
    import gated_linear_attention_gla_gb300 as gla
    d = gla_inputs.decode_inputs(gla_inputs.WORKLOADS["decode"], N=8, steps=1)
    S = cuda(d["state"])
    names = kernels_launched(lambda: gla.decode_step(cuda(d["q"][0]), cuda(d["k"][0]),
                                                     cuda(d["v"][0]), cuda(d["g"][0]), S))
    assert any("decode_kernel" in n for n in names), names
