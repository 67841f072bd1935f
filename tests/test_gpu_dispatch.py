"""Which kernel serves which call.

The dispatch rule is a pure host function of the C ABI (checked on the CPU):
bf16 I/O with chunk 128 runs a tcgen05 tensor-core kernel (the per-head gate
with dk = 64, 96 or 128 and dv = 64, 128 or 192; the per-key-channel gate with
dk = dv = 128), everything else the fp32 CUDA-core kernel.  On a GPU, where the CUDA profiler
can trace kernels, the launched kernel names are checked as well."""
import pytest
import torch

import gla_inputs
from gated_linear_attention_gla_gb300 import _binding, build as glabuild
from parity import cuda

F32 = _binding.GLA_FLAG_FP32_IO
VEC = _binding.GLA_FLAG_VECTOR_GATE
F32OUT = _binding.GLA_FLAG_FP32_OUT


@pytest.fixture(scope="module")
def L():
    glabuild.build()
    return _binding.lib()


@pytest.mark.parametrize("dk,dv,chunk,flags,expect", [
    (128, 128, 128, 0, "tensor_core"),
    (128, 64, 128, 0, "tensor_core"),
    (128, 128, 128, F32OUT, "tensor_core"),
    (128, 128, 64, 0, "cuda_core"),
    (128, 128, 128, F32, "cuda_core"),
    (64, 64, 128, 0, "tensor_core"),
    (64, 128, 128, 0, "tensor_core"),
    (64, 192, 128, 0, "tensor_core"),
    (64, 128, 128, VEC, "cuda_core"),
    (64, 128, 128, F32, "cuda_core"),
    (128, 128, 128, VEC, "tensor_core"),
    (128, 128, 128, VEC | F32OUT, "tensor_core"),
    (128, 64, 128, VEC, "cuda_core"),
    (128, 128, 64, VEC, "cuda_core"),
    (128, 128, 128, VEC | F32, "cuda_core"),
    (96, 192, 128, 0, "tensor_core"),
    (96, 128, 128, 0, "tensor_core"),
    (128, 192, 128, 0, "tensor_core"),
    (96, 192, 128, VEC, "cuda_core"),
    (96, 192, 64, 0, "cuda_core"),
    (80, 128, 128, 0, None),
    (128, 96, 128, 0, None),
    (128, 128, 100, 0, None),
    (128, 128, 128, 1 << 9, None),
])
def test_dispatch_rule(L, dk, dv, chunk, flags, expect):
    assert _binding.chunk_fwd_kernel(dk, dv, chunk, flags) == expect


def kernels_launched(fn):
    from torch.profiler import ProfilerActivity, profile
    torch.cuda.synchronize()
    with profile(activities=[ProfilerActivity.CUDA]) as prof:
        fn()
        torch.cuda.synchronize()
    return {e.name for e in prof.events() if e.device_type == torch.autograd.DeviceType.CUDA}


@pytest.mark.gpu
def test_launched_kernel_names(cuda_ok):
    import gated_linear_attention_gla_gb300 as gla
    x = gla_inputs.prefill_inputs(gla_inputs.WORKLOADS["prefill"], B=1, T=300, H=2)
    args = [cuda(x[n]) for n in ("q", "k", "v", "g")]
    probe = kernels_launched(lambda: args[0] * 2)
    if not probe:
        pytest.skip("the CUDA profiler traces no kernels on this machine")
    names = kernels_launched(lambda: gla.chunk_fwd(*args, chunk=128))
    assert any("chunk_tc_kernel" in n for n in names), names
    names = kernels_launched(lambda: gla.chunk_fwd(*args, chunk=64))
    assert any("chunk_simt_kernel" in n for n in names), names
