"""Helpers shared by the GPU parity tests: run both sides, measure the error.

Error norm (the one the tolerances are stated in): ``max |x - ref| / RMS(ref)``
over the whole tensor, with the reference in fp64.

bf16-input calls are checked in two parts.  The kernels accumulate in fp32 and
round once when they store a bf16 output; that last rounding alone can cost
up to 2^-8 * max|o| / RMS(o) (about 2e-2 for Gaussian-like outputs of a few
million elements), the whole tolerance.  So the tolerance is applied to the
fp32-accumulated result (the same call with an fp32 output), and the bf16
output is required to be exactly that result rounded to nearest-even.
"""
from __future__ import annotations

import numpy as np
import torch

TOL_OUT_BF16 = 2e-2   # bf16 inputs/outputs, fp32 accumulation
TOL_OUT_FP32 = 1e-5   # fp32 inputs/outputs
TOL_STATE = 1e-3      # final state (fp32), relative to its RMS


def rel_max(x, ref) -> float:
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0
    if ref.size == 0:
        return 0.0
    return float(np.max(np.abs(x - ref))) / max(rms, 1e-30)


def rel_fro(x, ref) -> float:
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return float(np.linalg.norm(x - ref)) / max(float(np.linalg.norm(ref)), 1e-30)


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().double().cpu().numpy()


def cuda(t):
    return None if t is None else t.cuda()


def out_tol(dtype) -> float:
    return TOL_OUT_FP32 if dtype == torch.float32 else TOL_OUT_BF16


def check_bf16_rounding(out_bf16: torch.Tensor, out_f32: torch.Tensor):
    """The bf16 output is the fp32 result of the same computation rounded once (RNE)."""
    assert out_bf16.dtype == torch.bfloat16 and out_f32.dtype == torch.float32
    same = torch.equal(out_bf16, out_f32.to(torch.bfloat16))
    assert same, "bf16 output differs from the fp32 result rounded to nearest-even"
