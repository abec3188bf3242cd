"""Shared helpers of the GPU parity tests.

Tolerances (stated for the method with bf16 inputs and fp32 accumulation,
and for the fp32 path):
  * bf16 path: max |gpu - ref| <= 2e-2 * RMS(ref), over the whole output
    tensor of a case, and separately over the final state;
  * fp32 path: max |gpu - ref| <= 1e-4 * RMS(ref), same normaliser.
ref is the fp64 CPU oracle run on exactly the values the GPU saw (bf16
inputs upcast exactly, lambda rounded to fp32).
"""
import numpy as np
import torch

TOL_BF16 = 2e-2
TOL_FP32 = 1e-4


def to64(t) -> np.ndarray:
    if isinstance(t, torch.Tensor):
        return t.detach().to("cpu").double().numpy()
    return np.asarray(t, dtype=np.float64)


def rel_err(got, ref) -> float:
    """max |got - ref| / RMS(ref); 0 when both are empty."""
    got, ref = to64(got), to64(ref)
    if ref.size == 0:
        return 0.0
    rms = float(np.sqrt(np.mean(ref ** 2)))
    err = float(np.max(np.abs(got - ref)))
    if rms == 0.0:
        return err
    return err / rms


def assert_close(got, ref, tol, what=""):
    e = rel_err(got, ref)
    assert np.isfinite(e) and e <= tol, f"{what}: max|err|/RMS = {e:.3e} > {tol:.1e}"
    return e
