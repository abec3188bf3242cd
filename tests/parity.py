"""Shared helpers of the GPU parity tests.

Tolerances.  The method's bound is on the arithmetic: with bf16 inputs and
fp32 accumulation, max |gpu - ref| <= 2e-2 * RMS(ref); on the fp32 path
1e-4 * RMS(ref).  ref is the fp64 CPU oracle run on exactly the values the
GPU saw (bf16 inputs upcast exactly, lambda rounded to fp32).

The output tensor is stored in the input dtype (bf16 for the measured
workloads), and storing even the exact result in bf16 moves an element by up
to u * |ref| with u = 2^-8 (round to nearest even, 8 significant bits).  For
heavy-tailed outputs an element near 10 RMS then misses 2e-2 * RMS by
rounding alone (test_bf16_storage_rounding_needs_the_u_term shows the
oracle's own result rounded to bf16 failing the plain bound), so each element
is allowed its storage rounding on top of the arithmetic bound:
    |gpu - ref| <= tol * RMS(ref) + u_out * |ref|
with u_out = 2^-8 for bf16 outputs and 2^-24 for fp32 outputs.  fp32 final
states are stored without extra rounding and take u_out = 2^-24.
"""
import numpy as np
import torch

TOL_BF16 = 2e-2
TOL_FP32 = 1e-4
U_BF16 = 2.0 ** -8
U_FP32 = 2.0 ** -24


def to64(t) -> np.ndarray:
    if isinstance(t, torch.Tensor):
        return t.detach().to("cpu").double().numpy()
    return np.asarray(t, dtype=np.float64)


def storage_u(t) -> float:
    if isinstance(t, torch.Tensor) and t.dtype == torch.bfloat16:
        return U_BF16
    return U_FP32


def rel_err(got, ref) -> float:
    """Plain max |got - ref| / RMS(ref) (diagnostic)."""
    got, ref = to64(got), to64(ref)
    if ref.size == 0:
        return 0.0
    rms = float(np.sqrt(np.mean(ref ** 2)))
    err = float(np.max(np.abs(got - ref)))
    return err / rms if rms > 0 else err


def excess_err(got, ref, u) -> float:
    """max over elements of (|got - ref| - u |ref|) / RMS(ref)."""
    got, ref = to64(got), to64(ref)
    if ref.size == 0:
        return 0.0
    rms = float(np.sqrt(np.mean(ref ** 2)))
    ex = float(np.max(np.abs(got - ref) - u * np.abs(ref)))
    return ex / rms if rms > 0 else ex


def assert_close(got, ref, tol, what="", u=None):
    """Elementwise |got - ref| <= tol * RMS(ref) + u * |ref|; u defaults to
    the storage rounding of got's dtype."""
    u = storage_u(got) if u is None else u
    e = excess_err(got, ref, u)
    plain = rel_err(got, ref)
    print(f"[parity] {what}: arithmetic {e:.3e} (bound {tol:.1e}), plain max|err|/RMS {plain:.3e}")
    assert np.isfinite(e) and e <= tol, f"{what}: (|err| - u|ref|)/RMS = {e:.3e} > {tol:.1e}"
    return e
