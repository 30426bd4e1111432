"""Tolerances for comparing the CUDA path with the fp64 oracle.

* fp32 io dtype: max |x - ref| <= 1e-5 * RMS(ref), every output.
* bf16 io dtype: outputs stored as fp32 (final state, dbeta, dg, dh0):
  max |x - ref| <= 2e-3 * RMS(ref).  Outputs stored as bf16 (o, dq, dk, dv,
  A) carry their own rounding, which alone can reach 1.6e-2 * RMS for a
  Gaussian tensor, so each element must satisfy
      |x - ref| <= 2e-3 * RMS(ref) + ulp_bf16(max(|x|, |ref|)) / 2,
  i.e. the value before the final rounding was within 2e-3 * RMS.
"""
import numpy as np
import torch

FP32_TOL = 1e-5
BF16_TOL = 2e-3


def _np(x):
    if isinstance(x, torch.Tensor):
        return x.detach().to("cpu", torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


def half_ulp_bf16(a):
    a = np.abs(a)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, 2.0 ** (e - 8), 0.0)


def check(name, got, ref, io_dtype, stored_dtype, tol=None):
    """Returns a dict of error figures; raises AssertionError past the bound."""
    g, r = _np(got), _np(ref)
    assert g.shape == r.shape, f"{name}: shape {g.shape} vs {r.shape}"
    assert np.isfinite(g).all(), f"{name}: non-finite values"
    rms = float(np.sqrt(np.mean(r * r))) if r.size else 0.0
    err = np.abs(g - r)
    if tol is None:
        tol = FP32_TOL if io_dtype == torch.float32 else BF16_TOL
    bound = tol * rms
    if stored_dtype == torch.bfloat16:
        bound = bound + half_ulp_bf16(np.maximum(np.abs(g), np.abs(r)))
    excess = err - bound
    info = dict(name=name, rms=rms, max_abs=float(err.max()) if err.size else 0.0,
                max_rel_rms=float(err.max() / rms) if rms > 0 else 0.0,
                rms_rel=float(np.sqrt(np.mean(err ** 2)) / rms) if rms > 0 else 0.0)
    if err.size and rms > 0:
        worst = np.unravel_index(np.argmax(excess), excess.shape)
        assert excess[worst] <= 0, (f"{name}: |x-ref|={err[worst]:.3e} at {worst} exceeds bound "
                                    f"{np.broadcast_to(bound, err.shape)[worst]:.3e} "
                                    f"(tol {tol:g} * rms {rms:.3e}); {info}")
    return info
