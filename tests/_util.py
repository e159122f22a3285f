"""Helpers shared by the test files: tolerances and device plumbing.

Tolerance: max |gpu - oracle| <= TOL * RMS(oracle), separately for o and for
the state, with TOL = 1e-4 for fp32 inputs and 2e-2 for bf16 inputs with fp32
accumulation.  A result that the method stores in bf16 (o for bf16 inputs,
the decode state pool) cannot be closer to the exact value than half a bf16
unit in the last place, so for those results that storage rounding,
2^(floor(log2 |x|) - 8) per element, is taken off each element's error before
the bound is applied.  fp32 results (the prefill final state) get no such
allowance.
"""
import numpy as np
import torch

TOL_F32 = 1e-4
TOL_BF16 = 2e-2


def _np(x):
    if hasattr(x, "detach"):
        return x.detach().cpu().double().numpy()
    return np.asarray(x, dtype=np.float64)


def bf16_half_ulp(x):
    """Largest round-to-nearest error of storing |x| in bf16 (8 significant bits)."""
    ax = np.abs(x)
    e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    return np.where(ax > 0, np.exp2(e - 8), 0.0)


def rel_max_err(got, ref, bf16_out=None):
    """max over elements of (|got - ref| - storage rounding) / RMS(ref)."""
    g = _np(got)
    r = np.asarray(ref, dtype=np.float64)
    if bf16_out is None:
        bf16_out = hasattr(got, "dtype") and got.dtype == torch.bfloat16
    err = np.abs(g - r)
    if bf16_out:
        err = np.maximum(err - bf16_half_ulp(np.maximum(np.abs(g), np.abs(r))), 0.0)
    rms = float(np.sqrt(np.mean(r * r)))
    if rms == 0.0:
        return float(np.max(err)) if err.size else 0.0
    return float(np.max(err) / rms) if err.size else 0.0


def assert_close(got, ref, tol, what):
    e = rel_max_err(got, ref)
    raw = rel_max_err(got, ref, bf16_out=False)
    assert np.isfinite(e) and e <= tol, (
        f"{what}: error {e:.3e} x RMS exceeds {tol:.1e} (raw max-abs {raw:.3e} x RMS)")
    return e


def to_dev(inp, device="cuda"):
    """Copy every tensor of a synth dict to the device."""
    out = {}
    for key, val in inp.items():
        out[key] = val.to(device) if isinstance(val, torch.Tensor) else val
    return out
