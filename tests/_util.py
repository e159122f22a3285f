"""Helpers shared by the test files: tolerances and device plumbing.

Tolerance: max |gpu - oracle| <= TOL * RMS(oracle), separately for o and for
the state, with TOL = 1e-4 for fp32 inputs and 2e-2 for bf16 inputs with fp32
accumulation.  The bound is applied to the raw element-wise error, storage
rounding included.  As a diagnostic only, each check also computes the error
left once every bf16-stored element's own storage rounding (half a bf16 unit
in the last place) is taken off; both figures are recorded and printed in the
session summary (tests/conftest.py), the bound never uses the second one.
"""
import numpy as np
import torch

TOL_F32 = 1e-4
TOL_BF16 = 2e-2

# (test id, what, raw error / RMS, storage-adjusted error / RMS, tolerance)
RECORDS = []
CURRENT_TEST = [""]


def _np(x):
    if hasattr(x, "detach"):
        return x.detach().cpu().double().numpy()
    return np.asarray(x, dtype=np.float64)


def bf16_half_ulp(x):
    """Largest round-to-nearest error of storing |x| in bf16 (8 significant bits)."""
    ax = np.abs(x)
    e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    return np.where(ax > 0, np.exp2(e - 8), 0.0)


def _rms(r):
    return float(np.sqrt(np.mean(r * r))) if r.size else 0.0


def rel_max_err(got, ref):
    """max over elements of |got - ref| / RMS(ref): the bound's quantity."""
    g = _np(got)
    r = np.asarray(ref, dtype=np.float64)
    if not g.size:
        return 0.0
    err = float(np.max(np.abs(g - r)))
    rms = _rms(r)
    return err / rms if rms > 0.0 else err


def storage_adjusted_err(got, ref):
    """Diagnostic: the error left once each bf16 element's storage rounding is
    taken off (a bf16 number cannot be closer to the exact value than that)."""
    g = _np(got)
    r = np.asarray(ref, dtype=np.float64)
    if not g.size:
        return 0.0
    err = np.abs(g - r)
    if hasattr(got, "dtype") and got.dtype == torch.bfloat16:
        err = np.maximum(err - bf16_half_ulp(np.maximum(np.abs(g), np.abs(r))), 0.0)
    rms = _rms(r)
    return float(np.max(err)) / rms if rms > 0.0 else float(np.max(err))


def assert_close(got, ref, tol, what):
    raw = rel_max_err(got, ref)
    adj = storage_adjusted_err(got, ref)
    RECORDS.append((CURRENT_TEST[0], what, raw, adj, tol))
    assert np.isfinite(raw) and raw <= tol, (
        f"{what}: max-abs error {raw:.3e} x RMS exceeds {tol:.1e} "
        f"(storage-adjusted diagnostic {adj:.3e})")
    return raw


def to_dev(inp, device="cuda"):
    """Copy every tensor of a synth dict to the device."""
    out = {}
    for key, val in inp.items():
        out[key] = val.to(device) if isinstance(val, torch.Tensor) else val
    return out
