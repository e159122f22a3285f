"""Helpers shared by the test files: tolerances and device plumbing."""
import numpy as np
import torch

# max |gpu - oracle| <= TOL * RMS(oracle), separately for o and for the state
TOL_F32 = 1e-4
TOL_BF16 = 2e-2


def rel_max_err(got, ref):
    """max |got - ref| / RMS(ref), with got/ref as torch tensors or arrays."""
    g = got.detach().cpu().double().numpy() if hasattr(got, "detach") else np.asarray(got, np.float64)
    r = np.asarray(ref, dtype=np.float64)
    rms = float(np.sqrt(np.mean(r * r)))
    if rms == 0.0:
        return float(np.max(np.abs(g - r)))
    return float(np.max(np.abs(g - r)) / rms)


def assert_close(got, ref, tol, what):
    e = rel_max_err(got, ref)
    assert np.isfinite(e) and e <= tol, f"{what}: max-abs error {e:.3e} x RMS exceeds {tol:.1e}"
    return e


def to_dev(inp, device="cuda"):
    """Copy every tensor of a synth dict to the device."""
    out = {}
    for key, val in inp.items():
        out[key] = val.to(device) if isinstance(val, torch.Tensor) else val
    return out
