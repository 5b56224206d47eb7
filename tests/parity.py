"""Helpers for the GPU-vs-oracle parity tests.

Error metric: max over elements of |gpu - ref| divided by RMS(ref) of the same tensor, taken
separately for outputs, final states and checkpoints.  Bounds: fp32 inputs 1e-4 on outputs
and states; bf16 inputs (fp32 state and accumulation) 2e-2 on outputs, 1e-2 on states and
checkpoints.
"""
from __future__ import annotations

import numpy as np
import torch

TOL = {
    "f32": {"out": 1e-4, "state": 1e-4},
    "bf16": {"out": 2e-2, "state": 1e-2},
}


def rel_err(gpu, ref) -> float:
    g = gpu.detach().to("cpu", torch.float64).numpy() if isinstance(gpu, torch.Tensor) else np.asarray(gpu)
    ref = np.asarray(ref, dtype=np.float64)
    assert g.shape == ref.shape, (g.shape, ref.shape)
    if ref.size == 0:
        return 0.0
    rms = float(np.sqrt(np.mean(ref * ref)))
    if rms == 0.0:
        return float(np.max(np.abs(g)))
    return float(np.max(np.abs(g - ref)) / rms)


def assert_close(name, gpu, ref, tol):
    e = rel_err(gpu, ref)
    assert np.isfinite(e) and e <= tol, f"{name}: max|err|/RMS = {e:.3e} > {tol:.1e}"
    return e


def head_slice(x: dict, heads, keys=("q", "k", "v", "g", "beta")):
    """CPU copies of the given heads of packed inputs (exact: bf16/fp32 -> fp64 later)."""
    idx = torch.as_tensor(heads, device=x["q"].device)
    return {key: x[key].index_select(1, idx).cpu() for key in keys}
