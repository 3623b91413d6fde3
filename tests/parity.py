"""Helpers shared by the GPU parity tests: tolerances and comparisons.

Deviation = max |got - want| / RMS(want), with ``want`` the float64 oracle; a
NaN/Inf pattern that differs from the oracle's fails outright. Tolerances:
  * noise: bit-exact;
  * fp32 (FFMA) path and gradients: 1e-4 of the oracle's RMS;
  * bf16 tensor-core path: 2e-2 of the oracle's RMS.
"""

import numpy as np
import torch

TOL_FP32 = 1e-4
TOL_BF16 = 2e-2


def to_np(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        t = t.float()
    return t.detach().cpu().numpy().astype(np.float64)


def deviation(got, want) -> float:
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, (got.shape, want.shape)
    assert np.array_equal(np.isfinite(got), np.isfinite(want)), "NaN/Inf pattern differs"
    rms = float(np.sqrt(np.mean(want ** 2)))
    err = float(np.max(np.abs(got - want))) if got.size else 0.0
    return err / rms if rms > 0 else err


def assert_close(got, want, tol: float, what: str = "") -> float:
    d = deviation(got, want)
    assert d <= tol, f"{what}: deviation {d:.3e} > {tol:.1e} (max abs err / oracle RMS)"
    return d
