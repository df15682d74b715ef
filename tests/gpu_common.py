"""Helpers shared by the GPU parity tests (test infrastructure only)."""

from __future__ import annotations

import numpy as np

# Acceptance bounds for bf16 outputs against the fp64 oracle.
O_MAX_ABS = 2e-2
O_MEAN_ABS = 2e-3
LSE_ABS = 1e-3


def to_np(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def assert_close(o_gpu, lse_gpu, o_ref, lse_ref, what=""):
    """o_*: same shape; lse_*: same shape (fp64 numpy arrays)."""
    err = np.abs(o_gpu - o_ref)
    lerr = np.abs(lse_gpu - lse_ref)
    assert np.isfinite(o_gpu).all() and np.isfinite(lse_gpu).all(), f"{what}: non-finite output"
    assert err.max() <= O_MAX_ABS, f"{what}: O max-abs {err.max():.3e} > {O_MAX_ABS}"
    assert err.mean() <= O_MEAN_ABS, f"{what}: O mean-abs {err.mean():.3e} > {O_MEAN_ABS}"
    assert lerr.max() <= LSE_ABS, f"{what}: LSE max-abs {lerr.max():.3e} > {LSE_ABS}"
    return float(err.max()), float(err.mean()), float(lerr.max())
