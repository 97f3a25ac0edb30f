"""Shared helpers for the parity tests (no attention arithmetic here)."""
from __future__ import annotations

import numpy as np
import torch

TOL_F32 = 1e-4   # max relative error bound for fp32 inputs
TOL_BF16 = 2e-2  # max relative error bound for bf16 inputs with fp32 accumulation


def tol_for(dtype) -> float:
    return TOL_BF16 if dtype == torch.bfloat16 else TOL_F32


def to_np(t) -> np.ndarray:
    if isinstance(t, torch.Tensor):
        return t.detach().float().cpu().double().numpy() if t.dtype == torch.bfloat16 else t.detach().cpu().double().numpy()
    return np.asarray(t, np.float64)


def rel_per_head(x, y) -> float:
    """max over (b, h) slices of max|x - y| / max|y| within the slice.

    The bound applies to every [.., N, D] head slice separately, normalised by
    that slice's largest magnitude, so near-zero entries cannot blow it up.
    """
    x, y = to_np(x), to_np(y)
    assert x.shape == y.shape, (x.shape, y.shape)
    if x.size == 0:
        return 0.0
    xs = x.reshape(-1, x.shape[-2] * x.shape[-1]) if x.ndim >= 2 else x.reshape(1, -1)
    ys = y.reshape(xs.shape)
    den = np.max(np.abs(ys), axis=1)
    den = np.where(den > 0, den, 1.0)
    err = np.max(np.abs(xs - ys), axis=1) / den
    if not np.all(np.isfinite(xs)):
        return float("inf")
    return float(np.max(err))
