"""Helpers for the GPU parity tests: building C-ABI items from torch tensors
and comparing device results with the fp64 oracle."""
from __future__ import annotations

import math

import numpy as np
import torch

BF16_TOL = (1e-2, 1e-3)    # max-abs, mean-abs for bf16 inputs
F32_TOL = (2e-4, 2e-5)     # max-abs, mean-abs for fp32 inputs


def tol_for(dtype):
    return BF16_TOL if dtype in (torch.bfloat16, "bf16") else F32_TOL


def errors(got, ref, finite_only=False):
    g = got.double().cpu().numpy() if hasattr(got, "cpu") else np.asarray(got, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, (g.shape, r.shape)
    inf_g, inf_r = np.isneginf(g), np.isneginf(r)
    assert np.array_equal(inf_g, inf_r), "-inf pattern differs"
    mask = ~inf_r
    d = np.abs(g[mask] - r[mask])
    assert np.all(np.isfinite(d)), "non-finite values"
    return (float(d.max()) if d.size else 0.0), (float(d.mean()) if d.size else 0.0)


def assert_close(name, got, ref, tol):
    mx, mn = errors(got, ref)
    assert mx <= tol[0] and mn <= tol[1], f"{name}: max-abs {mx:.3e} (tol {tol[0]}), mean-abs {mn:.3e} (tol {tol[1]})"
    return mx, mn


def scale_for(D):
    return 1.0 / math.sqrt(D)
