"""Helpers for the GPU parity tests: numpy <-> torch device copies (bit
patterns preserved) and the float tolerance rule.

Tolerance: the pages and the task fix "2e-3 max relative error" without a
denominator; pure elementwise relative error is ill-posed near zero, so a
float result g passes against the oracle r when, element by element,
    |g - r| <= 2e-3 * max(|r|, rms(r))      (rms over the compared tensor).
"""
import numpy as np
import torch

TOL = 2e-3

_TORCH = {np.dtype(np.uint16): torch.int16, np.dtype(np.int8): torch.int8, np.dtype(np.uint8): torch.uint8,
          np.dtype(np.float32): torch.float32, np.dtype(np.int32): torch.int32}


def dev(a):
    """numpy -> CUDA tensor with the same bytes (uint16 travels as int16)."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).cuda()


def host(t, dtype=None):
    a = t.detach().cpu().numpy()
    if dtype is not None:
        a = a.view(dtype)
    return a


def rel_err(g, r):
    """max over elements of |g - r| / max(|r|, rms(r))."""
    g = np.asarray(g, np.float64)
    r = np.asarray(r, np.float64)
    rms = np.sqrt(np.mean(r * r)) if r.size else 0.0
    den = np.maximum(np.abs(r), rms)
    den = np.where(den == 0, 1.0, den)
    return float(np.max(np.abs(g - r) / den)) if r.size else 0.0


def assert_close(g, r, tol=TOL, what=""):
    e = rel_err(g, r)
    assert np.all(np.isfinite(g)), f"{what}: non-finite values"
    assert e <= tol, f"{what}: max relative error {e:.3e} > {tol}"
    return e


def zeros_status():
    return torch.zeros(1, dtype=torch.int32, device="cuda")
