"""Shared test helpers: tolerance checks and library access."""
from __future__ import annotations

import os

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# Tolerances (torch.allclose semantics |a-b| <= atol + rtol |b|):
#   losses rel 1e-4; gradients rel 1e-3, abs 1e-5 (with the 1/B mean factor applied).
LOSS_RTOL = 1e-4
GRAD_RTOL = 1e-3
GRAD_ATOL = 1e-5


def ensure_built():
    from differentiable_series_alignment_gb300 import build
    return build.build()


def close_report(a, b, rtol, atol, what=""):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, (what, a.shape, b.shape)
    assert np.all(np.isfinite(a)), f"{what}: non-finite values in the CUDA result"
    bound = atol + rtol * np.abs(b)
    viol = np.abs(a - b) / bound
    k = int(np.argmax(viol))
    worst = float(viol.flat[k])
    msg = (f"{what}: worst |a-b|/(atol+rtol|b|) = {worst:.3g} at {np.unravel_index(k, a.shape)} "
           f"(a={a.flat[k]!r}, b={b.flat[k]!r})")
    return worst, msg


def assert_close(a, b, rtol, atol=0.0, what=""):
    worst, msg = close_report(a, b, rtol, atol, what)
    assert worst <= 1.0, msg
    return worst
