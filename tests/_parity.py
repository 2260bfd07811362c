"""Comparison helpers for the GPU parity tests.

Tolerance (fp32 kernels against the float64 oracle, per output tensor):
    relative L2  ||y - y_ref||_2 / ||y_ref||_2  <= 1e-5
    max abs      max |y - y_ref|                <= 1e-4 * sqrt(T)
"""
import math

import numpy as np

REL_L2 = 1e-5
ABS_PER_SQRT_T = 1e-4


def errors(gpu, ref):
    g = gpu.detach().double().cpu().numpy() if hasattr(gpu, "detach") else np.asarray(gpu, np.float64)
    r = np.asarray(ref, np.float64)
    assert g.shape == r.shape, (g.shape, r.shape)
    if r.size == 0:
        return 0.0, 0.0
    d = g - r
    nref = np.linalg.norm(r.ravel())
    rel = np.linalg.norm(d.ravel()) / nref if nref > 0 else np.linalg.norm(d.ravel())
    return float(rel), float(np.abs(d).max())


def assert_close(name, gpu, ref, T, rel_tol=REL_L2, abs_tol=None, scale_by_rms=False):
    """scale_by_rms: the max-abs bound is taken relative to the reference's RMS
    when that exceeds 1.  Used only for recurrences without a contracting gate
    (a rotation-only transition), whose states and adjoints grow like sqrt(T),
    so that a fixed absolute bound would test the magnitude, not the error."""
    rel, mx = errors(gpu, ref)
    lim = abs_tol if abs_tol is not None else ABS_PER_SQRT_T * math.sqrt(max(T, 1))
    if scale_by_rms and abs_tol is None:
        r = np.asarray(ref, np.float64)
        rms = float(np.sqrt(np.mean(r * r))) if r.size else 0.0
        lim *= max(1.0, rms)
    assert np.isfinite(rel) and rel <= rel_tol and mx <= lim, \
        f"{name}: rel_l2={rel:.3e} (<= {rel_tol:.1e}), max_abs={mx:.3e} (<= {lim:.2e})"
    return rel, mx
