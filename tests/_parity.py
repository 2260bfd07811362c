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


def assert_close(name, gpu, ref, T, rel_tol=REL_L2, abs_tol=None):
    rel, mx = errors(gpu, ref)
    lim = abs_tol if abs_tol is not None else ABS_PER_SQRT_T * math.sqrt(max(T, 1))
    assert np.isfinite(rel) and rel <= rel_tol and mx <= lim, \
        f"{name}: rel_l2={rel:.3e} (<= {rel_tol:.1e}), max_abs={mx:.3e} (<= {lim:.2e})"
    return rel, mx


class Streamed:
    """Relative L2 and max-abs of one output tensor compared part by part (for
    outputs too large to hold in float64 at once): the squared norms and the
    maximum accumulate over the parts, then check() applies the same bounds
    as assert_close to the whole tensor."""

    def __init__(self, name):
        self.name, self.d2, self.r2, self.mx, self.n = name, 0.0, 0.0, 0.0, 0

    def add(self, gpu, ref):
        g = gpu.detach().double().cpu().numpy() if hasattr(gpu, "detach") else np.asarray(gpu, np.float64)
        r = np.asarray(ref, np.float64)
        assert g.shape == r.shape, (g.shape, r.shape)
        d = g - r
        self.d2 += float(np.sum(d * d))
        self.r2 += float(np.sum(r * r))
        if d.size:
            self.mx = max(self.mx, float(np.abs(d).max()))
        self.n += r.size

    def check(self, T, rel_tol=REL_L2):
        rel = math.sqrt(self.d2 / self.r2) if self.r2 > 0 else math.sqrt(self.d2)
        lim = ABS_PER_SQRT_T * math.sqrt(max(T, 1))
        assert np.isfinite(rel) and rel <= rel_tol and self.mx <= lim, \
            f"{self.name}: rel_l2={rel:.3e} (<= {rel_tol:.1e}), max_abs={self.mx:.3e} (<= {lim:.2e})"
        return rel, self.mx
