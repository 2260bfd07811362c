"""Tensor-level API over the C ABI: shape checks, output/workspace allocation
with torch (device memory is torch's job here), then one libmgscan call.

Also provides ``torch.autograd.Function`` wrappers whose forward and backward
are the library's fwd/bwd entry points, for use inside models.
"""
from __future__ import annotations

import torch

from . import _binding as _b


def _check(t, name, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor (the library runs only on the GPU)")
    if t.dtype != torch.float32:
        raise ValueError(f"{name} must be float32")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def workspace(op, B, T, H_or_D, k, device):
    """A workspace tensor of the size the op needs (None when it needs none)."""
    n = _b.mgs_workspace_size(op, B, T, H_or_D, k)
    if n == 0:
        return None, 0
    return torch.empty(n, dtype=torch.uint8, device=device), n


# ---------------------------------------------------------------- matrix_affine_scan
def matrix_affine_scan_fwd(A, b, h0=None, out=None, stream=None):
    """h_t = A_t h_{t-1} + b_t.  A [B,T,H,k,k], b [B,T,H,k], h0 [B,H,k] or None."""
    B, T, H, k = b.shape
    _check(A, "A", (B, T, H, k, k)); _check(b, "b")
    if h0 is not None:
        _check(h0, "h0", (B, H, k))
    h = out if out is not None else torch.empty_like(b)
    ws, nws = workspace(_b.MGS_OP_MATRIX_AFFINE_SCAN_FWD, B, T, H, k, b.device)
    _b.mgs_matrix_affine_scan_fwd(A, b, h0, h, B, T, H, k, ws, nws, stream)
    return h


def matrix_affine_scan_bwd(A, h0, h, grad_h, need_dh0=True, stream=None):
    """Returns (dA, db, dh0) for L = sum <grad_h, h>; dh0 is None unless requested."""
    B, T, H, k = h.shape
    _check(A, "A", (B, T, H, k, k)); _check(h, "h"); _check(grad_h, "grad_h", (B, T, H, k))
    if h0 is not None:
        _check(h0, "h0", (B, H, k))
    dA = torch.empty_like(A)
    db = torch.empty_like(h)
    dh0 = torch.empty((B, H, k), dtype=torch.float32, device=h.device) if need_dh0 else None
    ws, nws = workspace(_b.MGS_OP_MATRIX_AFFINE_SCAN_BWD, B, T, H, k, h.device)
    _b.mgs_matrix_affine_scan_bwd(A, h0, h, grad_h, dA, db, dh0, B, T, H, k, ws, nws, stream)
    return dA, db, dh0


def matrix_affine_scan_bwd_recompute(A, b, h0, grad_h, need_dh0=True, stream=None):
    """The same gradients as matrix_affine_scan_bwd without the saved h: the
    call recomputes the forward from A, b and h0 (checkpoints in a workspace)."""
    B, T, H, k = b.shape
    _check(A, "A", (B, T, H, k, k)); _check(b, "b"); _check(grad_h, "grad_h", (B, T, H, k))
    if h0 is not None:
        _check(h0, "h0", (B, H, k))
    dA = torch.empty_like(A)
    db = torch.empty_like(b)
    dh0 = torch.empty((B, H, k), dtype=torch.float32, device=b.device) if need_dh0 else None
    ws, nws = workspace(_b.MGS_OP_MATRIX_AFFINE_SCAN_BWD_RECOMPUTE, B, T, H, k, b.device)
    _b.mgs_matrix_affine_scan_bwd_recompute(A, b, h0, grad_h, dA, db, dh0, B, T, H, k, ws, nws, stream)
    return dA, db, dh0


# ---------------------------------------------------------------- matrix_scan
def matrix_scan_fwd(A, out=None, stream=None):
    """P_t = A_t P_{t-1}, P_0 = I.  A [B,T,H,k,k]."""
    B, T, H, k, _ = A.shape
    _check(A, "A", (B, T, H, k, k))
    P = out if out is not None else torch.empty_like(A)
    ws, nws = workspace(_b.MGS_OP_MATRIX_SCAN_FWD, B, T, H, k, A.device)
    _b.mgs_matrix_scan_fwd(A, P, B, T, H, k, ws, nws, stream)
    return P


def matrix_scan_bwd(A, P, grad_P, stream=None):
    B, T, H, k, _ = A.shape
    _check(A, "A", (B, T, H, k, k)); _check(P, "P", A.shape); _check(grad_P, "grad_P", A.shape)
    dA = torch.empty_like(A)
    ws, nws = workspace(_b.MGS_OP_MATRIX_SCAN_BWD, B, T, H, k, A.device)
    _b.mgs_matrix_scan_bwd(A, P, grad_P, dA, B, T, H, k, ws, nws, stream)
    return dA


# ---------------------------------------------------------------- parallel_scan_log
def parallel_scan_log_fwd(log_coeffs, log_values, log_h0=None, want_log=False, stream=None):
    """Heinsen log-space scan; returns h (and log h when want_log)."""
    B, T, D = log_coeffs.shape
    _check(log_coeffs, "log_coeffs"); _check(log_values, "log_values", (B, T, D))
    if log_h0 is not None:
        _check(log_h0, "log_h0", (B, D))
    h = torch.empty_like(log_coeffs)
    lh = torch.empty_like(log_coeffs) if want_log else None
    _b.mgs_parallel_scan_log_fwd(log_coeffs, log_values, log_h0, h, lh, B, T, D, None, 0, stream)
    return (h, lh) if want_log else h


def parallel_scan_log_bwd(log_coeffs, log_values, log_h0, h, grad_h, stream=None):
    """Returns (d_log_coeffs, d_log_values, d_log_h0 or None).

    h is the saved forward output, or None to recompute it inside the call
    (checkpoints every 16 steps in a workspace of 4*B*ceil(T/16)*D bytes)."""
    B, T, D = log_coeffs.shape
    for t, n in ((log_coeffs, "log_coeffs"), (log_values, "log_values"), (grad_h, "grad_h")):
        _check(t, n, (B, T, D))
    if h is not None:
        _check(h, "h", (B, T, D))
    if log_h0 is not None:
        _check(log_h0, "log_h0", (B, D))
    dlc = torch.empty_like(log_coeffs)
    dlv = torch.empty_like(log_values)
    dl0 = torch.empty_like(log_h0) if log_h0 is not None else None
    ws, nws = (None, 0) if h is not None else \
        workspace(_b.MGS_OP_PARALLEL_SCAN_LOG_BWD, B, T, D, 0, log_coeffs.device)
    _b.mgs_parallel_scan_log_bwd(log_coeffs, log_values, log_h0, h, grad_h, dlc, dlv, dl0, B, T, D,
                                 ws, nws, stream)
    return dlc, dlv, dl0


# ---------------------------------------------------------------- Givens-mesh scans
GIVENS_K = 8
GIVENS_N = GIVENS_K * (GIVENS_K - 1) // 2


def givens_affine_scan_fwd(theta, a, b, h0=None, stream=None):
    """h_t = G(theta_t) diag(a_t) h_{t-1} + b_t.  theta [B,T,H,28], a [B,T,H,8] or None,
    b [B,T,H,8], h0 [B,H,8] or None."""
    B, T, H, k = b.shape
    _check(theta, "theta", (B, T, H, k * (k - 1) // 2)); _check(b, "b")
    if a is not None:
        _check(a, "a", (B, T, H, k))
    if h0 is not None:
        _check(h0, "h0", (B, H, k))
    h = torch.empty_like(b)
    ws, nws = workspace(_b.MGS_OP_GIVENS_AFFINE_SCAN_FWD, B, T, H, k, b.device)
    _b.mgs_givens_affine_scan_fwd(theta, a, b, h0, h, B, T, H, k, ws, nws, stream)
    return h


def givens_affine_scan_bwd(theta, a, h0, h, grad_h, need_dh0=True, stream=None):
    """Returns (d_theta, da or None, db, dh0 or None) for L = sum <grad_h, h>."""
    B, T, H, k = h.shape
    _check(theta, "theta", (B, T, H, k * (k - 1) // 2)); _check(h, "h"); _check(grad_h, "grad_h", (B, T, H, k))
    if a is not None:
        _check(a, "a", (B, T, H, k))
    if h0 is not None:
        _check(h0, "h0", (B, H, k))
    dth = torch.empty_like(theta)
    da = torch.empty_like(a) if a is not None else None
    db = torch.empty_like(h)
    dh0 = torch.empty((B, H, k), dtype=torch.float32, device=h.device) if need_dh0 else None
    ws, nws = workspace(_b.MGS_OP_GIVENS_AFFINE_SCAN_BWD, B, T, H, k, h.device)
    _b.mgs_givens_affine_scan_bwd(theta, a, h0, h, grad_h, dth, da, db, dh0, B, T, H, k, ws, nws, stream)
    return dth, da, db, dh0


def givens_matrix_scan_fwd(theta, k=GIVENS_K, stream=None):
    """P_t = G(theta_t) P_{t-1}, P_0 = I.  theta [B,T,H,28] -> P [B,T,H,8,8]."""
    B, T, H, n = theta.shape
    _check(theta, "theta", (B, T, H, k * (k - 1) // 2))
    P = torch.empty((B, T, H, k, k), dtype=torch.float32, device=theta.device)
    ws, nws = workspace(_b.MGS_OP_GIVENS_MATRIX_SCAN_FWD, B, T, H, k, theta.device)
    _b.mgs_givens_matrix_scan_fwd(theta, P, B, T, H, k, ws, nws, stream)
    return P


def givens_matrix_scan_bwd(theta, P, grad_P, stream=None):
    B, T, H, k, _ = P.shape
    _check(theta, "theta", (B, T, H, k * (k - 1) // 2)); _check(P, "P"); _check(grad_P, "grad_P", P.shape)
    dth = torch.empty_like(theta)
    ws, nws = workspace(_b.MGS_OP_GIVENS_MATRIX_SCAN_BWD, B, T, H, k, theta.device)
    _b.mgs_givens_matrix_scan_bwd(theta, P, grad_P, dth, B, T, H, k, ws, nws, stream)
    return dth


# ---------------------------------------------------------------- delta rule
def delta_scan_fwd(q, k, v, beta, S0=None, want_state=False, stream=None):
    """DeltaNet's delta rule: S_t = S_{t-1} + beta_t (v_t - S_{t-1} k_t) k_t^T,
    o_t = S_t q_t.  q, k, v [B,T,H,64], beta [B,T,H], S0 [B,H,64,64] or None.
    Returns o (and the final state when want_state)."""
    B, T, H, D = q.shape
    _check(q, "q"); _check(k, "k", q.shape); _check(v, "v", q.shape); _check(beta, "beta", (B, T, H))
    if S0 is not None:
        _check(S0, "S0", (B, H, D, D))
    o = torch.empty_like(q)
    ST = torch.empty((B, H, D, D), dtype=torch.float32, device=q.device) if want_state else None
    ws, nws = workspace(_b.MGS_OP_DELTA_SCAN_FWD, B, T, H, D, q.device)
    _b.mgs_delta_scan_fwd(q, k, v, beta, S0, o, ST, B, T, H, D, ws, nws, stream)
    return (o, ST) if want_state else o


# ---------------------------------------------------------------- linear_scan
def linear_scan_fwd(a, b, h0=None, stream=None):
    """h_t = a_t * h_{t-1} + b_t elementwise.  a, b [B,T,D], h0 [B,D] or None."""
    B, T, D = a.shape
    _check(a, "a"); _check(b, "b", (B, T, D))
    if h0 is not None:
        _check(h0, "h0", (B, D))
    h = torch.empty_like(b)
    ws, nws = workspace(_b.MGS_OP_LINEAR_SCAN_FWD, B, T, D, 1, b.device)
    _b.mgs_linear_scan_fwd(a, b, h0, h, B, T, D, ws, nws, stream)
    return h


def linear_scan_bwd(a, h0, h, grad_h, need_dh0=True, stream=None):
    """Returns (da, db, dh0 or None) for L = sum grad_h * h."""
    B, T, D = a.shape
    for t, n in ((a, "a"), (h, "h"), (grad_h, "grad_h")):
        _check(t, n, (B, T, D))
    if h0 is not None:
        _check(h0, "h0", (B, D))
    da, db = torch.empty_like(a), torch.empty_like(a)
    dh0 = torch.empty((B, D), dtype=torch.float32, device=a.device) if need_dh0 else None
    ws, nws = workspace(_b.MGS_OP_LINEAR_SCAN_BWD, B, T, D, 1, a.device)
    _b.mgs_linear_scan_bwd(a, h0, h, grad_h, da, db, dh0, B, T, D, ws, nws, stream)
    return da, db, dh0


# ---------------------------------------------------------------- autograd wrappers
class MatrixAffineScan(torch.autograd.Function):
    """h = matrix_affine_scan(A, b, h0) with the library's fused backward;
    recompute=True saves b instead of h and the backward rebuilds h."""

    @staticmethod
    def forward(ctx, A, b, h0=None, recompute=False):
        A, b = A.contiguous(), b.contiguous()
        h0c = h0.contiguous() if h0 is not None else None
        h = matrix_affine_scan_fwd(A, b, h0c)
        ctx.save_for_backward(A, h0c if h0c is not None else torch.empty(0, device=b.device), b if recompute else h)
        ctx.has_h0 = h0 is not None
        ctx.recompute = recompute
        return h

    @staticmethod
    def backward(ctx, grad_h):
        A, h0, x = ctx.saved_tensors
        h0 = h0 if ctx.has_h0 else None
        if ctx.recompute:
            dA, db, dh0 = matrix_affine_scan_bwd_recompute(A, x, h0, grad_h.contiguous(), need_dh0=ctx.has_h0)
        else:
            dA, db, dh0 = matrix_affine_scan_bwd(A, h0, x, grad_h.contiguous(), need_dh0=ctx.has_h0)
        return dA, db, dh0, None


class MatrixScan(torch.autograd.Function):
    @staticmethod
    def forward(ctx, A):
        A = A.contiguous()
        P = matrix_scan_fwd(A)
        ctx.save_for_backward(A, P)
        return P

    @staticmethod
    def backward(ctx, grad_P):
        A, P = ctx.saved_tensors
        return matrix_scan_bwd(A, P, grad_P.contiguous())


class ParallelScanLog(torch.autograd.Function):
    @staticmethod
    def forward(ctx, log_coeffs, log_values, log_h0=None, recompute=False):
        lc, lv = log_coeffs.contiguous(), log_values.contiguous()
        l0 = log_h0.contiguous() if log_h0 is not None else None
        h = parallel_scan_log_fwd(lc, lv, l0)
        empty = torch.empty(0, device=lc.device)
        ctx.save_for_backward(lc, lv, l0 if l0 is not None else empty, empty if recompute else h)
        ctx.has_h0 = log_h0 is not None
        ctx.recompute = recompute
        return h

    @staticmethod
    def backward(ctx, grad_h):
        lc, lv, l0, h = ctx.saved_tensors
        l0 = l0 if ctx.has_h0 else None
        h = None if ctx.recompute else h
        dlc, dlv, dl0 = parallel_scan_log_bwd(lc, lv, l0, h, grad_h.contiguous())
        return dlc, dlv, dl0, None


class LinearScan(torch.autograd.Function):
    @staticmethod
    def forward(ctx, a, b, h0=None):
        a, b = a.contiguous(), b.contiguous()
        h0c = h0.contiguous() if h0 is not None else None
        h = linear_scan_fwd(a, b, h0c)
        ctx.save_for_backward(a, h0c if h0c is not None else torch.empty(0, device=a.device), h)
        ctx.has_h0 = h0 is not None
        return h

    @staticmethod
    def backward(ctx, grad_h):
        a, h0, h = ctx.saved_tensors
        h0 = h0 if ctx.has_h0 else None
        da, db, dh0 = linear_scan_bwd(a, h0, h, grad_h.contiguous(), need_dh0=ctx.has_h0)
        return da, db, dh0


class GivensAffineScan(torch.autograd.Function):
    @staticmethod
    def forward(ctx, theta, a, b, h0=None):
        theta, b = theta.contiguous(), b.contiguous()
        a = a.contiguous() if a is not None else None
        h0c = h0.contiguous() if h0 is not None else None
        h = givens_affine_scan_fwd(theta, a, b, h0c)
        empty = torch.empty(0, device=b.device)
        ctx.save_for_backward(theta, a if a is not None else empty, h0c if h0c is not None else empty, h)
        ctx.has_a, ctx.has_h0 = a is not None, h0 is not None
        return h

    @staticmethod
    def backward(ctx, grad_h):
        theta, a, h0, h = ctx.saved_tensors
        a = a if ctx.has_a else None
        h0 = h0 if ctx.has_h0 else None
        dth, da, db, dh0 = givens_affine_scan_bwd(theta, a, h0, h, grad_h.contiguous(), need_dh0=ctx.has_h0)
        return dth, da, db, dh0


class GivensMatrixScan(torch.autograd.Function):
    @staticmethod
    def forward(ctx, theta):
        theta = theta.contiguous()
        P = givens_matrix_scan_fwd(theta)
        ctx.save_for_backward(theta, P)
        return P

    @staticmethod
    def backward(ctx, grad_P):
        theta, P = ctx.saved_tensors
        return givens_matrix_scan_bwd(theta, P, grad_P.contiguous())


def givens_affine_scan(theta, a, b, h0=None):
    """GivensMinGRU's angle-fused recurrence h_t = G(theta_t) diag(a_t) h_{t-1} + b_t (a may be None)."""
    return GivensAffineScan.apply(theta, a, b, h0)


def givens_matrix_scan(theta):
    return GivensMatrixScan.apply(theta)


def linear_scan(a, b, h0=None):
    return LinearScan.apply(a, b, h0)


def matrix_affine_scan(A, b, h0=None, recompute=False):
    """recompute=True keeps b rather than h for backward; backward rebuilds h."""
    return MatrixAffineScan.apply(A, b, h0, recompute)


def matrix_scan(A):
    return MatrixScan.apply(A)


def parallel_scan_log(log_coeffs, log_values, log_h0=None, recompute=False):
    """recompute=True keeps no copy of h for backward; backward rebuilds it."""
    return ParallelScanLog.apply(log_coeffs, log_values, log_h0, recompute)
