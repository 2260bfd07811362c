"""Float64 CPU oracle for matrix_affine_scan, matrix_scan, parallel_scan_log,
linear_scan, the Givens-mesh (angle-parameterised) affine and matrix scans and
the delta rule (DeltaNet) forward.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this package.  The
product library never loads it, and it shares no code with the CUDA path.

The arithmetic lives in ``mgs_oracle.c`` (plain sequential loops in double,
one lane at a time).  This module only compiles that file with gcc (once, into
``oracle/_build``), loads it with ctypes and marshals numpy arrays.  Inputs are
upcast to float64 (exact for the float32 buffers the GPU receives); outputs are
float64.

Each function's definition and source are documented in ``mgs_oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mgs_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "libmgs_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``mgs_oracle.c`` into a shared object (gcc, OpenMP). Returns its path."""
    os.makedirs(_BUILD, exist_ok=True)
    stale = (not os.path.exists(_LIB)) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-std=c11", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            # MGS_ORACLE_LIB points the loader at another build of mgs_oracle.c;
            # the mutation tests use it to run the pins against planted mistakes.
            lib = ctypes.CDLL(os.environ.get("MGS_ORACLE_LIB") or build())
            dp = ctypes.POINTER(ctypes.c_double)
            i64 = ctypes.c_int64
            lib.oracle_mas_fwd.argtypes = [dp, dp, dp, dp, i64, i64, i64, i64]
            lib.oracle_mas_bwd.argtypes = [dp, dp, dp, dp, dp, dp, dp, i64, i64, i64, i64]
            lib.oracle_ms_fwd.argtypes = [dp, dp, i64, i64, i64, i64]
            lib.oracle_ms_bwd.argtypes = [dp, dp, dp, i64, i64, i64, i64]
            lib.oracle_psl_fwd.argtypes = [dp, dp, dp, dp, dp, i64, i64, i64]
            lib.oracle_psl_bwd.argtypes = [dp, dp, dp, dp, dp, dp, dp, i64, i64, i64]
            lib.oracle_linear_fwd.argtypes = [dp, dp, dp, dp, i64, i64, i64]
            lib.oracle_linear_bwd.argtypes = [dp, dp, dp, dp, dp, dp, dp, i64, i64, i64]
            lib.oracle_gas_fwd.argtypes = [dp, dp, dp, dp, dp, i64, i64, i64, i64]
            lib.oracle_gas_bwd.argtypes = [dp, dp, dp, dp, dp, dp, dp, dp, dp, i64, i64, i64, i64]
            lib.oracle_gms_fwd.argtypes = [dp, dp, i64, i64, i64, i64]
            lib.oracle_gms_bwd.argtypes = [dp, dp, dp, i64, i64, i64, i64]
            lib.oracle_delta_fwd.argtypes = [dp, dp, dp, dp, dp, dp, dp, i64, i64, i64, i64]
            lib.oracle_num_threads.restype = ctypes.c_int
            for f in ("oracle_mas_fwd", "oracle_mas_bwd", "oracle_ms_fwd", "oracle_ms_bwd",
                      "oracle_psl_fwd", "oracle_psl_bwd", "oracle_linear_fwd", "oracle_linear_bwd",
                      "oracle_gas_fwd", "oracle_gas_bwd", "oracle_gms_fwd", "oracle_gms_bwd",
                      "oracle_delta_fwd"):
                getattr(lib, f).restype = None
            _lib = lib
    return _lib


def _f64(x):
    """Contiguous float64 copy/view of an array-like (None passes through)."""
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor
        x = x.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _p(a):
    if a is None:
        return ctypes.POINTER(ctypes.c_double)()
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def num_threads() -> int:
    """Host threads the oracle's lane loops run on."""
    return int(_load().oracle_num_threads())


# ---------------------------------------------------------------- mas
def mas_fwd(A, b, h0=None):
    """h_t = A_t h_{t-1} + b_t.  A [B,T,H,K,K], b [B,T,H,K], h0 [B,H,K] or None -> h [B,T,H,K]."""
    A, b, h0 = _f64(A), _f64(b), _f64(h0)
    B, T, H, K = b.shape
    assert A.shape == (B, T, H, K, K)
    assert h0 is None or h0.shape == (B, H, K)
    h = np.empty((B, T, H, K), dtype=np.float64)
    _load().oracle_mas_fwd(_p(A), _p(b), _p(h0), _p(h), B, T, H, K)
    return h


def mas_bwd(A, b, h0, grad_h):
    """Gradients of sum <grad_h, h> -> (dA, db, dh0); dh0 is None when h0 is None."""
    A, b, h0, g = _f64(A), _f64(b), _f64(h0), _f64(grad_h)
    B, T, H, K = b.shape
    assert A.shape == (B, T, H, K, K) and g.shape == (B, T, H, K)
    dA = np.empty_like(A)
    db = np.empty_like(b)
    dh0 = np.empty((B, H, K), dtype=np.float64) if h0 is not None else None
    _load().oracle_mas_bwd(_p(A), _p(b), _p(h0), _p(g), _p(dA), _p(db), _p(dh0), B, T, H, K)
    return dA, db, dh0


# ---------------------------------------------------------------- ms
def ms_fwd(A):
    """P_t = A_t P_{t-1}, P_0 = I.  A [B,T,H,K,K] -> P [B,T,H,K,K]."""
    A = _f64(A)
    B, T, H, K, K2 = A.shape
    assert K == K2
    P = np.empty_like(A)
    _load().oracle_ms_fwd(_p(A), _p(P), B, T, H, K)
    return P


def ms_bwd(A, grad_P):
    """Gradient of sum <grad_P, P>_F with respect to A -> dA [B,T,H,K,K]."""
    A, G = _f64(A), _f64(grad_P)
    B, T, H, K, _ = A.shape
    assert G.shape == A.shape
    dA = np.empty_like(A)
    _load().oracle_ms_bwd(_p(A), _p(G), _p(dA), B, T, H, K)
    return dA


# ---------------------------------------------------------------- psl
def psl_fwd(log_coeffs, log_values, log_h0=None, want_log=False):
    """Log-space diagonal scan.  lc, lv [B,T,D], log_h0 [B,D] or None -> h (and log h)."""
    lc, lv, l0 = _f64(log_coeffs), _f64(log_values), _f64(log_h0)
    B, T, D = lc.shape
    assert lv.shape == (B, T, D) and (l0 is None or l0.shape == (B, D))
    h = np.empty((B, T, D), dtype=np.float64)
    lh = np.empty((B, T, D), dtype=np.float64) if want_log else None
    _load().oracle_psl_fwd(_p(lc), _p(lv), _p(l0), _p(h), _p(lh), B, T, D)
    return (h, lh) if want_log else h


def psl_bwd(log_coeffs, log_values, log_h0, grad_h):
    """Gradients of sum grad_h * h -> (d_log_coeffs, d_log_values, d_log_h0 or None)."""
    lc, lv, l0, g = _f64(log_coeffs), _f64(log_values), _f64(log_h0), _f64(grad_h)
    B, T, D = lc.shape
    dlc = np.empty_like(lc)
    dlv = np.empty_like(lv)
    dl0 = np.empty((B, D), dtype=np.float64) if l0 is not None else None
    _load().oracle_psl_bwd(_p(lc), _p(lv), _p(l0), _p(g), _p(dlc), _p(dlv), _p(dl0), B, T, D)
    return dlc, dlv, dl0


# ---------------------------------------------------------------- linear_scan
def linear_fwd(a, b, h0=None):
    """h_t = a_t h_{t-1} + b_t elementwise.  a, b [B,T,D], h0 [B,D] or None -> h."""
    a, b, h0 = _f64(a), _f64(b), _f64(h0)
    B, T, D = a.shape
    assert b.shape == (B, T, D) and (h0 is None or h0.shape == (B, D))
    h = np.empty((B, T, D), dtype=np.float64)
    _load().oracle_linear_fwd(_p(a), _p(b), _p(h0), _p(h), B, T, D)
    return h


def linear_bwd(a, b, h0, grad_h, want_dh0=True):
    """Gradients of sum grad_h * h -> (da, db, dh0 or None)."""
    a, b, h0, g = _f64(a), _f64(b), _f64(h0), _f64(grad_h)
    B, T, D = a.shape
    da = np.empty_like(a)
    db = np.empty_like(a)
    dh0 = np.empty((B, D), dtype=np.float64) if want_dh0 else None
    _load().oracle_linear_bwd(_p(a), _p(b), _p(h0), _p(g), _p(da), _p(db), _p(dh0), B, T, D)
    return da, db, dh0


# ---------------------------------------------------------------- Givens mesh
def n_angles(K):
    """Angles of the K-coordinate brick-wall mesh: K(K-1)/2."""
    return K * (K - 1) // 2


def _k_of(N):
    K = int(round((1 + (1 + 8 * N) ** 0.5) / 2))
    assert n_angles(K) == N, f"{N} is not K(K-1)/2"
    return K


def gas_fwd(theta, a, b, h0=None):
    """h_t = G(theta_t) diag(a_t) h_{t-1} + b_t.  theta [B,T,H,N], a [B,T,H,K] or None,
    b [B,T,H,K], h0 [B,H,K] or None -> h [B,T,H,K]."""
    th, a, b, h0 = _f64(theta), _f64(a), _f64(b), _f64(h0)
    B, T, H, K = b.shape
    assert th.shape == (B, T, H, n_angles(K)) and (a is None or a.shape == b.shape)
    assert h0 is None or h0.shape == (B, H, K)
    h = np.empty((B, T, H, K), dtype=np.float64)
    _load().oracle_gas_fwd(_p(th), _p(a), _p(b), _p(h0), _p(h), B, T, H, K)
    return h


def gas_bwd(theta, a, b, h0, grad_h):
    """Gradients of sum <grad_h, h> -> (dtheta, da or None, db, dh0 or None)."""
    th, a, b, h0, g = _f64(theta), _f64(a), _f64(b), _f64(h0), _f64(grad_h)
    B, T, H, K = b.shape
    assert th.shape == (B, T, H, n_angles(K)) and g.shape == b.shape
    dth = np.empty_like(th)
    da = np.empty_like(b) if a is not None else None
    db = np.empty_like(b)
    dh0 = np.empty((B, H, K), dtype=np.float64) if h0 is not None else None
    _load().oracle_gas_bwd(_p(th), _p(a), _p(b), _p(h0), _p(g), _p(dth), _p(da), _p(db), _p(dh0),
                           B, T, H, K)
    return dth, da, db, dh0


def gms_fwd(theta):
    """P_t = G(theta_t) P_{t-1}, P_0 = I.  theta [B,T,H,N] -> P [B,T,H,K,K]."""
    th = _f64(theta)
    B, T, H, N = th.shape
    K = _k_of(N)
    P = np.empty((B, T, H, K, K), dtype=np.float64)
    _load().oracle_gms_fwd(_p(th), _p(P), B, T, H, K)
    return P


def gms_bwd(theta, grad_P):
    """Gradient of sum <grad_P, P>_F with respect to the angles -> dtheta [B,T,H,N]."""
    th, G = _f64(theta), _f64(grad_P)
    B, T, H, N = th.shape
    K = _k_of(N)
    assert G.shape == (B, T, H, K, K)
    dth = np.empty_like(th)
    _load().oracle_gms_bwd(_p(th), _p(G), _p(dth), B, T, H, K)
    return dth


# ---------------------------------------------------------------- delta rule
def delta_fwd(q, k, v, beta, S0=None, want_state=False):
    """S_t = S_{t-1} + beta_t (v_t - S_{t-1} k_t) k_t^T, o_t = S_t q_t.
    q, k, v [B,T,H,D], beta [B,T,H], S0 [B,H,D,D] or None -> o (and S_T)."""
    q, k, v, beta, S0 = _f64(q), _f64(k), _f64(v), _f64(beta), _f64(S0)
    B, T, H, D = q.shape
    assert k.shape == q.shape and v.shape == q.shape and beta.shape == (B, T, H)
    assert S0 is None or S0.shape == (B, H, D, D)
    o = np.empty_like(q)
    ST = np.empty((B, H, D, D), dtype=np.float64) if want_state else None
    _load().oracle_delta_fwd(_p(q), _p(k), _p(v), _p(beta), _p(S0), _p(o), _p(ST), B, T, H, D)
    return (o, ST) if want_state else o
