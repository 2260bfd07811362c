"""ctypes binding of libmgscan (include/mgscan.h).

Argument marshalling only: every function here converts tensors/ints to raw
pointers and sizes and calls the C entry point of the same name.  All
arithmetic runs in the CUDA library; if the library is missing the call raises
instead of computing anything another way.
"""
from __future__ import annotations

import ctypes
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmgscan.so")
HEADER_PATH = os.path.join(os.path.dirname(_PKG), "include", "mgscan.h")

MGS_OK = 0
MGS_ERR_INVALID_ARG = 1
MGS_ERR_UNSUPPORTED = 2
MGS_ERR_WORKSPACE = 3
MGS_ERR_CUDA = 4
MGS_ERR_TIMEOUT = 5
STATUS_NAMES = {0: "MGS_OK", 1: "MGS_ERR_INVALID_ARG", 2: "MGS_ERR_UNSUPPORTED",
                3: "MGS_ERR_WORKSPACE", 4: "MGS_ERR_CUDA", 5: "MGS_ERR_TIMEOUT"}

MGS_OP_MATRIX_AFFINE_SCAN_FWD = 1
MGS_OP_MATRIX_AFFINE_SCAN_BWD = 2
MGS_OP_MATRIX_SCAN_FWD = 3
MGS_OP_MATRIX_SCAN_BWD = 4
MGS_OP_PARALLEL_SCAN_LOG_FWD = 5
MGS_OP_PARALLEL_SCAN_LOG_BWD = 6
MGS_OP_LINEAR_SCAN_FWD = 7
MGS_OP_LINEAR_SCAN_BWD = 8
MGS_OP_GIVENS_AFFINE_SCAN_FWD = 9
MGS_OP_GIVENS_AFFINE_SCAN_BWD = 10
MGS_OP_GIVENS_MATRIX_SCAN_FWD = 11
MGS_OP_GIVENS_MATRIX_SCAN_BWD = 12
MGS_OP_DELTA_SCAN_FWD = 13
MGS_OP_MATRIX_AFFINE_SCAN_BWD_RECOMPUTE = 14


class MGSError(RuntimeError):
    """A libmgscan entry point returned a status other than MGS_OK."""

    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} returned {STATUS_NAMES.get(status, status)}")
        self.status = status


_lock = threading.Lock()
_lib = None

_vp = ctypes.c_void_p
_i64 = ctypes.c_int64
_int = ctypes.c_int
_sz = ctypes.c_size_t
_SIGNATURES = {
    "mgs_workspace_size": (_sz, [_int, _i64, _i64, _i64, _int]),
    "mgs_matrix_affine_scan_fwd": (_int, [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _int, _vp, _sz, _vp]),
    "mgs_matrix_affine_scan_bwd": (_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _int, _vp, _sz, _vp]),
    "mgs_matrix_affine_scan_bwd_recompute": (_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _int, _vp,
                                                    _sz, _vp]),
    "mgs_matrix_scan_fwd": (_int, [_vp, _vp, _i64, _i64, _i64, _int, _vp, _sz, _vp]),
    "mgs_matrix_scan_fwd_noalloc": (_int, [_vp, _vp, _i64, _i64, _i64, _int, _vp]),
    "mgs_matrix_scan_bwd": (_int, [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _int, _vp, _sz, _vp]),
    "mgs_parallel_scan_log_fwd": (_int, [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _vp, _sz, _vp]),
    "mgs_parallel_scan_log_bwd": (_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _vp, _sz, _vp]),
    "mgs_linear_scan_fwd": (_int, [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _vp, _sz, _vp]),
    "mgs_linear_scan_bwd": (_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _vp, _sz, _vp]),
    "mgs_givens_affine_scan_fwd": (_int, [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _int, _vp, _sz, _vp]),
    "mgs_givens_affine_scan_bwd": (_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _int,
                                          _vp, _sz, _vp]),
    "mgs_givens_matrix_scan_fwd": (_int, [_vp, _vp, _i64, _i64, _i64, _int, _vp, _sz, _vp]),
    "mgs_givens_matrix_scan_bwd": (_int, [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _int, _vp, _sz, _vp]),
    "mgs_delta_scan_fwd": (_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _int, _vp, _sz, _vp]),
    "mgs_check": (_int, [_vp]),
    "mgs_set_wait_timeout_ns": (None, [ctypes.c_uint64]),
    "mgs_debug_wait_flag": (_int, [_vp, _vp]),
    "mgs_status_string": (ctypes.c_char_p, [_int]),
    "mgs_version": (_int, []),
}


def lib():
    """The loaded CUDA library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it with scan_linear_recurrences_gb300.build.build() "
                    "(nvcc, sm_103a); there is no other implementation to fall back to")
            L = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in _SIGNATURES.items():
                f = getattr(L, name)
                f.restype = res
                f.argtypes = args
            _lib = L
    return _lib


def exported_symbols():
    """Names declared in the C header (used to check the library's exports)."""
    return list(_SIGNATURES)


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _call(name, *args):
    st = getattr(lib(), name)(*args)
    if st != MGS_OK:
        raise MGSError(name, st)
    return st


# ---------------------------------------------------------------- raw entry points
def mgs_workspace_size(op, B, T, H_or_D, k):
    return int(lib().mgs_workspace_size(op, B, T, H_or_D, k))


def mgs_matrix_affine_scan_fwd(A, b, h0, h, B, T, H, k, workspace=None, workspace_bytes=0, stream=None):
    return _call("mgs_matrix_affine_scan_fwd", _ptr(A), _ptr(b), _ptr(h0), _ptr(h), B, T, H, k,
                 _ptr(workspace), workspace_bytes, _stream(stream))


def mgs_matrix_affine_scan_bwd(A, h0, h, grad_h, dA, db, dh0, B, T, H, k, workspace=None,
                               workspace_bytes=0, stream=None):
    return _call("mgs_matrix_affine_scan_bwd", _ptr(A), _ptr(h0), _ptr(h), _ptr(grad_h), _ptr(dA),
                 _ptr(db), _ptr(dh0), B, T, H, k, _ptr(workspace), workspace_bytes, _stream(stream))


def mgs_matrix_affine_scan_bwd_recompute(A, b, h0, grad_h, dA, db, dh0, B, T, H, k, workspace=None,
                                         workspace_bytes=0, stream=None):
    return _call("mgs_matrix_affine_scan_bwd_recompute", _ptr(A), _ptr(b), _ptr(h0), _ptr(grad_h), _ptr(dA),
                 _ptr(db), _ptr(dh0), B, T, H, k, _ptr(workspace), workspace_bytes, _stream(stream))


def mgs_matrix_scan_fwd(A, P, B, T, H, k, workspace=None, workspace_bytes=0, stream=None):
    return _call("mgs_matrix_scan_fwd", _ptr(A), _ptr(P), B, T, H, k, _ptr(workspace), workspace_bytes,
                 _stream(stream))


def mgs_matrix_scan_fwd_noalloc(A, P, B, T, H, k, stream=None):
    """matrix_scan forward using the library's built-in device scratch; for
    callers that cannot allocate device memory (see include/mgscan.h)."""
    return _call("mgs_matrix_scan_fwd_noalloc", _ptr(A), _ptr(P), B, T, H, k, _stream(stream))


NOALLOC_SCRATCH_BYTES = 4 << 20  # MGS_NOALLOC_SCRATCH_BYTES in include/mgscan.h


def mgs_matrix_scan_bwd(A, P, grad_P, dA, B, T, H, k, workspace=None, workspace_bytes=0, stream=None):
    return _call("mgs_matrix_scan_bwd", _ptr(A), _ptr(P), _ptr(grad_P), _ptr(dA), B, T, H, k,
                 _ptr(workspace), workspace_bytes, _stream(stream))


def mgs_parallel_scan_log_fwd(log_coeffs, log_values, log_h0, h, log_h, B, T, D, workspace=None,
                              workspace_bytes=0, stream=None):
    return _call("mgs_parallel_scan_log_fwd", _ptr(log_coeffs), _ptr(log_values), _ptr(log_h0), _ptr(h),
                 _ptr(log_h), B, T, D, _ptr(workspace), workspace_bytes, _stream(stream))


def mgs_parallel_scan_log_bwd(log_coeffs, log_values, log_h0, h, grad_h, d_log_coeffs, d_log_values,
                              d_log_h0, B, T, D, workspace=None, workspace_bytes=0, stream=None):
    return _call("mgs_parallel_scan_log_bwd", _ptr(log_coeffs), _ptr(log_values), _ptr(log_h0), _ptr(h),
                 _ptr(grad_h), _ptr(d_log_coeffs), _ptr(d_log_values), _ptr(d_log_h0), B, T, D,
                 _ptr(workspace), workspace_bytes, _stream(stream))


def mgs_linear_scan_fwd(a, b, h0, h, B, T, D, workspace=None, workspace_bytes=0, stream=None):
    return _call("mgs_linear_scan_fwd", _ptr(a), _ptr(b), _ptr(h0), _ptr(h), B, T, D, _ptr(workspace),
                 workspace_bytes, _stream(stream))


def mgs_linear_scan_bwd(a, h0, h, grad_h, da, db, dh0, B, T, D, workspace=None, workspace_bytes=0, stream=None):
    return _call("mgs_linear_scan_bwd", _ptr(a), _ptr(h0), _ptr(h), _ptr(grad_h), _ptr(da), _ptr(db), _ptr(dh0),
                 B, T, D, _ptr(workspace), workspace_bytes, _stream(stream))


def mgs_givens_affine_scan_fwd(theta, a, b, h0, h, B, T, H, k, workspace=None, workspace_bytes=0, stream=None):
    return _call("mgs_givens_affine_scan_fwd", _ptr(theta), _ptr(a), _ptr(b), _ptr(h0), _ptr(h), B, T, H, k,
                 _ptr(workspace), workspace_bytes, _stream(stream))


def mgs_givens_affine_scan_bwd(theta, a, h0, h, grad_h, d_theta, da, db, dh0, B, T, H, k, workspace=None,
                               workspace_bytes=0, stream=None):
    return _call("mgs_givens_affine_scan_bwd", _ptr(theta), _ptr(a), _ptr(h0), _ptr(h), _ptr(grad_h),
                 _ptr(d_theta), _ptr(da), _ptr(db), _ptr(dh0), B, T, H, k, _ptr(workspace), workspace_bytes,
                 _stream(stream))


def mgs_givens_matrix_scan_fwd(theta, P, B, T, H, k, workspace=None, workspace_bytes=0, stream=None):
    return _call("mgs_givens_matrix_scan_fwd", _ptr(theta), _ptr(P), B, T, H, k, _ptr(workspace),
                 workspace_bytes, _stream(stream))


def mgs_givens_matrix_scan_bwd(theta, P, grad_P, d_theta, B, T, H, k, workspace=None, workspace_bytes=0,
                               stream=None):
    return _call("mgs_givens_matrix_scan_bwd", _ptr(theta), _ptr(P), _ptr(grad_P), _ptr(d_theta), B, T, H, k,
                 _ptr(workspace), workspace_bytes, _stream(stream))


def mgs_delta_scan_fwd(q, k, v, beta, S0, o, S_T, B, T, H, D, workspace=None, workspace_bytes=0, stream=None):
    return _call("mgs_delta_scan_fwd", _ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(S0), _ptr(o), _ptr(S_T),
                 B, T, H, D, _ptr(workspace), workspace_bytes, _stream(stream))


def mgs_check(stream=None):
    return _call("mgs_check", _stream(stream))


def mgs_set_wait_timeout_ns(ns: int):
    lib().mgs_set_wait_timeout_ns(int(ns))


def mgs_debug_wait_flag(flag, stream=None):
    return _call("mgs_debug_wait_flag", _ptr(flag), _stream(stream))


def mgs_status_string(status: int) -> str:
    return lib().mgs_status_string(status).decode()


def mgs_version() -> int:
    return int(lib().mgs_version())
