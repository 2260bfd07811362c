"""GB300-native scan primitives of the minGRU family (matrix_affine_scan,
matrix_scan, parallel_scan_log), forward and backward, as a C-ABI CUDA
library (libmgscan, include/mgscan.h) with a thin Python binding.

``_binding`` mirrors the C entry points one to one; ``api`` adds tensor-level
helpers and autograd wrappers; ``inputs`` draws the seeded synthetic inputs.
The CUDA library is loaded on first use and its absence is an error.
"""
from ._binding import (MGSError, lib, mgs_check, mgs_debug_wait_flag, mgs_linear_scan_bwd, mgs_linear_scan_fwd, mgs_matrix_affine_scan_bwd,
                       mgs_matrix_affine_scan_fwd, mgs_matrix_scan_bwd, mgs_matrix_scan_fwd, mgs_matrix_scan_fwd_noalloc,
                       mgs_parallel_scan_log_bwd, mgs_parallel_scan_log_fwd, mgs_set_wait_timeout_ns,
                       mgs_status_string, mgs_version, mgs_workspace_size)

__all__ = [
    "MGSError", "lib", "mgs_check", "mgs_debug_wait_flag", "mgs_linear_scan_bwd", "mgs_linear_scan_fwd", "mgs_matrix_affine_scan_bwd",
    "mgs_matrix_affine_scan_fwd", "mgs_matrix_scan_bwd", "mgs_matrix_scan_fwd", "mgs_matrix_scan_fwd_noalloc",
    "mgs_parallel_scan_log_bwd", "mgs_parallel_scan_log_fwd", "mgs_set_wait_timeout_ns",
    "mgs_status_string", "mgs_version", "mgs_workspace_size",
]
