"""C-ABI checks that need no GPU: the library loads, exports every function
include/mgscan.h declares, and rejects bad arguments with the documented status
before touching the device (fake, never-dereferenced addresses)."""
import os
import re

import pytest

from scan_linear_recurrences_gb300 import _binding as b
from scan_linear_recurrences_gb300.build import LIB, build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "mgscan.h")


@pytest.fixture(scope="module")
def L():
    build()
    return b.lib()


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mgs_[a-z0-9_]+)\s*\(", text)))


def test_library_exports_every_declared_symbol(L):
    names = _declared()
    assert len(names) >= 12
    for n in names:
        assert hasattr(L, n), f"{n} declared in mgscan.h but not exported by {LIB}"
    assert set(names) == set(b.exported_symbols())


def test_version_and_status_strings(L):
    assert b.mgs_version() == 100
    for code, name in b.STATUS_NAMES.items():
        assert b.mgs_status_string(code) == name


FAKE = 1 << 40  # aligned, never dereferenced: every case below fails validation first


def _st(fn, *args):
    try:
        fn(*args, stream=0)
        return b.MGS_OK
    except b.MGSError as e:
        return e.status


def test_mas_validation(L):
    A, bb, h = FAKE, FAKE + (1 << 30), FAKE + (2 << 30)
    assert _st(b.mgs_matrix_affine_scan_fwd, None, bb, None, h, 2, 8, 4, 8) == b.MGS_ERR_INVALID_ARG
    assert _st(b.mgs_matrix_affine_scan_fwd, A, bb, None, h, -1, 8, 4, 8) == b.MGS_ERR_INVALID_ARG
    assert _st(b.mgs_matrix_affine_scan_fwd, A, bb, None, h, 2, 8, 4, 3) == b.MGS_ERR_UNSUPPORTED
    assert _st(b.mgs_matrix_affine_scan_fwd, A, bb, None, h, 2, 8, 3, 1) == b.MGS_ERR_UNSUPPORTED  # H*k % 4
    assert _st(b.mgs_matrix_affine_scan_fwd, A + 4, bb, None, h, 2, 8, 4, 8) == b.MGS_ERR_UNSUPPORTED
    # output overlapping an input
    assert _st(b.mgs_matrix_affine_scan_fwd, A, bb, None, bb + 64, 2, 8, 4, 8) == b.MGS_ERR_INVALID_ARG
    # empty problems are successful no-ops, even with null pointers
    assert _st(b.mgs_matrix_affine_scan_fwd, None, None, None, None, 0, 8, 4, 8) == b.MGS_OK
    assert _st(b.mgs_matrix_affine_scan_fwd, None, None, None, None, 2, 8, 0, 8) == b.MGS_OK
    # overflow of B*T*H*k*k
    assert _st(b.mgs_matrix_affine_scan_fwd, A, bb, None, h, 1 << 40, 1 << 20, 4, 8) == b.MGS_ERR_INVALID_ARG
    # backward: dA overlapping h
    assert _st(b.mgs_matrix_affine_scan_bwd, A, None, h, FAKE + (3 << 30), h, FAKE + (4 << 30), None,
               2, 8, 4, 8) == b.MGS_ERR_INVALID_ARG
    assert _st(b.mgs_matrix_affine_scan_bwd, A, None, None, FAKE + (3 << 30), FAKE + (5 << 30),
               FAKE + (4 << 30), None, 2, 8, 4, 8) == b.MGS_ERR_INVALID_ARG


def test_ms_and_psl_validation(L):
    A, P = FAKE, FAKE + (1 << 30)
    assert _st(b.mgs_matrix_scan_fwd, A, A, 2, 8, 4, 8) == b.MGS_ERR_INVALID_ARG
    assert _st(b.mgs_matrix_scan_fwd, A, P, 2, 8, 4, 5) == b.MGS_ERR_UNSUPPORTED
    assert _st(b.mgs_matrix_scan_bwd, A, P, None, FAKE + (2 << 30), 2, 8, 4, 8) == b.MGS_ERR_INVALID_ARG
    lc, lv, h = FAKE, FAKE + (1 << 30), FAKE + (2 << 30)
    assert _st(b.mgs_parallel_scan_log_fwd, lc, lv, None, h, None, 2, 8, 6) == b.MGS_ERR_UNSUPPORTED  # D % 4
    assert _st(b.mgs_parallel_scan_log_fwd, lc, lv, None, lv, None, 2, 8, 8) == b.MGS_ERR_INVALID_ARG
    assert _st(b.mgs_parallel_scan_log_fwd, lc, lv, None, h, h, 2, 8, 8) == b.MGS_ERR_INVALID_ARG
    # d_log_h0 without log_h0 has no meaning
    assert _st(b.mgs_parallel_scan_log_bwd, lc, lv, None, h, FAKE + (3 << 30), FAKE + (4 << 30),
               FAKE + (5 << 30), FAKE + (6 << 30), 2, 8, 8) == b.MGS_ERR_INVALID_ARG
    # h == NULL: the recompute mode, which needs its checkpoint workspace
    assert _st(b.mgs_parallel_scan_log_bwd, lc, lv, None, None, FAKE + (3 << 30), FAKE + (4 << 30),
               FAKE + (5 << 30), None, 2, 8, 8) == b.MGS_ERR_WORKSPACE
    assert _st(b.mgs_parallel_scan_log_bwd, lc, lv, None, None, FAKE + (3 << 30), FAKE + (4 << 30),
               FAKE + (5 << 30), None, 2, 8, 8, FAKE + (6 << 30), 63) == b.MGS_ERR_WORKSPACE
    # still validated: outputs overlapping inputs
    assert _st(b.mgs_parallel_scan_log_bwd, lc, lv, None, None, FAKE + (3 << 30), lv,
               FAKE + (5 << 30), None, 2, 8, 8, FAKE + (6 << 30), 64) == b.MGS_ERR_INVALID_ARG


def test_psl_recompute_workspace_size(L):
    op = b.MGS_OP_PARALLEL_SCAN_LOG_BWD
    # 4 bytes per channel per 16-step segment: log2 h at each segment start
    assert b.mgs_workspace_size(op, 2, 8, 8, 0) == 4 * 2 * 1 * 8
    assert b.mgs_workspace_size(op, 2, 16, 8, 0) == 4 * 2 * 1 * 8
    assert b.mgs_workspace_size(op, 2, 17, 8, 0) == 4 * 2 * 2 * 8
    assert b.mgs_workspace_size(op, 64, 4096, 1024, 0) == 4 * 64 * 256 * 1024
    assert b.mgs_workspace_size(op, 2, 0, 8, 0) == 0
    assert b.mgs_workspace_size(op, 2, 16, 6, 0) == 0  # D % 4: the call reports it
    assert b.mgs_workspace_size(b.MGS_OP_PARALLEL_SCAN_LOG_FWD, 64, 4096, 1024, 0) == 0


def test_linear_scan_validation(L):
    a, bb, h = FAKE, FAKE + (1 << 30), FAKE + (2 << 30)
    assert _st(b.mgs_linear_scan_fwd, a, bb, None, h, 2, 8, 6) == b.MGS_ERR_UNSUPPORTED  # D % 4
    assert _st(b.mgs_linear_scan_fwd, a, bb, None, bb, 2, 8, 8) == b.MGS_ERR_INVALID_ARG
    assert _st(b.mgs_linear_scan_fwd, None, None, None, None, 0, 8, 8) == b.MGS_OK
    assert b.mgs_workspace_size(b.MGS_OP_LINEAR_SCAN_FWD, 1, 4096, 64, 1) > 0  # few lanes: chunked
    assert b.mgs_workspace_size(b.MGS_OP_LINEAR_SCAN_FWD, 64, 4096, 1024, 1) == 0


def test_workspace_size_queries(L):
    for op in range(1, 9):
        assert b.mgs_workspace_size(op, 2, 16, 8, 8) >= 0
    assert b.mgs_workspace_size(b.MGS_OP_MATRIX_SCAN_FWD, -1, 16, 8, 8) == 0
    # many lanes or short sequences: single pass, no workspace
    assert b.mgs_workspace_size(b.MGS_OP_MATRIX_SCAN_FWD, 128, 64, 8, 8) == 0
    # few lanes, long sequence: time chunks exchange carries through the workspace
    nf = b.mgs_workspace_size(b.MGS_OP_MATRIX_SCAN_FWD, 16, 1024, 8, 8)
    nb = b.mgs_workspace_size(b.MGS_OP_MATRIX_SCAN_BWD, 16, 1024, 8, 8)
    assert 0 < nf < nb


def test_workspace_errors(L):
    A, P = FAKE, FAKE + (1 << 30)
    n = b.mgs_workspace_size(b.MGS_OP_MATRIX_SCAN_FWD, 16, 1024, 8, 8)
    assert _st(b.mgs_matrix_scan_fwd, A, P, 16, 1024, 8, 8, None, 0) == b.MGS_ERR_WORKSPACE
    assert _st(b.mgs_matrix_scan_fwd, A, P, 16, 1024, 8, 8, FAKE + (3 << 30), n - 1) == b.MGS_ERR_WORKSPACE
    assert _st(b.mgs_matrix_scan_fwd, A, P, 16, 1024, 8, 8, FAKE + (3 << 30) + 16, n) == b.MGS_ERR_WORKSPACE


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(b, "LIB_PATH", str(tmp_path / "nope.so"))
    monkeypatch.setattr(b, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        b.lib()


def test_givens_workspace_only_for_few_lanes_and_long_T(L):
    for op in (b.MGS_OP_GIVENS_AFFINE_SCAN_FWD, b.MGS_OP_GIVENS_AFFINE_SCAN_BWD,
               b.MGS_OP_GIVENS_MATRIX_SCAN_FWD, b.MGS_OP_GIVENS_MATRIX_SCAN_BWD):
        assert b.mgs_workspace_size(op, 128, 64, 8, 8) == 0      # lab shape: angle-fused kernels
        assert b.mgs_workspace_size(op, 64, 1024, 64, 8) == 0    # many lanes
        assert b.mgs_workspace_size(op, 16, 128, 8, 8) == 0      # T < 256
        assert b.mgs_workspace_size(op, 16, 1024, 8, 4) == 0     # k != 8: the call reports it
    # long-T shape: time-chunked, still from the angles; the workspace holds only
    # the chunk aggregates and carries (those of the matrix scans' chunked
    # paths), never A_t or dA_t (256 bytes per step, 33.5 MB here)
    steps = 16 * 1024 * 8
    for op, same in ((b.MGS_OP_GIVENS_AFFINE_SCAN_FWD, b.MGS_OP_MATRIX_AFFINE_SCAN_FWD),
                     (b.MGS_OP_GIVENS_AFFINE_SCAN_BWD, b.MGS_OP_MATRIX_AFFINE_SCAN_BWD),
                     (b.MGS_OP_GIVENS_MATRIX_SCAN_FWD, b.MGS_OP_MATRIX_SCAN_FWD),
                     (b.MGS_OP_GIVENS_MATRIX_SCAN_BWD, b.MGS_OP_MATRIX_SCAN_BWD)):
        n = b.mgs_workspace_size(op, 16, 1024, 8, 8)
        assert 0 < n == b.mgs_workspace_size(same, 16, 1024, 8, 8)
        assert n < steps * 256 // 8
    th, bb, h = FAKE, FAKE + (1 << 30), FAKE + (2 << 30)
    assert _st(b.mgs_givens_affine_scan_fwd, th, None, bb, None, h, 16, 1024, 8, 8) == b.MGS_ERR_WORKSPACE


def test_delta_workspace_size(L):
    # R, M, (P U)^T and N^T of every lane's 64-step chunks, 64 x 64 floats each
    op = b.MGS_OP_DELTA_SCAN_FWD
    per_chunk = 4 * 64 * 64 * 4
    assert b.mgs_workspace_size(op, 128, 64, 1, 64) == 128 * per_chunk
    assert b.mgs_workspace_size(op, 16, 1024, 1, 64) == 16 * 16 * per_chunk
    assert b.mgs_workspace_size(op, 2, 70, 3, 64) == 2 * 3 * 2 * per_chunk   # ragged tail: a whole chunk
    assert b.mgs_workspace_size(op, 2, 0, 3, 64) == 0
    assert b.mgs_workspace_size(op, 2, 64, 3, 32) == 0                       # D != 64: the call reports it
    assert b.mgs_workspace_size(op, -1, 64, 3, 64) == 0


def test_mas_recompute_workspace_and_validation(L):
    # checkpoints: 32 floats per (lane group of 32/k heads, chunk of TS steps)
    op = b.MGS_OP_MATRIX_AFFINE_SCAN_BWD_RECOMPUTE
    assert b.mgs_workspace_size(op, 2, 40, 4, 8) == 2 * 1 * 5 * 32 * 4     # TS 8
    assert b.mgs_workspace_size(op, 2, 40, 4, 16) == 2 * 2 * 10 * 32 * 4   # TS 4
    assert b.mgs_workspace_size(op, 2, 40, 64, 1) == 2 * 2 * 3 * 32 * 4    # TS 16
    assert b.mgs_workspace_size(op, 32, 8192, 64, 8) == 32 * 16 * 1024 * 32 * 4
    # few lanes, long sequence: h plus the time-chunked kernels' workspace
    chunked = b.mgs_workspace_size(b.MGS_OP_MATRIX_AFFINE_SCAN_BWD, 16, 1024, 8, 8)
    assert chunked > 0
    assert b.mgs_workspace_size(op, 16, 1024, 8, 8) == 16 * 1024 * 8 * 8 * 4 + chunked
    assert b.mgs_workspace_size(op, 2, 0, 4, 8) == 0
    assert b.mgs_workspace_size(op, 2, 40, 4, 3) == 0                      # unsupported k: the call reports it
    A, bb, g = FAKE, FAKE + (1 << 30), FAKE + (2 << 30)
    dA, db = FAKE + (3 << 30), FAKE + (4 << 30)
    f = b.mgs_matrix_affine_scan_bwd_recompute
    assert _st(f, A, None, None, g, dA, db, None, 2, 40, 4, 8) == b.MGS_ERR_INVALID_ARG     # b required
    assert _st(f, A, bb, None, g, dA, bb, None, 2, 40, 4, 8) == b.MGS_ERR_INVALID_ARG       # db over b
    assert _st(f, A, bb, None, g, dA, db, None, 2, 40, 4, 8) == b.MGS_ERR_WORKSPACE         # none given
    assert _st(f, A, bb, None, g, dA, db, None, 2, 40, 4, 3) == b.MGS_ERR_UNSUPPORTED
    assert _st(f, None, None, None, None, None, None, None, 2, 40, 0, 8) == b.MGS_OK         # no lanes


def test_binding_op_ids_match_the_header():
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    ids = dict(re.findall(r"\b(MGS_OP_[A-Z_]+)\s*=\s*(\d+)", text))
    assert len(ids) >= 14
    for name, value in ids.items():
        assert getattr(b, name) == int(value), name
    statuses = dict(re.findall(r"\b(MGS_(?:OK|ERR_[A-Z_]+))\s*=\s*(\d+)", text))
    for name, value in statuses.items():
        assert getattr(b, name) == int(value), name
