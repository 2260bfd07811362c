"""GPU parity: the CUDA library (called through its C ABI) against the float64
oracle on the same seeded float32 inputs, at small sizes that span several
ring stages and ragged tails, at the benchmark's full sizes (every element,
compared in groups of batch rows), and on the degenerate cases."""
import numpy as np
import pytest
import torch

import oracle
from scan_linear_recurrences_gb300 import _binding as b
from scan_linear_recurrences_gb300 import api, inputs
from scan_linear_recurrences_gb300.build import build

from ._parity import Streamed, assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    build()
    b.lib()
    yield
    b.mgs_check()


def _cuda(d):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}


# ---------------------------------------------------------------- matrix_affine_scan
def _run_mas(B, T, H, k, seed, h0_mode, sample=None):
    d = _cuda(inputs.mas_inputs(B, T, H, k, seed, device="cpu", h0=h0_mode))
    h = api.matrix_affine_scan_fwd(d["A"], d["b"], d["h0"])
    dA, db, dh0 = api.matrix_affine_scan_bwd(d["A"], d["h0"], h, d["grad_h"], need_dh0=True)
    b.mgs_check()
    sel = slice(None) if sample is None else sample
    A, bb, g = d["A"][sel].cpu(), d["b"][sel].cpu(), d["grad_h"][sel].cpu()
    h0 = d["h0"][sel].cpu() if d["h0"] is not None else torch.zeros((A.shape[0], H, k))
    href = oracle.mas_fwd(A, bb, h0)
    dAr, dbr, dh0r = oracle.mas_bwd(A, bb, h0, g)
    assert_close("h", h[sel], href, T)
    assert_close("dA", dA[sel], dAr, T)
    assert_close("db", db[sel], dbr, T)
    assert_close("dh0", dh0[sel], dh0r, T)


@pytest.mark.parametrize("cid", [0, 1])
def test_mas_configs_full(cid):
    w = inputs.WORKLOADS[cid]
    _run_mas(w.B, w.T, w.H, w.k, w.seed, w.h0)


@pytest.mark.parametrize("B,T,H,k,h0", [
    (1, 1, 1, 8, "normal"),     # single step
    (3, 37, 5, 8, "normal"),    # ragged T (not a multiple of the stage), partial head group
    (2, 70, 9, 8, "zeros"),     # explicit zero initial state
    (2, 45, 3, 4, "normal"),
    (2, 33, 3, 16, "normal"),
    (2, 50, 6, 2, "normal"),
    (2, 81, 12, 1, "normal"),   # k = 1: the diagonal (linear_scan) case
    (1, 300, 4, 8, "none"),
    # 256 or more lane groups (one pass per lane group), ragged head groups
    (96, 200, 11, 8, "none"), (300, 90, 7, 4, "normal"), (64, 1100, 16, 8, "normal"),
    # few lanes, long sequences: the time-chunked path
    (1, 1000, 3, 16, "normal"), (2, 515, 5, 4, "normal"), (1, 2048, 8, 8, "none"), (3, 4099, 2, 2, "normal"),
    # k = 1, few lanes, past the one-launch path's T = 1024: time chunks
    (2, 5000, 40, 1, "normal"), (1, 40000, 8, 1, "none"),
])
def test_mas_shapes(B, T, H, k, h0):
    _run_mas(B, T, H, k, seed=100 + B * T + H + k, h0_mode=h0)


def test_mas_long_T_shape_of_the_pages():
    """The pages' long-T benchmark shape (B=16, T=1024) with d=64 as H=8 blocks
    of k=8: 32 lane groups, so the sequence is split into time chunks."""
    assert b.mgs_workspace_size(b.MGS_OP_MATRIX_AFFINE_SCAN_FWD, 16, 1024, 8, 8) > 0
    _run_mas(16, 1024, 8, 8, seed=4242, h0_mode="normal")


def test_mas_config4_full():
    """Full benchmark size (B=32, T=8192, H=64, k=8) in the launch
    configuration the benchmark times, every output element compared with the
    oracle (streamed over groups of 4 batch rows)."""
    w = inputs.WORKLOADS[4]
    d = w.make(device="cuda")
    h = api.matrix_affine_scan_fwd(d["A"], d["b"], d["h0"])
    dA, db, dh0 = api.matrix_affine_scan_bwd(d["A"], d["h0"], h, d["grad_h"])
    b.mgs_check()
    acc = {n: Streamed(n) for n in ("h", "dA", "db", "dh0")}
    for r0 in range(0, w.B, 4):
        rows = slice(r0, min(w.B, r0 + 4))
        A, bb, h0, g = (d[k][rows].cpu() for k in ("A", "b", "h0", "grad_h"))
        acc["h"].add(h[rows], oracle.mas_fwd(A, bb, h0))
        dAr, dbr, dh0r = oracle.mas_bwd(A, bb, h0, g)
        acc["dA"].add(dA[rows], dAr)
        acc["db"].add(db[rows], dbr)
        acc["dh0"].add(dh0[rows], dh0r)
        del A, bb, h0, g, dAr, dbr, dh0r
    for a in acc.values():
        assert a.n > 0
        a.check(w.T)


def test_mas_empty_and_T0():
    dev = "cuda"
    A = torch.empty((2, 0, 3, 8, 8), device=dev)
    bb = torch.empty((2, 0, 3, 8), device=dev)
    h = api.matrix_affine_scan_fwd(A, bb, None)
    assert h.shape == (2, 0, 3, 8)
    h0 = torch.randn((2, 3, 8), device=dev)
    dh0 = torch.full((2, 3, 8), float("nan"), device=dev)
    b.mgs_matrix_affine_scan_bwd(A, h0, bb, bb, A, bb, dh0, 2, 0, 3, 8)
    b.mgs_check()
    assert torch.equal(dh0, torch.zeros_like(dh0))


# ---------------------------------------------------------------- matrix_affine_scan, recompute-mode backward
@pytest.mark.parametrize("B,T,H,k,h0", [
    (1, 1, 1, 8, "normal"),      # one step
    (3, 37, 5, 8, "normal"),     # ragged last chunk, partial head group
    (2, 8, 4, 8, "none"),        # exactly one chunk
    (2, 32, 4, 8, "normal"),     # exactly the four ring slots
    (2, 40, 4, 8, "normal"),     # the ring refilled
    (2, 70, 9, 8, "zeros"),
    (2, 45, 3, 4, "normal"), (2, 33, 3, 16, "normal"), (2, 50, 6, 2, "normal"), (2, 81, 12, 1, "normal"),
    (1, 300, 4, 8, "normal"),
    # few lanes, long sequences: chunked forward into the workspace, chunked backward
    (1, 1000, 3, 16, "normal"), (16, 1024, 8, 8, "normal"), (3, 4099, 2, 2, "none"),
])
def test_mas_recompute_backward(B, T, H, k, h0):
    """No saved h: checkpoints at every chunk start, chunks rebuilt downwards."""
    d = _cuda(inputs.mas_inputs(B, T, H, k, seed=900 + B * T + H + k, device="cpu", h0=h0))
    rec = api.matrix_affine_scan_bwd_recompute(d["A"], d["b"], d["h0"], d["grad_h"], need_dh0=True)
    b.mgs_check()
    A, bb, g = d["A"].cpu(), d["b"].cpu(), d["grad_h"].cpu()
    h0c = d["h0"].cpu() if d["h0"] is not None else torch.zeros((B, H, k))
    dAr, dbr, dh0r = oracle.mas_bwd(A, bb, h0c, g)
    assert_close("dA", rec[0], dAr, T)
    assert_close("db", rec[1], dbr, T)
    assert_close("dh0", rec[2], dh0r, T)
    if b.mgs_workspace_size(b.MGS_OP_MATRIX_AFFINE_SCAN_FWD, B, T, H, k) == 0:
        # single-pass shapes: the recomputed h follows the forward kernel's
        # arithmetic step for step, so the two backwards agree to rounding
        h = api.matrix_affine_scan_fwd(d["A"], d["b"], d["h0"])
        saved = api.matrix_affine_scan_bwd(d["A"], d["h0"], h, d["grad_h"], need_dh0=True)
        b.mgs_check()
        for name, x, y in zip(("dA", "db", "dh0"), rec, saved):
            assert_close(name + " (vs saved h)", x, y.double().cpu().numpy(), T, rel_tol=1e-6, abs_tol=1e-5)


def test_mas_recompute_config4_full():
    """Full benchmark size (B=32, T=8192, H=64, k=8), recompute mode, every
    element compared (streamed over groups of 4 batch rows)."""
    w = inputs.WORKLOADS[4]
    d = w.make(device="cuda")
    dA, db, dh0 = api.matrix_affine_scan_bwd_recompute(d["A"], d["b"], d["h0"], d["grad_h"])
    b.mgs_check()
    acc = {n: Streamed(n) for n in ("dA", "db", "dh0")}
    for r0 in range(0, w.B, 4):
        rows = slice(r0, min(w.B, r0 + 4))
        A, bb, h0, g = (d[k][rows].cpu() for k in ("A", "b", "h0", "grad_h"))
        dAr, dbr, dh0r = oracle.mas_bwd(A, bb, h0, g)
        acc["dA"].add(dA[rows], dAr)
        acc["db"].add(db[rows], dbr)
        acc["dh0"].add(dh0[rows], dh0r)
        del A, bb, h0, g, dAr, dbr, dh0r
    for a in acc.values():
        a.check(w.T)


def test_mas_recompute_T0_and_errors():
    dev = "cuda"
    A = torch.empty((2, 0, 3, 8, 8), device=dev)
    bb = torch.empty((2, 0, 3, 8), device=dev)
    dh0 = torch.full((2, 3, 8), float("nan"), device=dev)
    b.mgs_matrix_affine_scan_bwd_recompute(A, bb, None, bb, A, bb, dh0, 2, 0, 3, 8)
    b.mgs_check()
    assert torch.equal(dh0, torch.zeros_like(dh0))
    d = _cuda(inputs.mas_inputs(2, 40, 4, 8, seed=5, device="cpu", h0="normal"))
    dA, db = torch.empty_like(d["A"]), torch.empty_like(d["b"])
    with pytest.raises(b.MGSError) as err:  # the checkpoints need a workspace
        b.mgs_matrix_affine_scan_bwd_recompute(d["A"], d["b"], d["h0"], d["grad_h"], dA, db, None, 2, 40, 4, 8)
    assert err.value.status == b.MGS_ERR_WORKSPACE


# ---------------------------------------------------------------- matrix_scan
def _run_ms(B, T, H, k, seed):
    d = _cuda(inputs.ms_inputs(B, T, H, k, seed))
    P = api.matrix_scan_fwd(d["A"])
    dA = api.matrix_scan_bwd(d["A"], P, d["grad_P"])
    b.mgs_check()
    assert_close("P", P, oracle.ms_fwd(d["A"].cpu()), T)
    assert_close("dA", dA, oracle.ms_bwd(d["A"].cpu(), d["grad_P"].cpu()), T)


def test_ms_config2_full():
    w = inputs.WORKLOADS[2]
    _run_ms(w.B, w.T, w.H, w.k, w.seed)


@pytest.mark.parametrize("B,T,H,k", [
    (1, 1, 1, 8), (2, 13, 5, 8), (2, 21, 3, 4), (2, 17, 3, 16), (1, 40, 2, 2), (2, 30, 8, 1),
    # long sequences with few lanes take the time-chunked path
    (1, 333, 2, 8), (2, 1000, 3, 4), (1, 515, 3, 16), (1, 257, 4, 1), (1, 130, 2, 2), (3, 4099, 5, 8),
    # 32 chunks with a ragged last one, and 33 chunks
    (1, 1019, 3, 8), (1, 1056, 4, 8),
])
def test_ms_shapes(B, T, H, k):
    _run_ms(B, T, H, k, seed=200 + B * T + H + k)


def test_ms_chunked_repeat_reuses_workspace():
    """Two calls in a row on one workspace: nothing in it has to start at
    zero, and the chunked path adds in a fixed order, so the two results are
    equal bit for bit."""
    d = _cuda(inputs.ms_inputs(2, 700, 4, 8, seed=17))
    n = b.mgs_workspace_size(b.MGS_OP_MATRIX_SCAN_FWD, 2, 700, 4, 8)
    assert n > 0
    ws = torch.full((n,), 0xA5, dtype=torch.uint8, device="cuda")  # garbage, not zeros
    P1 = torch.empty_like(d["A"]); P2 = torch.empty_like(d["A"])
    b.mgs_matrix_scan_fwd(d["A"], P1, 2, 700, 4, 8, ws, n)
    b.mgs_matrix_scan_fwd(d["A"], P2, 2, 700, 4, 8, ws, n)
    b.mgs_check()
    ref = oracle.ms_fwd(d["A"].cpu())
    assert_close("P first call", P1, ref, 700)
    assert torch.equal(P1, P2)


@pytest.mark.timeout(300)
def test_chunked_repeated_calls_stay_correct():
    """Many back-to-back chunked calls sharing their workspaces: every call
    finishes and matches the oracle."""
    B, T, H, k = 2, 2050, 3, 8
    dm = _cuda(inputs.mas_inputs(B, T, H, k, seed=77, h0="normal"))
    ds = _cuda(inputs.ms_inputs(B, T, H, k, seed=78))
    href = oracle.mas_fwd(dm["A"].cpu(), dm["b"].cpu(), dm["h0"].cpu())
    dAr, _, _ = oracle.mas_bwd(dm["A"].cpu(), dm["b"].cpu(), dm["h0"].cpu(), dm["grad_h"].cpu())
    Pref = oracle.ms_fwd(ds["A"].cpu())
    for _ in range(25):
        h = api.matrix_affine_scan_fwd(dm["A"], dm["b"], dm["h0"])
        dA, _, _ = api.matrix_affine_scan_bwd(dm["A"], dm["h0"], h, dm["grad_h"])
        P = api.matrix_scan_fwd(ds["A"])
        dAs = api.matrix_scan_bwd(ds["A"], P, ds["grad_P"])
    b.mgs_check()
    assert_close("h", h, href, T)
    assert_close("dA", dA, dAr, T)
    assert_close("P", P, Pref, T)


# ---------------------------------------------------------------- parallel_scan_log
def _run_psl(B, T, D, seed, with_h0=True, rows=None):
    d = _cuda(inputs.psl_inputs(B, T, D, seed, device="cpu", with_h0=with_h0))
    return _check_psl(d, T, rows)


def _check_psl(d, T, rows=None):
    h, lh = api.parallel_scan_log_fwd(d["log_coeffs"], d["log_values"], d["log_h0"], want_log=True)
    dlc, dlv, dl0 = api.parallel_scan_log_bwd(d["log_coeffs"], d["log_values"], d["log_h0"], h, d["grad_h"])
    b.mgs_check()
    sel = slice(None) if rows is None else rows
    lc, lv, g = (d[k][sel].cpu() for k in ("log_coeffs", "log_values", "grad_h"))
    l0 = d["log_h0"][sel].cpu() if d["log_h0"] is not None else None
    href, lhref = oracle.psl_fwd(lc, lv, l0, want_log=True)
    assert_close("h", h[sel], href, T)
    assert_close("log_h", lh[sel], lhref, T)
    dlcr, dlvr, dl0r = oracle.psl_bwd(lc, lv, l0, g)
    assert_close("d_log_coeffs", dlc[sel], dlcr, T)
    assert_close("d_log_values", dlv[sel], dlvr, T)
    if l0 is not None:
        assert_close("d_log_h0", dl0[sel], dl0r, T)


@pytest.mark.parametrize("B,T,D,h0", [
    (2, 1, 4, True), (3, 50, 132, True), (2, 257, 1024, True), (2, 100, 260, False), (1, 2000, 128, True),
    # the pages' lab and long-T shapes (one-launch time-parallel path), and
    # the edges of that path: 8 -> 16 steps a block past T = 512, one ->
    # several blocks a warp past T = 1024 (odd block counts, ragged last
    # blocks), its end at T = 32768, 2048 channel groups
    (128, 64, 64, True), (16, 1024, 64, True), (3, 512, 20, True), (2, 513, 20, False),
    (1, 1024, 8, False), (1, 1025, 8, True), (2, 3000, 20, True), (1, 8192, 64, False), (1, 8193, 8, True),
    (1, 32768, 8, True), (1, 32769, 4, False),
    (63, 40, 1024, True), (64, 40, 1024, True),
])
def test_psl_shapes(B, T, D, h0):
    _run_psl(B, T, D, seed=300 + B * T + D, with_h0=h0)


def test_psl_config3_full():
    """Full benchmark size (B=64, T=4096, D=1024), every element of h, log h
    and the three gradients compared (streamed over groups of 8 batch rows)."""
    w = inputs.WORKLOADS[3]
    d = w.make(device="cuda")
    h, lh = api.parallel_scan_log_fwd(d["log_coeffs"], d["log_values"], d["log_h0"], want_log=True)
    dlc, dlv, dl0 = api.parallel_scan_log_bwd(d["log_coeffs"], d["log_values"], d["log_h0"], h, d["grad_h"])
    b.mgs_check()
    acc = {n: Streamed(n) for n in ("h", "log_h", "d_log_coeffs", "d_log_values", "d_log_h0")}
    for r0 in range(0, w.B, 8):
        rows = slice(r0, min(w.B, r0 + 8))
        lc, lv, l0, g = (d[k][rows].cpu() for k in ("log_coeffs", "log_values", "log_h0", "grad_h"))
        href, lhref = oracle.psl_fwd(lc, lv, l0, want_log=True)
        acc["h"].add(h[rows], href)
        acc["log_h"].add(lh[rows], lhref)
        dlcr, dlvr, dl0r = oracle.psl_bwd(lc, lv, l0, g)
        acc["d_log_coeffs"].add(dlc[rows], dlcr)
        acc["d_log_values"].add(dlv[rows], dlvr)
        acc["d_log_h0"].add(dl0[rows], dl0r)
        del lc, lv, l0, g, href, lhref, dlcr, dlvr, dl0r
    for a in acc.values():
        a.check(w.T)


def test_psl_zero_coefficients_and_empty():
    # log_coeffs = -inf: h_t = exp(log_values_t); gradients through the coefficient vanish
    B, T, D = 2, 20, 8
    lc = torch.full((B, T, D), float("-inf"), device="cuda")
    lv = torch.randn((B, T, D), device="cuda")
    l0 = torch.randn((B, D), device="cuda")
    h = api.parallel_scan_log_fwd(lc, lv, l0)
    b.mgs_check()
    assert_close("h", h, oracle.psl_fwd(lc.cpu(), lv.cpu(), l0.cpu()), T)
    empty = torch.empty((0, 5, 8), device="cuda")
    assert api.parallel_scan_log_fwd(empty, empty).shape == (0, 5, 8)


@pytest.mark.parametrize("B,T,D,h0", [
    (2, 1, 4, True), (3, 15, 132, True), (2, 16, 8, False), (2, 17, 1024, True), (3, 50, 260, False),
    (2, 257, 1024, True), (1, 2000, 128, True), (5, 33, 36, True),
    # the pages' long-T and lab shapes, on the one-launch cluster path (one
    # and several blocks a warp)
    (16, 1024, 64, True), (128, 64, 64, False), (2, 600, 12, True), (2, 2500, 36, True), (1, 8192, 8, False),
    (1, 30000, 4, True), (2, 1025, 40, True), (1, 32768, 8, True),
    # 2048 channel groups, ragged last segment: the checkpointing kernel
    (64, 33, 1024, True),
])
def test_psl_recompute_backward(B, T, D, h0):
    """h == NULL.  With many lanes: checkpoints every 16 steps, segments rebuilt
    in reverse (ragged last segments, T below one segment, partial 128-channel
    groups); with few lanes and T <= 1024: h recomputed in registers by the
    one-launch cluster kernel."""
    d = _cuda(inputs.psl_inputs(B, T, D, seed=700 + B * T + D, with_h0=h0))
    lc, lv, l0, g = d["log_coeffs"], d["log_values"], d["log_h0"], d["grad_h"]
    h = api.parallel_scan_log_fwd(lc, lv, l0)
    saved = api.parallel_scan_log_bwd(lc, lv, l0, h, g)
    rec = api.parallel_scan_log_bwd(lc, lv, l0, None, g)
    b.mgs_check()
    dlcr, dlvr, dl0r = oracle.psl_bwd(lc.cpu(), lv.cpu(), l0.cpu() if h0 else None, g.cpu())
    assert_close("d_log_coeffs", rec[0], dlcr, T)
    assert_close("d_log_values", rec[1], dlvr, T)
    if h0:
        assert_close("d_log_h0", rec[2], dl0r, T)
    else:
        assert rec[2] is None
    # the recomputed h follows the forward kernel's arithmetic step for step
    for name, x, y in zip(("d_log_coeffs", "d_log_values", "d_log_h0"), rec, saved):
        if y is not None:
            assert_close(name + " (vs saved h)", x, y.double().cpu().numpy(), T, rel_tol=1e-6, abs_tol=1e-5)


def test_psl_recompute_config3_full():
    """Full benchmark size, recompute mode (h not saved), every element of the
    three gradients compared (streamed over groups of 8 batch rows)."""
    w = inputs.WORKLOADS[3]
    d = w.make(device="cuda")
    dlc, dlv, dl0 = api.parallel_scan_log_bwd(d["log_coeffs"], d["log_values"], d["log_h0"], None, d["grad_h"])
    b.mgs_check()
    acc = {n: Streamed(n) for n in ("d_log_coeffs", "d_log_values", "d_log_h0")}
    for r0 in range(0, w.B, 8):
        rows = slice(r0, min(w.B, r0 + 8))
        dlcr, dlvr, dl0r = oracle.psl_bwd(*(d[k][rows].cpu() for k in ("log_coeffs", "log_values", "log_h0",
                                                                       "grad_h")))
        acc["d_log_coeffs"].add(dlc[rows], dlcr)
        acc["d_log_values"].add(dlv[rows], dlvr)
        acc["d_log_h0"].add(dl0[rows], dl0r)
        del dlcr, dlvr, dl0r
    for a in acc.values():
        a.check(w.T)


def test_psl_recompute_autograd_and_T0():
    d = _cuda(inputs.psl_inputs(2, 70, 12, seed=9))
    lc = d["log_coeffs"].clone().requires_grad_(True)
    lv = d["log_values"].clone().requires_grad_(True)
    l0 = d["log_h0"].clone().requires_grad_(True)
    (api.parallel_scan_log(lc, lv, l0, recompute=True) * d["grad_h"]).sum().backward()
    dlcr, dlvr, dl0r = oracle.psl_bwd(*(d[k].cpu() for k in ("log_coeffs", "log_values", "log_h0", "grad_h")))
    assert_close("d_log_coeffs", lc.grad, dlcr, 70)
    assert_close("d_log_values", lv.grad, dlvr, 70)
    assert_close("d_log_h0", l0.grad, dl0r, 70)
    # T = 0: d_log_h0 = 0, nothing else written
    e = torch.empty((2, 0, 12), device="cuda")
    z = torch.randn((2, 12), device="cuda")
    _, _, dz = api.parallel_scan_log_bwd(e, e, z, None, e)
    b.mgs_check()
    assert torch.equal(dz, torch.zeros_like(z))


# ---------------------------------------------------------------- linear_scan
@pytest.mark.parametrize("B,T,D,h0", [
    (2, 1, 4, True), (3, 77, 132, True), (2, 300, 64, True), (1, 2000, 32, False), (4, 500, 1024, True),
    (16, 1024, 64, True), (128, 64, 64, True),
    # edges of the one-launch time-parallel path: 8 -> 16 steps a warp past
    # T = 512, the three-launch chunked path past T = 1024, and 2048 channel
    # groups
    (3, 512, 36, True), (2, 513, 20, False), (1, 1024, 8, False), (1, 1025, 8, True),
    (2, 3000, 20, True), (1, 8192, 64, False), (1, 8193, 8, True), (1, 32768, 8, True), (1, 32769, 4, False),
    (63, 40, 1024, True), (64, 40, 1024, True),
])
def test_linear_scan(B, T, D, h0):
    d = _cuda(inputs.linear_inputs(B, T, D, seed=500 + B * T + D, with_h0=h0))
    h = api.linear_scan_fwd(d["a"], d["b"], d["h0"])
    da, db, dh0 = api.linear_scan_bwd(d["a"], d["h0"], h, d["grad_h"], need_dh0=True)
    b.mgs_check()
    a, bb, g = d["a"].cpu(), d["b"].cpu(), d["grad_h"].cpu()
    hz = d["h0"].cpu() if d["h0"] is not None else torch.zeros((B, D))
    assert_close("h", h, oracle.linear_fwd(a, bb, hz), T)
    dar, dbr, dh0r = oracle.linear_bwd(a, bb, hz, g)
    assert_close("da", da, dar, T)
    assert_close("db", db, dbr, T)
    assert_close("dh0", dh0, dh0r, T)


# ---------------------------------------------------------------- autograd wrappers
def test_linear_scan_autograd():
    d = _cuda(inputs.linear_inputs(2, 90, 8, seed=8))
    a = d["a"].clone().requires_grad_(True)
    bb = d["b"].clone().requires_grad_(True)
    h0 = d["h0"].clone().requires_grad_(True)
    (api.linear_scan(a, bb, h0) * d["grad_h"]).sum().backward()
    dar, dbr, dh0r = oracle.linear_bwd(d["a"].cpu(), d["b"].cpu(), d["h0"].cpu(), d["grad_h"].cpu())
    assert_close("da", a.grad, dar, 90)
    assert_close("db", bb.grad, dbr, 90)
    assert_close("dh0", h0.grad, dh0r, 90)


@pytest.mark.parametrize("recompute", [False, True])
def test_autograd_wrappers_match_oracle(recompute):
    d = _cuda(inputs.mas_inputs(2, 30, 3, 8, seed=7, h0="normal"))
    A = d["A"].clone().requires_grad_(True)
    bb = d["b"].clone().requires_grad_(True)
    h0 = d["h0"].clone().requires_grad_(True)
    h = api.matrix_affine_scan(A, bb, h0, recompute=recompute)
    (h * d["grad_h"]).sum().backward()
    dAr, dbr, dh0r = oracle.mas_bwd(d["A"].cpu(), d["b"].cpu(), d["h0"].cpu(), d["grad_h"].cpu())
    assert_close("dA", A.grad, dAr, 30)
    assert_close("db", bb.grad, dbr, 30)
    assert_close("dh0", h0.grad, dh0r, 30)


# ---------------------------------------------------------------- failure detection
def test_bounded_wait_reports_timeout_and_context_survives():
    """A wait on a flag that nothing sets gives up after the timeout, the error
    word reports it, and the device keeps working afterwards."""
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    b.mgs_set_wait_timeout_ns(20_000_000)  # 20 ms
    try:
        b.mgs_debug_wait_flag(flag)
        with pytest.raises(b.MGSError) as ei:
            b.mgs_check()
        assert ei.value.status == b.MGS_ERR_TIMEOUT
        b.mgs_check()  # cleared
        flag.fill_(1)
        b.mgs_debug_wait_flag(flag)
        b.mgs_check()
    finally:
        b.mgs_set_wait_timeout_ns(1_000_000_000)
    _run_mas(1, 16, 4, 8, seed=1, h0_mode="normal")
