"""Randomised parity sweep: every entry point on a few dozen small shapes drawn
with a fixed seed (sizes that cross stage, chunk and lane-group boundaries,
optional initial states and gates), each checked against the float64 oracle.
Complements the hand-picked shapes of the other GPU tests."""
import numpy as np
import pytest
import torch

import oracle
from scan_linear_recurrences_gb300 import _binding as b
from scan_linear_recurrences_gb300 import api, inputs
from scan_linear_recurrences_gb300.build import build

from ._parity import assert_close

pytestmark = pytest.mark.gpu
R = np.random.default_rng(20261202)


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


def _cpu(x):
    return x.cpu() if x is not None else None


MAS = [(int(R.integers(1, 6)), int(R.integers(1, 400)), int(R.integers(1, 9)), int(R.choice([1, 2, 4, 8, 16])),
        str(R.choice(["none", "normal"]))) for _ in range(12)]


@pytest.mark.parametrize("B,T,H,k,h0", MAS)
def test_random_matrix_affine_scan(B, T, H, k, h0):
    if k < 4:  # the library needs H*k to be a multiple of 4 for k = 1, 2
        m = 4 // k
        H = (H + m - 1) // m * m
    d = _cuda(inputs.mas_inputs(B, T, H, k, seed=B * 7919 + T * 31 + H * k, h0=h0))
    h = api.matrix_affine_scan_fwd(d["A"], d["b"], d["h0"])
    dA, db, dh0 = api.matrix_affine_scan_bwd(d["A"], d["h0"], h, d["grad_h"])
    b.mgs_check()
    A, bb, g = _cpu(d["A"]), _cpu(d["b"]), _cpu(d["grad_h"])
    z0 = _cpu(d["h0"]) if d["h0"] is not None else torch.zeros((B, H, k))
    assert_close("h", h, oracle.mas_fwd(A, bb, z0), T)
    rA, rb, r0 = oracle.mas_bwd(A, bb, z0, g)
    assert_close("dA", dA, rA, T)
    assert_close("db", db, rb, T)
    assert_close("dh0", dh0, r0, T)
    # the recompute-mode backward (no saved h) on the same draw
    qA, qb, q0 = api.matrix_affine_scan_bwd_recompute(d["A"], d["b"], d["h0"], d["grad_h"])
    b.mgs_check()
    assert_close("dA (recompute)", qA, rA, T)
    assert_close("db (recompute)", qb, rb, T)
    assert_close("dh0 (recompute)", q0, r0, T)


MS = [(int(R.integers(1, 5)), int(R.integers(1, 300)), int(R.integers(1, 6)), int(R.choice([4, 8, 16])))
      for _ in range(8)]


@pytest.mark.parametrize("B,T,H,k", MS)
def test_random_matrix_scan(B, T, H, k):
    d = _cuda(inputs.ms_inputs(B, T, H, k, seed=B * 101 + T * 7 + H))
    P = api.matrix_scan_fwd(d["A"])
    dA = api.matrix_scan_bwd(d["A"], P, d["grad_P"])
    b.mgs_check()
    assert_close("P", P, oracle.ms_fwd(_cpu(d["A"])), T)
    assert_close("dA", dA, oracle.ms_bwd(_cpu(d["A"]), _cpu(d["grad_P"])), T)


PSL = [(int(R.integers(1, 5)), int(R.integers(1, 700)), 4 * int(R.integers(1, 80)), bool(R.integers(0, 2)))
       for _ in range(8)]


@pytest.mark.parametrize("B,T,D,h0", PSL)
def test_random_parallel_scan_log(B, T, D, h0):
    d = _cuda(inputs.psl_inputs(B, T, D, seed=B * 13 + T + D, with_h0=h0))
    h = api.parallel_scan_log_fwd(d["log_coeffs"], d["log_values"], d["log_h0"])
    saved = api.parallel_scan_log_bwd(d["log_coeffs"], d["log_values"], d["log_h0"], h, d["grad_h"])
    rec = api.parallel_scan_log_bwd(d["log_coeffs"], d["log_values"], d["log_h0"], None, d["grad_h"])
    b.mgs_check()
    lc, lv, l0, g = (_cpu(d[k]) for k in ("log_coeffs", "log_values", "log_h0", "grad_h"))
    assert_close("h", h, oracle.psl_fwd(lc, lv, l0), T)
    rlc, rlv, rl0 = oracle.psl_bwd(lc, lv, l0, g)
    for got in (saved, rec):
        assert_close("d_log_coeffs", got[0], rlc, T)
        assert_close("d_log_values", got[1], rlv, T)
        if h0:
            assert_close("d_log_h0", got[2], rl0, T)


LIN = [(int(R.integers(1, 5)), int(R.integers(1, 900)), 4 * int(R.integers(1, 40))) for _ in range(6)]


@pytest.mark.parametrize("B,T,D", LIN)
def test_random_linear_scan(B, T, D):
    d = _cuda(inputs.linear_inputs(B, T, D, seed=B * 17 + T + D))
    h = api.linear_scan_fwd(d["a"], d["b"], d["h0"])
    da, db, dh0 = api.linear_scan_bwd(d["a"], d["h0"], h, d["grad_h"], need_dh0=True)
    b.mgs_check()
    a, bb, g, z0 = (_cpu(d[k]) for k in ("a", "b", "grad_h", "h0"))
    assert_close("h", h, oracle.linear_fwd(a, bb, z0), T)
    ra, rb, r0 = oracle.linear_bwd(a, bb, z0, g)
    assert_close("da", da, ra, T)
    assert_close("db", db, rb, T)
    assert_close("dh0", dh0, r0, T)


GIV = [(int(R.integers(1, 5)), int(R.integers(1, 600)), int(R.integers(1, 12)), bool(R.integers(0, 2)))
       for _ in range(8)]


@pytest.mark.parametrize("B,T,H,with_a", GIV)
def test_random_givens_scans(B, T, H, with_a):
    d = _cuda(inputs.givens_affine_inputs(B, T, H, 8, seed=B * 3 + T * 5 + H, h0="normal", with_a=with_a))
    h = api.givens_affine_scan_fwd(d["theta"], d["a"], d["b"], d["h0"])
    dth, da, dbv, dh0 = api.givens_affine_scan_bwd(d["theta"], d["a"], d["h0"], h, d["grad_h"])
    P = api.givens_matrix_scan_fwd(d["theta"])
    G = torch.randn_like(P)
    dthm = api.givens_matrix_scan_bwd(d["theta"], P, G)
    b.mgs_check()
    th, a, bb, z0, g = (_cpu(d[k]) for k in ("theta", "a", "b", "h0", "grad_h"))
    assert_close("h", h, oracle.gas_fwd(th, a, bb, z0), T)
    rth, ra, rb, r0 = oracle.gas_bwd(th, a, bb, z0, g)
    assert_close("d_theta", dth, rth, T)
    assert_close("db", dbv, rb, T)
    assert_close("dh0", dh0, r0, T)
    if with_a:
        assert_close("da", da, ra, T)
    assert_close("P", P, oracle.gms_fwd(th), T)
    assert_close("d_theta (matrix)", dthm, oracle.gms_bwd(th, _cpu(G)), T)


DEL = [(int(R.integers(1, 4)), int(R.integers(1, 300)), int(R.integers(1, 4)), bool(R.integers(0, 2)))
       for _ in range(6)]


@pytest.mark.parametrize("B,T,H,S0", DEL)
def test_random_delta_rule(B, T, H, S0):
    d = _cuda(inputs.delta_inputs(B, T, H, 64, seed=B * 11 + T + H, with_S0=S0))
    o, ST = api.delta_scan_fwd(d["q"], d["k"], d["v"], d["beta"], d["S0"], want_state=True)
    b.mgs_check()
    ro, rST = oracle.delta_fwd(*(_cpu(d[k]) for k in ("q", "k", "v", "beta", "S0")), want_state=True)
    assert_close("o", o, ro, T)
    assert_close("S_T", ST, rST, T)
