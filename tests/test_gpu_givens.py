"""GPU parity of the Givens-mesh (angle-fused) affine and matrix scans against
the float64 oracle: shapes spanning several ring stages, ragged tails, heads
that do not fill a warp, every lanes-per-warp choice of the affine scan, the
pages' lab and long-sequence shapes in full, the degenerate cases, and the
autograd wrappers."""
import pytest
import torch

import oracle
from scan_linear_recurrences_gb300 import _binding as b
from scan_linear_recurrences_gb300 import api, inputs
from scan_linear_recurrences_gb300.build import build

from ._parity import assert_close

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


def _cpu(x):
    return x.cpu() if x is not None else None


def _run_gas(B, T, H, seed, h0, with_a, rows=None):
    d = _cuda(inputs.givens_affine_inputs(B, T, H, 8, seed, device="cpu", h0=h0, with_a=with_a))
    th, a, bb, z0, g = d["theta"], d["a"], d["b"], d["h0"], d["grad_h"]
    h = api.givens_affine_scan_fwd(th, a, bb, z0)
    dth, da, db, dh0 = api.givens_affine_scan_bwd(th, a, z0, h, g, need_dh0=True)
    b.mgs_check()
    sel = slice(None) if rows is None else rows
    pick = lambda x: _cpu(x[sel]) if x is not None else None
    href = oracle.gas_fwd(pick(th), pick(a), pick(bb), pick(z0))
    assert_close("h", h[sel], href, T)
    z0c = pick(z0) if z0 is not None else torch.zeros((len(href), H, 8))
    dthr, dar, dbr, dh0r = oracle.gas_bwd(pick(th), pick(a), pick(bb), z0c, pick(g))
    assert_close("d_theta", dth[sel], dthr, T)
    assert_close("db", db[sel], dbr, T)
    assert_close("dh0", dh0[sel], dh0r, T)
    if a is not None:
        assert_close("da", da[sel], dar, T)
    else:
        assert da is None


@pytest.mark.parametrize("B,T,H,h0,with_a", [
    (1, 1, 1, "normal", True),
    (2, 7, 3, "none", True),
    (3, 130, 5, "normal", False),     # 1 lane per block, 64-step stages, ragged
    (5, 33, 100, "normal", True),     # 2 lanes per block, partial head group
    (128, 64, 8, "normal", True),     # the pages' lab shape: 4 lanes per block
    (2, 45, 1000, "normal", True),    # 8 lanes per block, partial head groups
    (64, 20, 64, "none", True),       # 8 lanes per block, 8-step stages, ragged
    (40, 9, 256, "normal", True),     # 8 lanes per block, a block shorter than a stage
])
def test_givens_affine_scan(B, T, H, h0, with_a):
    _run_gas(B, T, H, seed=900 + B * T + H, h0=h0, with_a=with_a)


@pytest.mark.parametrize("B,T,H,h0,with_a", [
    (2, 300, 3, "normal", True),      # few lanes, long T: time-chunked from the angles
    (1, 517, 4, "none", False),       # ragged chunks, no gate, zero initial state
    (40, 300, 64, "normal", True),    # many lanes, long T: angle-fused kernels
])
def test_givens_affine_scan_long_sequences(B, T, H, h0, with_a):
    _run_gas(B, T, H, seed=980 + B * T + H, h0=h0, with_a=with_a, rows=[0, B - 1])


def test_givens_affine_scan_long_T_shape():
    w = inputs.EXTRA_WORKLOADS[10]
    _run_gas(w.B, w.T, w.H, seed=w.seed, h0=w.h0, with_a=True, rows=[0, 7, w.B - 1])


def _run_gms(B, T, H, seed, rows=None):
    d = _cuda(inputs.givens_matrix_inputs(B, T, H, 8, seed, device="cpu"))
    th, G = d["theta"], d["grad_P"]
    P = api.givens_matrix_scan_fwd(th)
    dth = api.givens_matrix_scan_bwd(th, P, G)
    b.mgs_check()
    sel = slice(None) if rows is None else rows
    assert_close("P", P[sel], oracle.gms_fwd(_cpu(th[sel])), T)
    assert_close("d_theta", dth[sel], oracle.gms_bwd(_cpu(th[sel]), _cpu(G[sel])), T)


@pytest.mark.parametrize("B,T,H", [(1, 1, 1), (2, 50, 3), (3, 33, 9), (128, 64, 8), (2, 300, 4)])
def test_givens_matrix_scan(B, T, H):
    _run_gms(B, T, H, seed=950 + B * T + H)


@pytest.mark.parametrize("B,T,H", [(2, 300, 3), (1, 517, 5)])
def test_givens_matrix_scan_few_lanes_long_T(B, T, H):
    _run_gms(B, T, H, seed=990 + B * T + H)


def test_givens_matrix_scan_long_T_shape():
    w = inputs.EXTRA_WORKLOADS[12]
    _run_gms(w.B, w.T, w.H, seed=w.seed, rows=[0, w.B - 1])


def test_givens_matches_materialised_scans():
    """The angle-fused ops against the matrix ops fed the same meshes as
    matrices (both on the GPU, both checked against the oracle elsewhere)."""
    d = _cuda(inputs.givens_affine_inputs(4, 40, 8, 8, seed=77, h0="normal"))
    A = (inputs.givens_mesh(d["theta"].double().cpu(), 8) * d["a"].double().cpu().unsqueeze(-2)).float().cuda()
    h1 = api.givens_affine_scan_fwd(d["theta"], d["a"], d["b"], d["h0"])
    h2 = api.matrix_affine_scan_fwd(A, d["b"], d["h0"])
    b.mgs_check()
    assert_close("h fused vs materialised", h1, h2.double().cpu().numpy(), 40)


def test_givens_empty_and_errors():
    th = torch.empty((0, 5, 8, 28), device="cuda")
    v = torch.empty((0, 5, 8, 8), device="cuda")
    assert api.givens_affine_scan_fwd(th, None, v).shape == (0, 5, 8, 8)
    assert api.givens_matrix_scan_fwd(th).shape == (0, 5, 8, 8, 8)
    # T = 0: dh0 = 0
    th = torch.empty((2, 0, 3, 28), device="cuda")
    v = torch.empty((2, 0, 3, 8), device="cuda")
    z0 = torch.randn((2, 3, 8), device="cuda")
    _, _, _, dz = api.givens_affine_scan_bwd(th, None, z0, v, v)
    b.mgs_check()
    assert torch.equal(dz, torch.zeros_like(z0))
    # k other than 8 is unsupported; da without a is an argument error
    t4 = torch.zeros((1, 2, 1, 6), device="cuda")
    with pytest.raises(b.MGSError) as e:
        b.mgs_givens_matrix_scan_fwd(t4, torch.empty((1, 2, 1, 4, 4), device="cuda"), 1, 2, 1, 4)
    assert e.value.status == b.MGS_ERR_UNSUPPORTED
    d = _cuda(inputs.givens_affine_inputs(1, 3, 1, 8, seed=5))
    with pytest.raises(b.MGSError) as e:
        b.mgs_givens_affine_scan_bwd(d["theta"], None, None, d["b"], d["grad_h"], torch.empty_like(d["theta"]),
                                     torch.empty_like(d["b"]), torch.empty_like(d["b"]), None, 1, 3, 1, 8)
    assert e.value.status == b.MGS_ERR_INVALID_ARG


def test_givens_autograd_wrappers():
    d = _cuda(inputs.givens_affine_inputs(2, 30, 3, 8, seed=11, h0="normal"))
    th = d["theta"].clone().requires_grad_(True)
    a = d["a"].clone().requires_grad_(True)
    bb = d["b"].clone().requires_grad_(True)
    z0 = d["h0"].clone().requires_grad_(True)
    (api.givens_affine_scan(th, a, bb, z0) * d["grad_h"]).sum().backward()
    dthr, dar, dbr, dh0r = oracle.gas_bwd(*(_cpu(d[k]) for k in ("theta", "a", "b", "h0", "grad_h")))
    assert_close("d_theta", th.grad, dthr, 30)
    assert_close("da", a.grad, dar, 30)
    assert_close("db", bb.grad, dbr, 30)
    assert_close("dh0", z0.grad, dh0r, 30)
    m = _cuda(inputs.givens_matrix_inputs(2, 25, 5, 8, seed=12))
    thm = m["theta"].clone().requires_grad_(True)
    (api.givens_matrix_scan(thm) * m["grad_P"]).sum().backward()
    assert_close("d_theta (matrix)", thm.grad, oracle.gms_bwd(_cpu(m["theta"]), _cpu(m["grad_P"])), 25)
