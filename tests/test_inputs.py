"""Checks of the seeded input generators against independent constructions."""
import math

import numpy as np
import torch

from scan_linear_recurrences_gb300 import inputs


def test_haar_matches_householder_qr_with_sign_fix():
    g = torch.Generator().manual_seed(3)
    G = torch.randn((500, 8, 8), generator=g, dtype=torch.float64)
    Q = inputs.haar_orthogonal(G).numpy()
    Qn, Rn = np.linalg.qr(G.numpy())
    Qn = Qn * np.sign(np.diagonal(Rn, axis1=-2, axis2=-1))[:, None, :]
    np.testing.assert_allclose(Q, Qn, atol=1e-12)


def test_givens_mesh_matches_explicit_rotation_product():
    k = 8
    g = torch.Generator().manual_seed(4)
    theta = (torch.rand((20, k * (k - 1) // 2), generator=g, dtype=torch.float64) * 2 - 1) * math.pi
    A = inputs.givens_mesh(theta, k).numpy()
    th = theta.numpy()
    for n in range(20):
        M = np.eye(k)
        idx = 0
        for layer in range(1, k + 1):
            L = np.eye(k)
            for i in range(0 if layer % 2 else 1, k - 1, 2):
                R = np.eye(k)
                c, s = np.cos(th[n, idx]), np.sin(th[n, idx])
                R[i, i], R[i, i + 1], R[i + 1, i], R[i + 1, i + 1] = c, -s, s, c
                L = R @ L  # rotations of one layer act on disjoint pairs, so they commute
                idx += 1
            M = L @ M
        np.testing.assert_allclose(A[n], M, atol=1e-13)
        np.testing.assert_allclose(np.linalg.det(A[n]), 1.0, atol=1e-12)


def test_mas_inputs_structure():
    d = inputs.mas_inputs(2, 300, 3, 8, seed=1, h0="normal")
    A = d["A"].double().numpy()
    # A = Q diag(a): column norms are the a_j in (0, 1), and A^T A is diagonal
    AtA = np.einsum("...ji,...jk->...ik", A, A)
    off = AtA - np.eye(8) * np.diagonal(AtA, axis1=-2, axis2=-1)[..., None, :]
    assert np.abs(off).max() < 1e-6
    a = np.sqrt(np.diagonal(AtA, axis1=-2, axis2=-1))
    assert a.min() > 0 and a.max() < 1
    assert d["h0"].shape == (2, 3, 8) and d["grad_h"].shape == (2, 300, 3, 8)
    # deterministic in the seed
    d2 = inputs.mas_inputs(2, 300, 3, 8, seed=1, h0="normal")
    assert torch.equal(d["A"], d2["A"]) and torch.equal(d["b"], d2["b"])
    assert inputs.mas_inputs(1, 4, 1, 8, seed=1)["h0"] is None


def test_psl_inputs_gate_identities():
    d = inputs.psl_inputs(2, 300, 16, seed=2)
    lc = d["log_coeffs"].double().numpy()
    assert lc.max() < 0  # 1 - sigmoid(u) in (0, 1)
    assert d["log_h0"].shape == (2, 16)
    assert np.isfinite(d["log_values"].numpy()).all()


def test_workloads_table():
    w = inputs.WORKLOADS
    assert (w[1].B, w[1].T, w[1].H, w[1].k) == (128, 64, 8, 8)
    assert (w[2].B, w[2].T, w[2].H, w[2].k) == (16, 1024, 8, 8)
    assert (w[3].B, w[3].T, w[3].H) == (64, 4096, 1024)
    assert (w[4].B, w[4].T, w[4].H, w[4].k) == (32, 8192, 64, 8)
    assert len({x.seed for x in w.values()}) == 5
