"""Pins for the oracle's Givens-mesh scans (GivensMinGRU's angle-parameterised
transition): a hand-worked fixture, the K=2 closed form, explicit products of
textbook Givens matrices built here independently, reduction to the pinned
matrix_affine_scan / matrix_scan oracles, invariants of orthogonal products,
finite differences and directional derivatives.  CPU only."""
import json
import math
import os

import numpy as np
import pytest

import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng(4321)


def _givens(K, p, th):
    """The K x K plane rotation of angle th on coordinates (p, p+1)."""
    R = np.eye(K)
    c, s = math.cos(th), math.sin(th)
    R[p, p], R[p, p + 1], R[p + 1, p], R[p + 1, p + 1] = c, -s, s, c
    return R


def _mesh(theta, K):
    """Brick-wall mesh as an explicit matrix product: layer l = 1..K holds the
    rotations of pairs (0,1),(2,3).. (odd l) or (1,2),(3,4).. (even l)."""
    M = np.eye(K)
    n = 0
    for layer in range(1, K + 1):
        L = np.eye(K)
        for p in range(0 if layer % 2 else 1, K - 1, 2):
            L = _givens(K, p, theta[n]) @ L
            n += 1
        M = L @ M
    assert n == len(theta)
    return M


def _meshes(theta, K):
    B, T, H, N = theta.shape
    out = np.empty((B, T, H, K, K))
    for idx in np.ndindex(B, T, H):
        out[idx] = _mesh(theta[idx], K)
    return out


def _rand(B, T, H, K, r, with_a=True, h0=True):
    th = r.uniform(-math.pi, math.pi, (B, T, H, K * (K - 1) // 2))
    a = r.uniform(0.2, 1.0, (B, T, H, K)) if with_a else None
    b = r.standard_normal((B, T, H, K))
    h0v = r.standard_normal((B, H, K)) if h0 else None
    g = r.standard_normal((B, T, H, K))
    return th, a, b, h0v, g


# --------------------------------------------------------------- forward
def test_givens_hand_worked_example():
    d = json.load(open(os.path.join(GOLD, "givens_k3_worked.json")))
    th = np.array(d["theta_over_pi"], float)[None, :, None] * math.pi
    a = np.array(d["a"], float)[None, :, None]
    b = np.array(d["b"], float)[None, :, None]
    h0 = np.array(d["h0"], float)[None, None]
    h = oracle.gas_fwd(th, a, b, h0)
    np.testing.assert_allclose(h[0, :, 0], np.array(d["h"], float), atol=1e-14)


def test_gms_k2_is_rotation_by_cumulative_angle():
    th = rng.uniform(-3, 3, (2, 40, 3, 1))
    P = oracle.gms_fwd(th)
    c = np.cumsum(th[..., 0], axis=1)
    np.testing.assert_allclose(P[..., 0, 0], np.cos(c), atol=1e-13)
    np.testing.assert_allclose(P[..., 1, 0], np.sin(c), atol=1e-13)
    np.testing.assert_allclose(P[..., 0, 1], -np.sin(c), atol=1e-13)
    np.testing.assert_allclose(P[..., 1, 1], np.cos(c), atol=1e-13)


@pytest.mark.parametrize("K", [3, 4, 5, 8])
def test_gms_matches_explicit_rotation_products(K):
    th = rng.uniform(-math.pi, math.pi, (2, 6, 2, K * (K - 1) // 2))
    P = oracle.gms_fwd(th)
    G = _meshes(th, K)
    for bb in range(2):
        for hd in range(2):
            Q = np.eye(K)
            for t in range(6):
                Q = G[bb, t, hd] @ Q
                np.testing.assert_allclose(P[bb, t, hd], Q, atol=1e-13)


def test_gms_orthogonal_with_unit_determinant():
    K = 8
    th = rng.uniform(-math.pi, math.pi, (1, 50, 2, 28))
    P = oracle.gms_fwd(th)
    PtP = np.einsum("...ji,...jk->...ik", P, P)
    np.testing.assert_allclose(PtP, np.broadcast_to(np.eye(K), PtP.shape), atol=1e-12)
    np.testing.assert_allclose(np.linalg.det(P), 1.0, atol=1e-12)


@pytest.mark.parametrize("K,with_a", [(2, True), (3, False), (8, True), (8, False)])
def test_gas_reduces_to_matrix_affine_scan(K, with_a):
    th, a, b, h0, g = _rand(2, 9, 3, K, rng, with_a=with_a)
    A = _meshes(th, K)
    if a is not None:
        A = A * a[..., None, :]  # G diag(a): column j scaled by a_j
    np.testing.assert_allclose(oracle.gas_fwd(th, a, b, h0), oracle.mas_fwd(A, b, h0), atol=1e-12)
    dth, da, db, dh0 = oracle.gas_bwd(th, a, b, h0, g)
    _, dbm, dh0m = oracle.mas_bwd(A, b, h0, g)
    np.testing.assert_allclose(db, dbm, atol=1e-12)
    np.testing.assert_allclose(dh0, dh0m, atol=1e-12)
    assert (da is None) == (a is None)


def test_gas_null_a_and_null_h0():
    th, a, b, h0, g = _rand(1, 7, 2, 8, rng)
    ones = np.ones_like(a)
    np.testing.assert_array_equal(oracle.gas_fwd(th, None, b, h0), oracle.gas_fwd(th, ones, b, h0))
    np.testing.assert_array_equal(oracle.gas_fwd(th, a, b, None), oracle.gas_fwd(th, a, b, np.zeros_like(h0)))
    r1 = oracle.gas_bwd(th, None, b, h0, g)
    r2 = oracle.gas_bwd(th, ones, b, h0, g)
    for x, y in zip((r1[0], r1[2], r1[3]), (r2[0], r2[2], r2[3])):
        np.testing.assert_array_equal(x, y)


def test_gas_rotation_only_preserves_norm():
    th, _, b, h0, _ = _rand(2, 200, 2, 8, rng)
    h = oracle.gas_fwd(th, None, np.zeros_like(b), h0)
    np.testing.assert_allclose(np.linalg.norm(h, axis=-1),
                               np.broadcast_to(np.linalg.norm(h0, axis=-1)[:, None], h.shape[:-1]), rtol=1e-12)


def test_gas_unit_start_gives_matrix_scan_columns():
    K = 8
    th = rng.uniform(-math.pi, math.pi, (1, 12, 1, 28))
    P = oracle.gms_fwd(th)
    zeros = np.zeros((1, 12, 1, K))
    for j in range(K):
        h0 = np.zeros((1, 1, K))
        h0[0, 0, j] = 1.0
        np.testing.assert_allclose(oracle.gas_fwd(th, None, zeros, h0)[0, :, 0], P[0, :, 0, :, j], atol=1e-13)


# --------------------------------------------------------------- backward
def _fd(f, x, eps=1e-6):
    grad = np.zeros_like(x)
    for i in np.ndindex(x.shape):
        xp = x.copy(); xp[i] += eps
        xm = x.copy(); xm[i] -= eps
        grad[i] = (f(xp) - f(xm)) / (2 * eps)
    return grad


@pytest.mark.parametrize("K", [2, 3, 4, 8])
def test_gas_bwd_finite_differences(K):
    th, a, b, h0, g = _rand(1, 4, 1, K, rng)
    dth, da, db, dh0 = oracle.gas_bwd(th, a, b, h0, g)
    L = lambda th_, a_, b_, h0_: float(np.sum(g * oracle.gas_fwd(th_, a_, b_, h0_)))
    np.testing.assert_allclose(dth, _fd(lambda x: L(x, a, b, h0), th), rtol=1e-7, atol=1e-8)
    np.testing.assert_allclose(da, _fd(lambda x: L(th, x, b, h0), a), rtol=1e-7, atol=1e-8)
    np.testing.assert_allclose(db, _fd(lambda x: L(th, a, x, h0), b), rtol=1e-7, atol=1e-8)
    np.testing.assert_allclose(dh0, _fd(lambda x: L(th, a, b, x), h0), rtol=1e-7, atol=1e-8)


@pytest.mark.parametrize("K", [2, 3, 8])
def test_gms_bwd_finite_differences(K):
    th = rng.uniform(-math.pi, math.pi, (1, 4, 1, K * (K - 1) // 2))
    G = rng.standard_normal((1, 4, 1, K, K))
    dth = oracle.gms_bwd(th, G)
    np.testing.assert_allclose(dth, _fd(lambda x: float(np.sum(G * oracle.gms_fwd(x))), th),
                               rtol=1e-7, atol=1e-8)


def test_directional_derivatives_at_longer_T():
    """<grad, v> against the central difference of the loss along v, for all
    inputs at once, on a shape with several lanes and T = 40."""
    th, a, b, h0, g = _rand(2, 40, 2, 8, rng)
    v = [rng.standard_normal(x.shape) for x in (th, a, b, h0)]
    dth, da, db, dh0 = oracle.gas_bwd(th, a, b, h0, g)
    eps = 1e-6
    L = lambda s: float(np.sum(g * oracle.gas_fwd(th + s * v[0], a + s * v[1], b + s * v[2], h0 + s * v[3])))
    fd = (L(eps) - L(-eps)) / (2 * eps)
    an = sum(float(np.sum(x * y)) for x, y in zip((dth, da, db, dh0), v))
    assert abs(fd - an) <= 1e-6 * max(1.0, abs(an))
    G = rng.standard_normal((2, 40, 2, 8, 8))
    dthm = oracle.gms_bwd(th, G)
    Lm = lambda s: float(np.sum(G * oracle.gms_fwd(th + s * v[0])))
    fdm = (Lm(eps) - Lm(-eps)) / (2 * eps)
    anm = float(np.sum(dthm * v[0]))
    assert abs(fdm - anm) <= 1e-6 * max(1.0, abs(anm))


def test_empty_shapes():
    th = np.zeros((0, 3, 2, 28))
    assert oracle.gms_fwd(th).shape == (0, 3, 2, 8, 8)
    th = np.zeros((2, 0, 2, 28))
    b = np.zeros((2, 0, 2, 8))
    assert oracle.gas_fwd(th, None, b, None).shape == (2, 0, 2, 8)
    dth, da, db, dh0 = oracle.gas_bwd(th, None, b, np.ones((2, 2, 8)), b)
    assert dth.shape == th.shape and da is None
    np.testing.assert_array_equal(dh0, 0.0)
