"""Pins for the float64 oracle: each test checks it against something other than
itself (closed forms, invariants, brute force in a different loop order, special
cases that reduce to another primitive, hand-worked fixtures, finite
differences and forward-mode tangents).  CPU only."""
import json
import os

import numpy as np
import pytest

import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng(1234)


def _haar(n, k, r):
    G = r.standard_normal((n, k, k))
    Q, R = np.linalg.qr(G)
    return Q * np.sign(np.diagonal(R, axis1=-2, axis2=-1))[..., None, :]


def _rand_mas(B, T, H, K, r, h0=True, scale=0.6):
    A = r.standard_normal((B, T, H, K, K)) * (scale / np.sqrt(K))
    b = r.standard_normal((B, T, H, K))
    h0v = r.standard_normal((B, H, K)) if h0 else None
    g = r.standard_normal((B, T, H, K))
    return A, b, h0v, g


# --------------------------------------------------------------- golden, hand-worked
def test_mas_hand_worked_example():
    d = json.load(open(os.path.join(GOLD, "mas_k2_worked.json")))
    A = np.array(d["A"], float)[None, :, None]
    b = np.array(d["b"], float)[None, :, None]
    h0 = np.array(d["h0"], float)[None, None]
    g = np.array(d["g"], float)[None, :, None]
    h = oracle.mas_fwd(A, b, h0)
    assert np.array_equal(h[0, :, 0], np.array(d["h"], float))
    assert np.sum(h * g) == d["loss"]
    dA, db, dh0 = oracle.mas_bwd(A, b, h0, g)
    assert np.array_equal(db[0, :, 0], np.array(d["db"], float))
    assert np.array_equal(dA[0, :, 0], np.array(d["dA"], float))
    assert np.array_equal(dh0[0, 0], np.array(d["dh0"], float))


def test_psl_hand_worked_example():
    d = json.load(open(os.path.join(GOLD, "psl_worked.json")))
    lc = np.full((1, 3, 1), np.log(d["e_lc"]))
    lv = np.log(np.array(d["e_lv"], float)).reshape(1, 3, 1)
    l0 = np.full((1, 1), np.log(d["h0"]))
    g = np.array(d["g"], float).reshape(1, 3, 1)
    h = oracle.psl_fwd(lc, lv, l0)
    np.testing.assert_allclose(h.ravel(), d["h"], rtol=1e-14)
    dlc, dlv, dl0 = oracle.psl_bwd(lc, lv, l0, g)
    np.testing.assert_allclose(dlv.ravel(), d["d_lv"], rtol=1e-14)
    np.testing.assert_allclose(dlc.ravel(), d["d_lc"], rtol=1e-14)
    np.testing.assert_allclose(dl0.ravel(), [d["d_log_h0"]], rtol=1e-14)


def test_ms_quarter_turns():
    # two 90-degree rotations compose to -I; four to I (exact in binary fp)
    R = np.array([[0.0, -1.0], [1.0, 0.0]])
    A = np.broadcast_to(R, (1, 4, 1, 2, 2)).copy()
    P = oracle.ms_fwd(A)
    assert np.array_equal(P[0, 0, 0], R)
    assert np.array_equal(P[0, 1, 0], -np.eye(2))
    assert np.array_equal(P[0, 2, 0], -R)
    assert np.array_equal(P[0, 3, 0], np.eye(2))


# --------------------------------------------------------------- mas forward
@pytest.mark.parametrize("K", [1, 3, 8])
def test_mas_constant_scalar_closed_form(K):
    """A_t = a I: h_t = a^t h0 + sum_s a^{t-s} b_s; with constant b also the
    geometric closed form a^t h0 + b (1 - a^t)/(1 - a)."""
    B, T, H = 2, 40, 3
    a = 0.83
    A = np.broadcast_to(a * np.eye(K), (B, T, H, K, K)).copy()
    bconst = rng.standard_normal((B, 1, H, K))
    b = np.broadcast_to(bconst, (B, T, H, K)).copy()
    h0 = rng.standard_normal((B, H, K))
    h = oracle.mas_fwd(A, b, h0)
    t = np.arange(1, T + 1).reshape(1, T, 1, 1)
    closed = a ** t * h0[:, None] + bconst * (1 - a ** t) / (1 - a)
    np.testing.assert_allclose(h, closed, rtol=1e-12, atol=1e-12)
    # varying b: explicit power sum
    b2 = rng.standard_normal((B, T, H, K))
    h2 = oracle.mas_fwd(A, b2, h0)
    for tt in range(T):
        ref = a ** (tt + 1) * h0 + sum(a ** (tt - s) * b2[:, s] for s in range(tt + 1))
        np.testing.assert_allclose(h2[:, tt], ref, rtol=1e-12, atol=1e-12)


def test_mas_orthogonal_preserves_norm():
    B, T, H, K = 2, 50, 3, 8
    A = _haar(B * T * H, K, rng).reshape(B, T, H, K, K)
    h0 = rng.standard_normal((B, H, K))
    h = oracle.mas_fwd(A, np.zeros((B, T, H, K)), h0)
    np.testing.assert_allclose(np.linalg.norm(h, axis=-1),
                               np.broadcast_to(np.linalg.norm(h0, axis=-1)[:, None], (B, T, H)),
                               rtol=1e-12)


@pytest.mark.parametrize("K", [1, 2, 5, 8])
def test_mas_brute_force_products(K):
    """h_t = (A_t...A_1) h0 + sum_s (A_t...A_{s+1}) b_s, via explicit matrix
    products (numpy matmul), a different loop order than the recurrence."""
    B, T, H = 2, 9, 2
    A, b, h0, _ = _rand_mas(B, T, H, K, rng, scale=1.1)
    h = oracle.mas_fwd(A, b, h0)
    for bb in range(B):
        for hd in range(H):
            for t in range(T):
                acc = np.zeros(K)
                for s in range(-1, t + 1):
                    M = np.eye(K)
                    for u in range(s + 1, t + 1):
                        M = A[bb, u, hd] @ M
                    acc += M @ (h0[bb, hd] if s == -1 else b[bb, s, hd])
                np.testing.assert_allclose(h[bb, t, hd], acc, rtol=1e-11, atol=1e-11)


def test_mas_null_h0_equals_zero_h0():
    A, b, _, _ = _rand_mas(2, 7, 3, 4, rng)
    assert np.array_equal(oracle.mas_fwd(A, b, None), oracle.mas_fwd(A, b, np.zeros((2, 3, 4))))


def test_mas_diagonal_reduces_to_log_scan():
    """Diagonal positive A with positive b, h0: each coordinate is an
    independent scalar recurrence, i.e. parallel_scan_log with lc = log a,
    lv = log b, log_h0 = log h0."""
    B, T, H, K = 2, 30, 2, 4
    a = rng.uniform(0.2, 1.3, (B, T, H, K))
    b = rng.uniform(0.1, 2.0, (B, T, H, K))
    h0 = rng.uniform(0.1, 2.0, (B, H, K))
    A = np.zeros((B, T, H, K, K))
    idx = np.arange(K)
    A[..., idx, idx] = a
    h = oracle.mas_fwd(A, b, h0)
    # channels: D = H*K
    hp = oracle.psl_fwd(np.log(a).reshape(B, T, H * K), np.log(b).reshape(B, T, H * K),
                        np.log(h0).reshape(B, H * K))
    np.testing.assert_allclose(h.reshape(B, T, H * K), hp, rtol=1e-12)


def test_mas_equals_augmented_matrix_scan():
    """[[A_t, b_t], [0, 1]] prefix products applied to [h0; 1] give [h_t; 1]."""
    B, T, H, K = 2, 20, 3, 5
    A, b, h0, _ = _rand_mas(B, T, H, K, rng, scale=0.9)
    Aug = np.zeros((B, T, H, K + 1, K + 1))
    Aug[..., :K, :K] = A
    Aug[..., :K, K] = b
    Aug[..., K, K] = 1.0
    P = oracle.ms_fwd(Aug)
    v = np.concatenate([h0, np.ones((B, H, 1))], -1)
    out = np.einsum("bthij,bhj->bthi", P, v)
    np.testing.assert_allclose(out[..., :K], oracle.mas_fwd(A, b, h0), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(out[..., K], 1.0, rtol=0, atol=1e-13)


# --------------------------------------------------------------- ms forward
def test_ms_last_prefix_is_explicit_product():
    B, T, H, K = 2, 17, 2, 6
    A = rng.standard_normal((B, T, H, K, K)) * 0.5
    P = oracle.ms_fwd(A)
    for bb in range(B):
        for hd in range(H):
            M = np.linalg.multi_dot([A[bb, t, hd] for t in reversed(range(T))])
            np.testing.assert_allclose(P[bb, -1, hd], M, rtol=1e-11, atol=1e-13)
    P1 = oracle.ms_fwd(A[:, :1])
    assert np.array_equal(P1, A[:, :1])


def test_ms_givens_orthogonal_det_one():
    from scan_linear_recurrences_gb300.inputs import ms_inputs
    inp = ms_inputs(2, 64, 2, 8, seed=5)
    P = oracle.ms_fwd(inp["A"])
    I = np.eye(8)
    PtP = np.einsum("...ji,...jk->...ik", P, P)
    np.testing.assert_allclose(PtP, np.broadcast_to(I, PtP.shape), atol=2e-5)  # fp32 inputs
    np.testing.assert_allclose(np.linalg.det(P), 1.0, atol=5e-5)


# --------------------------------------------------------------- psl forward
def test_psl_matches_linear_recurrence_positive():
    B, T, D = 3, 200, 5
    lc = np.log(rng.uniform(0.05, 0.99, (B, T, D)))
    lv = rng.standard_normal((B, T, D))
    l0 = rng.standard_normal((B, D))
    h, lh = oracle.psl_fwd(lc, lv, l0, want_log=True)
    ref = np.empty((B, T, D))
    prev = np.exp(l0)
    for t in range(T):
        prev = np.exp(lc[:, t]) * prev + np.exp(lv[:, t])
        ref[:, t] = prev
    np.testing.assert_allclose(h, ref, rtol=1e-12)
    np.testing.assert_allclose(lh, np.log(ref), rtol=1e-12, atol=1e-13)


def test_psl_matches_heinsen_closed_form():
    """exp(a*_t + logcumsumexp_{s=0..t}(lv_s - a*_s)) with a*_t = cumsum lc,
    the s = 0 term being log h0 with a*_0 = 0 (Heinsen 2023)."""
    B, T, D = 2, 300, 4
    lc = -np.log1p(np.exp(rng.standard_normal((B, T, D))))
    lv = rng.standard_normal((B, T, D))
    l0 = rng.standard_normal((B, D))
    astar = np.cumsum(lc, axis=1)
    terms = np.concatenate([l0[:, None], lv - astar], axis=1)
    lcse = np.logaddexp.accumulate(terms, axis=1)[:, 1:]
    ref = np.exp(astar + lcse)
    np.testing.assert_allclose(oracle.psl_fwd(lc, lv, l0), ref, rtol=1e-10)


def test_psl_constant_closed_form_and_null_h0():
    B, T, D = 1, 50, 3
    a, v, h0 = 0.7, 1.3, 2.5
    lc = np.full((B, T, D), np.log(a))
    lv = np.full((B, T, D), np.log(v))
    t = np.broadcast_to(np.arange(1, T + 1)[None, :, None], (B, T, D))
    h = oracle.psl_fwd(lc, lv, np.full((B, D), np.log(h0)))
    np.testing.assert_allclose(h, a ** t * h0 + v * (1 - a ** t) / (1 - a), rtol=1e-13)
    h_null = oracle.psl_fwd(lc, lv, None)
    np.testing.assert_allclose(h_null, v * (1 - a ** t) / (1 - a), rtol=1e-13)


def test_psl_zero_coefficient_gives_values():
    B, T, D = 2, 10, 3
    lc = np.full((B, T, D), -np.inf)
    lv = rng.standard_normal((B, T, D))
    h = oracle.psl_fwd(lc, lv, rng.standard_normal((B, D)))
    np.testing.assert_allclose(h, np.exp(lv), rtol=1e-15)


# --------------------------------------------------------------- backward: finite differences
def _fd(f, x, eps=1e-6):
    """Central differences of scalar f at x (array), returned with x's shape."""
    grad = np.zeros_like(x)
    it = np.nditer(x, flags=["multi_index"])
    for _ in it:
        i = it.multi_index
        xp = x.copy(); xp[i] += eps
        xm = x.copy(); xm[i] -= eps
        grad[i] = (f(xp) - f(xm)) / (2 * eps)
    return grad


@pytest.mark.parametrize("K", [1, 3, 8])
def test_mas_bwd_finite_differences(K):
    B, T, H = 1, 5, 1
    A, b, h0, g = _rand_mas(B, T, H, K, rng, scale=0.9)
    dA, db, dh0 = oracle.mas_bwd(A, b, h0, g)
    L = lambda A_, b_, h0_: float(np.sum(g * oracle.mas_fwd(A_, b_, h0_)))
    np.testing.assert_allclose(dA, _fd(lambda x: L(x, b, h0), A), rtol=1e-7, atol=1e-8)
    np.testing.assert_allclose(db, _fd(lambda x: L(A, x, h0), b), rtol=1e-7, atol=1e-8)
    np.testing.assert_allclose(dh0, _fd(lambda x: L(A, b, x), h0), rtol=1e-7, atol=1e-8)


@pytest.mark.parametrize("K", [1, 3, 8])
def test_ms_bwd_finite_differences(K):
    B, T, H = 1, 4, 1
    A = rng.standard_normal((B, T, H, K, K)) * (0.9 / np.sqrt(K))
    G = rng.standard_normal((B, T, H, K, K))
    dA = oracle.ms_bwd(A, G)
    fd = _fd(lambda x: float(np.sum(G * oracle.ms_fwd(x))), A)
    np.testing.assert_allclose(dA, fd, rtol=1e-7, atol=1e-8)


def test_psl_bwd_finite_differences():
    B, T, D = 1, 6, 3
    lc = -np.log1p(np.exp(rng.standard_normal((B, T, D))))
    lv = rng.standard_normal((B, T, D))
    l0 = rng.standard_normal((B, D))
    g = rng.standard_normal((B, T, D))
    dlc, dlv, dl0 = oracle.psl_bwd(lc, lv, l0, g)
    L = lambda a, v, z: float(np.sum(g * oracle.psl_fwd(a, v, z)))
    np.testing.assert_allclose(dlc, _fd(lambda x: L(x, lv, l0), lc), rtol=1e-7, atol=1e-8)
    np.testing.assert_allclose(dlv, _fd(lambda x: L(lc, x, l0), lv), rtol=1e-7, atol=1e-8)
    np.testing.assert_allclose(dl0, _fd(lambda x: L(lc, lv, x), l0), rtol=1e-7, atol=1e-8)
    # without an initial state the d_log_h0 output does not exist and h_0 = 0
    dlc0, dlv0, none = oracle.psl_bwd(lc, lv, None, g)
    assert none is None
    np.testing.assert_allclose(dlc0, _fd(lambda x: float(np.sum(g * oracle.psl_fwd(x, lv, None))), lc),
                               rtol=1e-7, atol=1e-8)


# --------------------------------------------------------------- backward: adjoint identities
def test_mas_bwd_linearity_adjoint():
    """h is linear in (b, h0) for fixed A, so <g, h(b, h0)> = <db, b> + <dh0, h0>
    exactly (up to rounding) at a medium size."""
    B, T, H, K = 3, 64, 4, 8
    A, b, h0, g = _rand_mas(B, T, H, K, rng, scale=0.95)
    dA, db, dh0 = oracle.mas_bwd(A, b, h0, g)
    lhs = np.sum(g * oracle.mas_fwd(A, b, h0))
    rhs = np.sum(db * b) + np.sum(dh0 * h0)
    assert abs(lhs - rhs) <= 1e-10 * (abs(lhs) + np.sum(np.abs(db * b)))


def test_mas_bwd_forward_mode_tangent():
    """<g, dh> for a tangent dA computed in forward mode
    (dh_t = A_t dh_{t-1} + dA_t h_{t-1}, dh_0 = 0) equals <dA_oracle, dA>."""
    B, T, H, K = 2, 40, 3, 8
    A, b, h0, g = _rand_mas(B, T, H, K, rng, scale=0.95)
    V = rng.standard_normal(A.shape)
    h = oracle.mas_fwd(A, b, h0)
    hprev = np.concatenate([h0[:, None], h[:, :-1]], axis=1)
    dh = np.zeros((B, H, K))
    tangent = 0.0
    for t in range(T):
        dh = np.einsum("bhij,bhj->bhi", A[:, t], dh) + np.einsum("bhij,bhj->bhi", V[:, t], hprev[:, t])
        tangent += np.sum(g[:, t] * dh)
    dA, _, _ = oracle.mas_bwd(A, b, h0, g)
    assert abs(tangent - np.sum(dA * V)) <= 1e-10 * np.sum(np.abs(dA * V))


def test_mas_bwd_scalar_closed_form():
    """K = 1, constant a: db_s = sum_{t >= s} a^{t-s} g_t, dh0 = a db_1."""
    B, T, H = 2, 30, 2
    a = 0.9
    A = np.full((B, T, H, 1, 1), a)
    b = rng.standard_normal((B, T, H, 1))
    h0 = rng.standard_normal((B, H, 1))
    g = rng.standard_normal((B, T, H, 1))
    _, db, dh0 = oracle.mas_bwd(A, b, h0, g)
    for s in range(T):
        ref = sum(a ** (t - s) * g[:, t] for t in range(s, T))
        np.testing.assert_allclose(db[:, s], ref, rtol=1e-12)
    np.testing.assert_allclose(dh0, a * db[:, 0], rtol=1e-13)


def test_ms_bwd_forward_mode_tangent_and_T1():
    B, T, H, K = 2, 30, 2, 8
    from scan_linear_recurrences_gb300.inputs import ms_inputs
    inp = ms_inputs(B, T, H, K, seed=9)
    A = inp["A"].double().numpy()
    G = inp["grad_P"].double().numpy()
    V = rng.standard_normal(A.shape)
    P = oracle.ms_fwd(A)
    Pprev = np.concatenate([np.broadcast_to(np.eye(K), (B, 1, H, K, K)), P[:, :-1]], axis=1)
    dP = np.zeros((B, H, K, K))
    tangent = 0.0
    for t in range(T):
        dP = A[:, t] @ dP + V[:, t] @ Pprev[:, t]
        tangent += np.sum(G[:, t] * dP)
    dA = oracle.ms_bwd(A, G)
    assert abs(tangent - np.sum(dA * V)) <= 1e-10 * np.sum(np.abs(dA * V))
    # T = 1: P_1 = A_1 so dA_1 = G_1 exactly
    assert np.array_equal(oracle.ms_bwd(A[:, :1], G[:, :1]), G[:, :1])


def test_psl_bwd_forward_mode_tangent():
    B, T, D = 2, 500, 6
    lc = -np.log1p(np.exp(rng.standard_normal((B, T, D))))
    lv = rng.standard_normal((B, T, D))
    l0 = rng.standard_normal((B, D))
    g = rng.standard_normal((B, T, D))
    Vc, Vv, V0 = rng.standard_normal(lc.shape), rng.standard_normal(lv.shape), rng.standard_normal(l0.shape)
    # linear-space tangent: dh_t = a_t dh_{t-1} + (Vc_t a_t h_{t-1}) + Vv_t e^{lv_t}, dh_0 = V0 h_0
    a, v = np.exp(lc), np.exp(lv)
    h = np.exp(l0)
    dh = V0 * h
    tangent = 0.0
    for t in range(T):
        dh_new = a[:, t] * dh + Vc[:, t] * a[:, t] * h + Vv[:, t] * v[:, t]
        h = a[:, t] * h + v[:, t]
        dh = dh_new
        tangent += np.sum(g[:, t] * dh)
    dlc, dlv, dl0 = oracle.psl_bwd(lc, lv, l0, g)
    rhs = np.sum(dlc * Vc) + np.sum(dlv * Vv) + np.sum(dl0 * V0)
    assert abs(tangent - rhs) <= 1e-10 * (np.sum(np.abs(dlc * Vc)) + np.sum(np.abs(dlv * Vv)))


# --------------------------------------------------------------- degenerate shapes
def test_empty_shapes():
    A = np.zeros((2, 0, 3, 4, 4)); b = np.zeros((2, 0, 3, 4))
    assert oracle.mas_fwd(A, b).shape == (2, 0, 3, 4)
    dA, db, dh0 = oracle.mas_bwd(A, b, np.ones((2, 3, 4)), b)
    assert dA.shape == A.shape and np.array_equal(dh0, np.zeros((2, 3, 4)))
    assert oracle.ms_fwd(A).shape == A.shape
    lc = np.zeros((0, 5, 3))
    assert oracle.psl_fwd(lc, lc, np.zeros((0, 3))).shape == (0, 5, 3)


# --------------------------------------------------------------- linear_scan
def test_linear_scan_equals_k1_block_scan_and_closed_form():
    """k = 1 matrix_affine_scan is the same recurrence (separate oracle loops);
    constant a gives the geometric closed form; signed a is allowed."""
    B, T, D = 2, 60, 5
    a = rng.uniform(-0.95, 0.95, (B, T, D))
    b = rng.standard_normal((B, T, D))
    h0 = rng.standard_normal((B, D))
    h = oracle.linear_fwd(a, b, h0)
    hm = oracle.mas_fwd(a[..., None, None], b[..., None], h0[..., None])[..., 0]
    np.testing.assert_allclose(h, hm, rtol=1e-13, atol=1e-14)
    ac = np.full((B, T, D), -0.7)
    bc = np.broadcast_to(b[:, :1], (B, T, D)).copy()
    t = np.broadcast_to(np.arange(1, T + 1)[None, :, None], (B, T, D))
    ref = (-0.7) ** t * h0[:, None] + bc * (1 - (-0.7) ** t) / (1 + 0.7)
    np.testing.assert_allclose(oracle.linear_fwd(ac, bc, h0), ref, rtol=1e-12, atol=1e-12)
    assert np.array_equal(oracle.linear_fwd(a, b, None), oracle.linear_fwd(a, b, np.zeros((B, D))))


def test_linear_scan_bwd_finite_differences_and_tangent():
    B, T, D = 1, 6, 3
    a = rng.uniform(-0.9, 0.9, (B, T, D))
    b = rng.standard_normal((B, T, D))
    h0 = rng.standard_normal((B, D))
    g = rng.standard_normal((B, T, D))
    da, db, dh0 = oracle.linear_bwd(a, b, h0, g)
    L = lambda a_, b_, h_: float(np.sum(g * oracle.linear_fwd(a_, b_, h_)))
    np.testing.assert_allclose(da, _fd(lambda x: L(x, b, h0), a), rtol=1e-7, atol=1e-8)
    np.testing.assert_allclose(db, _fd(lambda x: L(a, x, h0), b), rtol=1e-7, atol=1e-8)
    np.testing.assert_allclose(dh0, _fd(lambda x: L(a, b, x), h0), rtol=1e-7, atol=1e-8)
    # forward-mode tangent in da at a medium size
    B, T, D = 2, 300, 4
    a = rng.uniform(-0.99, 0.99, (B, T, D))
    b = rng.standard_normal((B, T, D)); h0 = rng.standard_normal((B, D)); g = rng.standard_normal((B, T, D))
    V = rng.standard_normal(a.shape)
    h = oracle.linear_fwd(a, b, h0)
    hprev = np.concatenate([h0[:, None], h[:, :-1]], axis=1)
    dh = np.zeros((B, D)); tangent = 0.0
    for tt in range(T):
        dh = a[:, tt] * dh + V[:, tt] * hprev[:, tt]
        tangent += np.sum(g[:, tt] * dh)
    da, _, _ = oracle.linear_bwd(a, b, h0, g)
    assert abs(tangent - np.sum(da * V)) <= 1e-10 * np.sum(np.abs(da * V))
