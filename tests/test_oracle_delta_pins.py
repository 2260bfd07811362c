"""Pins for the oracle's delta rule (DeltaNet, behind DeltaMinGRU): a
hand-worked fixture, reduction of every state row to the pinned
matrix_affine_scan oracle, the chunked WY form (a different algorithm, written
here in numpy), and the rule's own invariants.  CPU only."""
import json
import os

import numpy as np
import pytest

import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng(777)


def _rand(B, T, H, D, r, S0=True):
    def unit(x):
        return x / np.linalg.norm(x, axis=-1, keepdims=True)
    q = unit(r.standard_normal((B, T, H, D)))
    k = unit(r.standard_normal((B, T, H, D)))
    v = r.standard_normal((B, T, H, D))
    beta = 1.0 / (1.0 + np.exp(-r.standard_normal((B, T, H))))
    S = r.standard_normal((B, H, D, D)) / np.sqrt(D) if S0 else None
    return q, k, v, beta, S


def test_delta_hand_worked_example():
    d = json.load(open(os.path.join(GOLD, "delta_d2_worked.json")))
    q = np.array(d["q"], float)[None, :, None]
    k = np.array(d["k"], float)[None, :, None]
    v = np.array(d["v"], float)[None, :, None]
    beta = np.array(d["beta"], float)[None, :, None]
    S0 = np.array(d["S0"], float)[None, None]
    o, ST = oracle.delta_fwd(q, k, v, beta, S0, want_state=True)
    assert np.array_equal(o[0, :, 0], np.array(d["o"], float))
    assert np.array_equal(ST[0, 0], np.array(d["ST"], float))


@pytest.mark.parametrize("D", [1, 3, 8])
def test_delta_rows_are_matrix_affine_scans(D):
    """Row i of the state follows s_t = (I - beta k k^T) s_{t-1} + beta v_t[i] k_t."""
    B, T, H = 2, 7, 2
    q, k, v, beta, S0 = _rand(B, T, H, D, rng)
    A = np.eye(D) - beta[..., None, None] * k[..., :, None] * k[..., None, :]      # [B,T,H,D,D]
    A = np.repeat(A[:, :, :, None], D, axis=3).reshape(B, T, H * D, D, D)         # one lane per (head, row)
    bvec = (beta[..., None, None] * v[..., :, None] * k[..., None, :]).reshape(B, T, H * D, D)
    rows = oracle.mas_fwd(A, bvec, S0.reshape(B, H * D, D)).reshape(B, T, H, D, D)  # S_t
    o_ref = np.einsum("bthij,bthj->bthi", rows, q)
    o, ST = oracle.delta_fwd(q, k, v, beta, S0, want_state=True)
    np.testing.assert_allclose(o, o_ref, atol=1e-12)
    np.testing.assert_allclose(ST, rows[:, -1], atol=1e-12)


def _wy_chunked(q, k, v, beta, S0, C):
    """The chunked WY form (Yang et al. 2024) in float64: per chunk,
    (I + strict_tril(diag(beta) K K^T)) [W | U] = diag(beta) [K | V],
    U' = U - W S^T, O = Q S^T + tril(Q K^T) U', S <- S + U'^T K."""
    B, T, H, D = q.shape
    o = np.empty_like(q)
    ST = np.empty((B, H, D, D))
    for b in range(B):
        for h in range(H):
            S = S0[b, h].copy() if S0 is not None else np.zeros((D, D))
            for c0 in range(0, T, C):
                Q, K, V, bt = q[b, c0:c0 + C, h], k[b, c0:c0 + C, h], v[b, c0:c0 + C, h], beta[b, c0:c0 + C, h]
                n = len(bt)
                A = np.tril(bt[:, None] * (K @ K.T), -1)
                WU = np.linalg.solve(np.eye(n) + A, bt[:, None] * np.concatenate([K, V], axis=1))
                W, U = WU[:, :D], WU[:, D:]
                Up = U - W @ S.T
                o[b, c0:c0 + C, h] = Q @ S.T + np.tril(Q @ K.T) @ Up
                S = S + Up.T @ K
            ST[b, h] = S
    return o, ST


@pytest.mark.parametrize("C", [1, 4, 5, 64])
def test_delta_equals_chunked_wy_form(C):
    q, k, v, beta, S0 = _rand(2, 23, 3, 6, rng)
    o, ST = oracle.delta_fwd(q, k, v, beta, S0, want_state=True)
    o2, ST2 = _wy_chunked(q, k, v, beta, S0, C)
    np.testing.assert_allclose(o, o2, atol=1e-11)
    np.testing.assert_allclose(ST, ST2, atol=1e-11)


def test_delta_zero_beta_keeps_state():
    q, k, v, beta, S0 = _rand(2, 9, 2, 5, rng)
    o, ST = oracle.delta_fwd(q, k, v, np.zeros_like(beta), S0, want_state=True)
    np.testing.assert_allclose(o, np.einsum("bhij,bthj->bthi", S0, q), atol=1e-13)
    np.testing.assert_array_equal(ST, S0)


def test_delta_unit_beta_writes_the_value_at_its_key():
    """With a unit key and beta = 1 the rule overwrites: S_t k_t = v_t."""
    q, k, v, beta, S0 = _rand(2, 12, 2, 6, rng)
    o = oracle.delta_fwd(k, k, v, np.ones_like(beta), S0)
    np.testing.assert_allclose(o, v, atol=1e-12)


def test_delta_linear_in_values_and_initial_state():
    q, k, v1, beta, S1 = _rand(1, 15, 2, 4, rng)
    v2 = rng.standard_normal(v1.shape)
    S2 = rng.standard_normal(S1.shape)
    o = oracle.delta_fwd(q, k, v1 + 2 * v2, beta, S1 - S2)
    o_sum = oracle.delta_fwd(q, k, v1, beta, S1) + 2 * oracle.delta_fwd(q, k, v2, beta, None) \
        - oracle.delta_fwd(q, k, np.zeros_like(v1), beta, S2)
    np.testing.assert_allclose(o, o_sum, atol=1e-12)


def test_delta_null_initial_state_and_empty():
    q, k, v, beta, _ = _rand(1, 5, 1, 3, rng, S0=False)
    np.testing.assert_array_equal(oracle.delta_fwd(q, k, v, beta, None),
                                  oracle.delta_fwd(q, k, v, beta, np.zeros((1, 1, 3, 3))))
    e = np.zeros((2, 0, 1, 3))
    o, ST = oracle.delta_fwd(e, e, e, np.zeros((2, 0, 1)), np.ones((2, 1, 3, 3)), want_state=True)
    assert o.shape == e.shape
    np.testing.assert_array_equal(ST, 1.0)
