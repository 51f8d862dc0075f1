"""Pins of the rank-r truncation oracle ("How much of a Gated DeltaNet state
is used" blog, Sec. 3) that do not lean on the SVD routine it calls."""
import numpy as np
import pytest

import oracle


def _orthonormal(rng, n, m):
    Q, R = np.linalg.qr(rng.standard_normal((n, m)))
    return Q * np.sign(np.diag(R))[None, :]


def test_constructed_spectrum():
    """S = A diag(sigma) B^T with A, B orthonormal by construction: the
    truncation is the first r terms, whatever the routine."""
    rng = np.random.default_rng(0)
    V, K = 12, 9
    A, Bm = _orthonormal(rng, V, K), _orthonormal(rng, K, K)
    sigma = np.array([9.0, 7.5, 6.0, 4.0, 3.0, 2.0, 1.0, 0.5, 0.1])
    S = (A * sigma) @ Bm.T
    for r in (1, 3, 5, 8):
        want = (A[:, :r] * sigma[:r]) @ Bm[:, :r].T
        assert np.allclose(oracle.truncate_state(S, r), want, atol=1e-12)
    assert np.array_equal(oracle.truncate_state(S, 9), S)


def test_low_rank_state_unchanged_and_idempotent():
    rng = np.random.default_rng(1)
    S = rng.standard_normal((2, 3, 10, 3)) @ rng.standard_normal((2, 3, 3, 8))  # rank 3
    for r in (3, 4, 7):
        assert np.allclose(oracle.truncate_state(S, r), S, atol=1e-10)
    X = rng.standard_normal((4, 10, 8))
    once = oracle.truncate_state(X, 2)
    assert np.allclose(oracle.truncate_state(once, 2), once, atol=1e-12)
    assert np.linalg.matrix_rank(once[0], tol=1e-9) == 2


def _problem(rng, B=1, T=40, H=2, K=6, V=5):
    q = rng.standard_normal((B, T, H, K))
    k = rng.standard_normal((B, T, H, K))
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, T, H, V))
    alpha = rng.uniform(0.6, 1.0, size=(B, T, H))
    beta = rng.uniform(0.1, 1.0, size=(B, T, H))
    return q, k, v, alpha, beta


@pytest.mark.parametrize("seg_len,r", [(40, 1), (100, 2), (10, 5)])
def test_no_truncation_cases_equal_the_plain_recurrence(seg_len, r):
    """One segment covering the sequence, or r = min(V, K): nothing is cut."""
    q, k, v, alpha, beta = _problem(np.random.default_rng(2))
    o0, S0 = oracle.recurrence(q, k, v, alpha, beta)
    o1, S1 = oracle.recurrence_truncated(q, k, v, alpha, beta, seg_len=seg_len, r=r)
    if seg_len >= 40 or r >= 5:
        assert np.allclose(o1, o0, atol=1e-12) and np.allclose(S1, S0, atol=1e-12)
    else:
        assert not np.allclose(S1, S0)


def test_memory_older_than_a_segment_keeps_r_directions():
    """Second segment with no writes (beta = 0) and no decay (alpha = 1): the
    final state is exactly the truncated boundary state, of rank r, and the
    outputs there read it: o_t = S_r q_t."""
    rng = np.random.default_rng(3)
    q, k, v, alpha, beta = _problem(rng, T=20, H=1, K=6, V=5)
    alpha[:, 10:] = 1.0
    beta[:, 10:] = 0.0
    _, S_mid = oracle.recurrence(q[:, :10], k[:, :10], v[:, :10], alpha[:, :10], beta[:, :10])
    for r in (1, 2, 3):
        o, ST = oracle.recurrence_truncated(q, k, v, alpha, beta, seg_len=10, r=r)
        Sr = oracle.truncate_state(S_mid, r)
        assert np.allclose(ST, Sr, atol=1e-12)
        assert np.linalg.matrix_rank(ST[0, 0], tol=1e-9) == r
        assert np.allclose(o[:, 10:], np.einsum("bhvk,bthk->bthv", Sr, q[:, 10:]), atol=1e-12)


def test_truncation_error_is_the_discarded_energy():
    """Eckart-Young on a constructed spectrum: |S - S_r|_F^2 = sum of the
    discarded sigma^2, and no other rank-r projection of the rows does better
    (checked against random rank-r projections)."""
    rng = np.random.default_rng(4)
    A, Bm = _orthonormal(rng, 8, 8), _orthonormal(rng, 8, 8)
    sigma = np.linspace(4.0, 0.5, 8)
    S = (A * sigma) @ Bm.T
    for r in (2, 5):
        err = np.sum((S - oracle.truncate_state(S, r)) ** 2)
        assert np.isclose(err, np.sum(sigma[r:] ** 2), rtol=1e-12)
        for _ in range(20):
            P = _orthonormal(rng, 8, r)
            assert np.sum((S - P @ (P.T @ S)) ** 2) >= err - 1e-12


def test_final_state_and_initial_state_are_not_truncated():
    """Only boundaries inside the sequence cut: a full-rank S0 with one
    segment passes through untouched, and writes after the last boundary
    raise the final rank above r."""
    rng = np.random.default_rng(5)
    q, k, v, alpha, beta = _problem(rng, T=20, H=1, K=6, V=5)
    S0 = rng.standard_normal((1, 1, 5, 6))
    o0, S_plain = oracle.recurrence(q, k, v, alpha, beta, S0=S0)
    o1, S_one = oracle.recurrence_truncated(q, k, v, alpha, beta, S0=S0, seg_len=20, r=1)
    assert np.allclose(S_one, S_plain, atol=1e-12) and np.allclose(o1, o0, atol=1e-12)
    _, ST = oracle.recurrence_truncated(q, k, v, alpha, beta, seg_len=10, r=1)
    assert np.linalg.matrix_rank(ST[0, 0], tol=1e-9) > 1
