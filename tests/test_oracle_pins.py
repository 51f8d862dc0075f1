"""Pins of the float64 oracle against what the pages and the mathematics fix.

Each test would fail for a plausible mistake in the oracle: a dropped decay,
an error formed against the undecayed state, a transposed outer product, a
read before the write, a wrong cumulative-decay index, a mixed-up row/column
convention, or a stable rank with the wrong normalisation.
"""
import numpy as np
import pytest

import oracle
from load import load

pytestmark = pytest.mark.filterwarnings("ignore")


def _rand_problem(rng, B=1, T=8, H=1, K=6, V=5, S0=True):
    q = rng.standard_normal((B, T, H, K))
    k = rng.standard_normal((B, T, H, K))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    v = rng.standard_normal((B, T, H, V))
    alpha = rng.uniform(0.3, 1.0, size=(B, T, H))
    beta = rng.uniform(0.05, 1.5, size=(B, T, H))
    S = rng.standard_normal((B, H, V, K)) if S0 else None
    return q, k, v, alpha, beta, S


# P2 -- worked example, "Linear Attention Architectures" notes, Sec. 2.3.
def test_scalar_worked_example():
    g = load("scalar_worked_example.txt")
    one = np.ones((1, 1, 1, 1))
    o, ST = oracle.recurrence(one * g["k"], one * g["k"], one * g["v"],
                              np.full((1, 1, 1), g["alpha"]), np.full((1, 1, 1), g["beta"]),
                              S0=one * g["S_prev"])
    assert ST[0, 0, 0, 0] == pytest.approx(g["S_new"], abs=1e-15)
    assert o[0, 0, 0, 0] == pytest.approx(g["S_new"], abs=1e-15)  # q = k: read = prediction


# P2, general form: for a unit key, S_t k = (1 - beta) alpha S_{t-1} k + beta v.
def test_unit_key_interpolation():
    rng = np.random.default_rng(1)
    q, k, v, alpha, beta, S0 = _rand_problem(rng, T=1, K=7, V=4)
    _, ST = oracle.recurrence(q, k, v, alpha, beta, S0=S0)
    kk = k[0, 0, 0]
    lhs = ST[0, 0] @ kk
    rhs = (1 - beta[0, 0, 0]) * alpha[0, 0, 0] * (S0[0, 0] @ kk) + beta[0, 0, 0] * v[0, 0, 0]
    np.testing.assert_allclose(lhs, rhs, atol=1e-14, rtol=0)


# P1 -- beta = 1 with a unit key: after the write the key retrieves v exactly,
# whatever the decay and the old state ("On State Reduction" notes, Eq. (2)).
def test_beta_one_unit_key_writes_exactly():
    rng = np.random.default_rng(2)
    q, k, v, alpha, beta, S0 = _rand_problem(rng, T=6, K=9, V=5)
    beta[..., -1] = 1.0
    _, ST = oracle.recurrence(q, k, v, alpha, beta, S0=S0)
    np.testing.assert_allclose(ST[0, 0] @ k[0, -1, 0], v[0, -1, 0], atol=1e-14, rtol=0)


# P3 -- linear attention, "On State Reduction" notes, Sec. 2.1 Eq. (1):
# S_T = sum_t v_t k_t^T with S_0 = 0 and o_t = S_t q_t.
def test_linear_attention_sum_of_outer_products():
    rng = np.random.default_rng(3)
    q, k, v, _, beta, _ = _rand_problem(rng, T=11, K=6, V=4, S0=False)
    alpha = np.ones_like(beta)
    o, ST = oracle.recurrence(q, k, v, alpha, beta, mode="linear")
    want = np.einsum("tv,tk->vk", v[0, :, 0], k[0, :, 0])
    np.testing.assert_allclose(ST[0, 0], want, atol=1e-13, rtol=0)
    # read after write: o_t uses the state including token t
    t = 4
    St = np.einsum("tv,tk->vk", v[0, : t + 1, 0], k[0, : t + 1, 0])
    np.testing.assert_allclose(o[0, t, 0], St @ q[0, t, 0], atol=1e-13, rtol=0)


# P3 -- with orthonormal keys (T <= K), S_0 = 0, beta = 1, alpha = 1, the
# delta rule's prediction S_{t-1} k_t is zero, so it equals linear attention.
def test_delta_rule_orthonormal_keys_is_linear_attention():
    rng = np.random.default_rng(4)
    K, V, T = 8, 5, 8
    Qm, _ = np.linalg.qr(rng.standard_normal((K, K)))
    k = Qm.T[:T].reshape(1, T, 1, K)
    q = rng.standard_normal((1, T, 1, K))
    v = rng.standard_normal((1, T, 1, V))
    ones = np.ones((1, T, 1))
    o, ST = oracle.recurrence(q, k, v, ones, ones)
    np.testing.assert_allclose(ST[0, 0], np.einsum("tv,tk->vk", v[0, :, 0], k[0, :, 0]),
                               atol=1e-13, rtol=0)


# P4 -- decay only: beta = 0 leaves S_T = (prod alpha) S_0 and
# o_t = (prod_{s<=t} alpha_s) S_0 q_t.
def test_decay_only():
    rng = np.random.default_rng(5)
    q, k, v, alpha, beta, S0 = _rand_problem(rng, T=9, K=5, V=3)
    beta[:] = 0.0
    o, ST = oracle.recurrence(q, k, v, alpha, beta, S0=S0)
    cum = np.cumprod(alpha[0, :, 0])
    np.testing.assert_allclose(ST[0, 0], cum[-1] * S0[0, 0], atol=1e-14, rtol=0)
    want = cum[:, None] * np.einsum("vk,tk->tv", S0[0, 0], q[0, :, 0])
    np.testing.assert_allclose(o[0, :, 0], want, atol=1e-14, rtol=0)


# The spec product form S_t = alpha S_{t-1}(I - beta k k^T) + beta v k^T,
# o_t = S_t q_t, written with explicit matrices, equals the oracle's
# error-correction form (decay first, then error) on random inputs.
def test_matches_explicit_product_form():
    rng = np.random.default_rng(6)
    B, T, H, K, V = 2, 13, 3, 6, 4
    q, k, v, alpha, beta, S0 = _rand_problem(rng, B=B, T=T, H=H, K=K, V=V)
    o, ST = oracle.recurrence(q, k, v, alpha, beta, S0=S0)
    I = np.eye(K)
    for b in range(B):
        for h in range(H):
            S = S0[b, h].copy()
            for t in range(T):
                kt = k[b, t, h][:, None]
                S = alpha[b, t, h] * S @ (I - beta[b, t, h] * kt @ kt.T) \
                    + beta[b, t, h] * v[b, t, h][:, None] @ kt.T
                np.testing.assert_allclose(o[b, t, h], S @ q[b, t, h], atol=1e-12, rtol=0)
            np.testing.assert_allclose(ST[b, h], S, atol=1e-12, rtol=0)


# The order matters: an error formed against the undecayed state is a
# different update ("Linear Attention Architectures" notes, Sec. 2.4).
def test_decay_before_error_is_distinguishable():
    rng = np.random.default_rng(7)
    q, k, v, alpha, beta, S0 = _rand_problem(rng, T=1, K=4, V=3)
    _, ST = oracle.recurrence(q, k, v, alpha, beta, S0=S0)
    kk, a, b = k[0, 0, 0], alpha[0, 0, 0], beta[0, 0, 0]
    wrong = a * S0[0, 0] + b * np.outer(v[0, 0, 0] - S0[0, 0] @ kk, kk)
    assert np.abs(ST[0, 0] - wrong).max() > 1e-3


# P5 -- rank bound, "On State Reduction" notes, Eq. (3):
# rank S_t <= min(rank K_t, rank V_t) <= t, brute force on tiny inputs.
@pytest.mark.parametrize("rk,rv", [(2, 5), (5, 2), (3, 3), (8, 8)])
def test_rank_bound(rk, rv):
    rng = np.random.default_rng(10 + rk * 10 + rv)
    K = V = 8
    T = 12
    Bk = np.linalg.qr(rng.standard_normal((K, rk)))[0]
    Bv = np.linalg.qr(rng.standard_normal((V, rv)))[0]
    k = (rng.standard_normal((T, rk)) @ Bk.T)
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, rv)) @ Bv.T
    q = rng.standard_normal((T, K))
    alpha = rng.uniform(0.5, 1.0, size=T)
    beta = rng.uniform(0.1, 1.0, size=T)
    for t in range(1, T + 1):
        _, ST = oracle.recurrence(q[None, :t, None], k[None, :t, None], v[None, :t, None],
                                  alpha[None, :t, None], beta[None, :t, None])
        rs = np.linalg.matrix_rank(ST[0, 0], tol=1e-10)
        bound = min(np.linalg.matrix_rank(k[:t], tol=1e-10),
                    np.linalg.matrix_rank(v[:t], tol=1e-10))
        assert rs <= bound <= t


# P6 -- 1 <= er <= rank <= min(V, K); er = 1 at rank one; er = d (u = 1)
# when all singular values are equal ("On State Reduction" notes, Sec. 2.2.1).
def test_stable_rank_bounds():
    rng = np.random.default_rng(11)
    mats = [rng.standard_normal((7, 5)), rng.standard_normal((4, 9))]
    mats.append(rng.standard_normal((6, 2)) @ rng.standard_normal((2, 6)))
    for M in mats:
        _, s1, er = oracle.stable_rank(M)
        r = np.linalg.matrix_rank(M)
        assert 1.0 - 1e-12 <= er <= r + 1e-12 <= min(M.shape) + 1e-12
    rank1 = np.outer(rng.standard_normal(6), rng.standard_normal(4))
    assert oracle.stable_rank(rank1)[2] == pytest.approx(1.0, abs=1e-12)
    _, s1, er = oracle.stable_rank(3.0 * np.eye(5))
    assert er == pytest.approx(5.0, abs=1e-12) and s1 == pytest.approx(3.0, abs=1e-12)
    rect = np.zeros((6, 4))
    rect[:4, :4] = 2.0 * np.eye(4)
    assert oracle.stable_rank(rect)[2] / min(rect.shape) == pytest.approx(1.0, abs=1e-12)
    # the Frobenius term is the sum of squared singular values
    M = mats[0]
    f2, _, _ = oracle.stable_rank(M)
    assert f2 == pytest.approx(np.sum(np.linalg.svd(M, compute_uv=False) ** 2), rel=1e-12)


# P7 -- worked example, "On State Reduction" notes, Sec. 2.4:
# S = diag(1, 0.01) has er = 1.0001 and u = 0.50005.
def test_stable_rank_worked_example():
    g = load("diag_stable_rank.txt")
    S = np.array(g["S"])
    f2, s1, er = oracle.stable_rank(S)
    assert er == pytest.approx(g["er"], abs=1e-12)
    assert er / min(S.shape) == pytest.approx(g["u"], abs=1e-12)
    sv = np.linalg.svd(S, compute_uv=False)
    assert sv[0] / sv[-1] == pytest.approx(g["kappa"], rel=1e-12)
    # embedded zero-padded in a 32 x 32 matrix, as the GPU test uses it
    Z = np.zeros((32, 32))
    Z[:2, :2] = S
    assert oracle.stable_rank(Z)[2] == pytest.approx(g["er"], abs=1e-12)


def test_stable_rank_zero_state():
    f2, s1, er = oracle.stable_rank(np.zeros((2, 4, 4)))
    assert np.all(f2 == 0) and np.all(s1 == 0) and np.all(er == 0)


# P8 -- orthogonal invariance, "On State Reduction" notes, Sec. 3.1, Prop. 3.1:
# k' = T k, q' = T q, S' = S T^T leave the outputs unchanged (also with decay).
def test_orthogonal_invariance():
    rng = np.random.default_rng(12)
    B, T, H, K, V = 1, 17, 2, 8, 5
    q, k, v, alpha, beta, S0 = _rand_problem(rng, B=B, T=T, H=H, K=K, V=V)
    Tm = np.linalg.qr(rng.standard_normal((K, K)))[0]
    o, ST = oracle.recurrence(q, k, v, alpha, beta, S0=S0)
    o2, ST2 = oracle.recurrence(q @ Tm.T, k @ Tm.T, v, alpha, beta, S0=S0 @ Tm.T)
    np.testing.assert_allclose(o2, o, atol=1e-12, rtol=0)
    np.testing.assert_allclose(ST2, ST @ Tm.T, atol=1e-12, rtol=0)


# P9 -- coordinate selection ("On State Reduction" notes, Sec. 2.6): running
# on the kept channels equals running on all channels with the dropped q/k
# channels (and S_0 columns) zeroed; dropped state columns stay exactly zero.
def test_pruning_equals_zeroing():
    rng = np.random.default_rng(13)
    B, T, H, K, V, Kp = 1, 15, 2, 10, 4, 5
    q, k, v, alpha, beta, S0 = _rand_problem(rng, B=B, T=T, H=H, K=K, V=V)
    idx = np.stack([np.sort(rng.permutation(K)[:Kp]) for _ in range(H)])
    hh = np.arange(H)[:, None]
    qp, kp = q[:, :, hh, idx], k[:, :, hh, idx]
    S0p = np.take_along_axis(S0, idx[None, :, None, :], axis=-1)
    mask = np.zeros((H, K))
    mask[hh, idx] = 1.0
    o, ST = oracle.recurrence(q * mask[None, None], k * mask[None, None], v, alpha, beta,
                              S0=S0 * mask[None, :, None, :])
    op, STp = oracle.recurrence(qp, kp, v, alpha, beta, S0=S0p)
    np.testing.assert_allclose(op, o, atol=1e-13, rtol=0)
    np.testing.assert_allclose(STp, np.take_along_axis(ST, idx[None, :, None, :], axis=-1),
                               atol=1e-13, rtol=0)
    assert np.all(ST * (1 - mask[None, :, None, :]) == 0.0)


# P10 -- value channels are independent systems ("On State Reduction" notes,
# Sec. 2.5): perturbing v[..., i] changes only row i of S and o[..., i].
def test_row_independence():
    rng = np.random.default_rng(14)
    q, k, v, alpha, beta, S0 = _rand_problem(rng, T=10, K=6, V=5)
    o, ST = oracle.recurrence(q, k, v, alpha, beta, S0=S0)
    v2 = v.copy()
    v2[..., 2] += rng.standard_normal(v.shape[:-1])
    o2, ST2 = oracle.recurrence(q, k, v2, alpha, beta, S0=S0)
    others = [0, 1, 3, 4]
    np.testing.assert_array_equal(o2[..., others], o[..., others])
    np.testing.assert_array_equal(ST2[:, :, others], ST[:, :, others])
    assert np.abs(ST2[:, :, 2] - ST[:, :, 2]).max() > 1e-6


def test_batch_heads_are_independent_sequences():
    rng = np.random.default_rng(15)
    q, k, v, alpha, beta, S0 = _rand_problem(rng, B=2, T=7, H=3, K=4, V=3)
    o, ST = oracle.recurrence(q, k, v, alpha, beta, S0=S0, threads=4)
    o1, ST1 = oracle.recurrence(q[1:2, :, 2:3], k[1:2, :, 2:3], v[1:2, :, 2:3],
                                alpha[1:2, :, 2:3], beta[1:2, :, 2:3], S0=S0[1:2, 2:3],
                                threads=1)
    np.testing.assert_array_equal(o1[0, :, 0], o[1, :, 2])
    np.testing.assert_array_equal(ST1[0, 0], ST[1, 2])


def test_continuation_equals_one_pass():
    """Resuming from S_T of a prefix equals one pass over the whole sequence."""
    rng = np.random.default_rng(16)
    q, k, v, alpha, beta, S0 = _rand_problem(rng, T=12, K=5, V=4)
    o, ST = oracle.recurrence(q, k, v, alpha, beta, S0=S0)
    oa, Sa = oracle.recurrence(q[:, :5], k[:, :5], v[:, :5], alpha[:, :5], beta[:, :5], S0=S0)
    ob, Sb = oracle.recurrence(q[:, 5:], k[:, 5:], v[:, 5:], alpha[:, 5:], beta[:, 5:], S0=Sa)
    np.testing.assert_allclose(np.concatenate([oa, ob], axis=1), o, atol=1e-13, rtol=0)
    np.testing.assert_allclose(Sb, ST, atol=1e-13, rtol=0)


# Channel selection with renormalisation ("On State Reduction" notes, Sec. 2.6,
# Alg. 1): checked against the selection matrix P_I = [e_i1 .. e_id']^T of the
# notes (a matrix product, not an index gather), unit norm, and direction.
def test_gather_normalize_matches_selection_matrix():
    rng = np.random.default_rng(21)
    H, K, Kp = 3, 16, 6
    x = rng.standard_normal((5, 4, H, K)) * rng.uniform(0.1, 10.0, size=(5, 4, H, 1))
    idx = np.stack([rng.permutation(K)[:Kp] for _ in range(H)])  # unsorted on purpose
    y = oracle.gather_normalize(x, idx)
    for h in range(H):
        P = np.zeros((Kp, K))
        P[np.arange(Kp), idx[h]] = 1.0
        z = x[..., h, :] @ P.T
        z = z / np.linalg.norm(z, axis=-1, keepdims=True)
        np.testing.assert_allclose(y[..., h, :], z, atol=1e-15, rtol=0)
    np.testing.assert_allclose(np.linalg.norm(y, axis=-1), 1.0, atol=1e-14)


def test_gather_normalize_keeps_direction_and_handles_zero():
    rng = np.random.default_rng(22)
    x = rng.standard_normal((7, 2, 8))
    idx = np.array([[0, 3, 5, 7], [1, 2, 4, 6]])
    y = oracle.gather_normalize(x, idx)
    g = np.take_along_axis(x, np.broadcast_to(idx, (7, 2, 4)), axis=-1)
    cos = (y * g).sum(-1) / np.linalg.norm(g, axis=-1)
    np.testing.assert_allclose(cos, 1.0, atol=1e-14)
    # normalisation is scale invariant: a full-width L2 norm first changes nothing
    xn = x / np.linalg.norm(x, axis=-1, keepdims=True)
    np.testing.assert_allclose(oracle.gather_normalize(xn, idx), y, atol=1e-14)
    z = np.zeros((1, 2, 8))
    assert np.all(oracle.gather_normalize(z, idx) == 0.0)
