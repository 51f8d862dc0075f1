"""Pins of the DRRQR channel-selection oracle ("On State Reduction in Linear
Attention" notes, Sec. 2.8) that do not lean on its own formulas."""
import itertools

import numpy as np
import pytest

import oracle


def _volume(M, cols):
    """sqrt(det(M_I^T M_I)): the k-volume spanned by the chosen columns."""
    Mi = M[:, list(cols)]
    return np.sqrt(max(np.linalg.det(Mi.T @ Mi), 0.0))


def _structured(rng, rows, n, rank=None):
    X = rng.standard_normal((rows, n)) * rng.lognormal(0.0, 0.7, size=n)
    if rank is not None:
        X = X[:, :rank] @ rng.standard_normal((rank, n))
    return X


def test_gram_is_the_sum_over_tokens():
    rng = np.random.default_rng(0)
    k = rng.standard_normal((2, 5, 3, 4))
    q = rng.standard_normal((2, 5, 3, 4))
    G = oracle.channel_gram(k, q)
    for h in range(3):
        want = np.zeros((4, 4))
        for b in range(2):
            for t in range(5):
                want += np.outer(k[b, t, h], k[b, t, h]) + np.outer(q[b, t, h], q[b, t, h])
        assert np.allclose(G[h], want, atol=1e-12)


def test_gram_hand_computed_case():
    """Two tokens, one head, K = 2, integer entries, worked by hand:
    k rows (1, 2), (3, -1); q rows (0, 1), (1, 1) give
    [[1+9+0+1, 2-3+0+1], [2-3+0+1, 4+1+1+1]] = [[11, 0], [0, 7]]."""
    k = np.array([[[1.0, 2.0]], [[3.0, -1.0]]])
    q = np.array([[[0.0, 1.0]], [[1.0, 1.0]]])
    assert np.array_equal(oracle.channel_gram(k, q)[0], np.array([[11.0, 0.0], [0.0, 7.0]]))


def test_gram_spectrum_is_the_squared_singular_values_of_the_stacked_rows():
    """G_h = M_h^T M_h for M_h the keys and queries of head h stacked as rows:
    its eigenvalues are the squared singular values of M_h (an SVD, not a sum
    of outer products), its trace is the summed squared row norms (2N for
    unit rows), and it is symmetric positive semi-definite."""
    rng = np.random.default_rng(5)
    N, H, K = 37, 3, 6
    k = rng.standard_normal((N, H, K))
    q = rng.standard_normal((N, H, K))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    G = oracle.channel_gram(k, q)
    for h in range(H):
        M = np.concatenate([k[:, h], q[:, h]], axis=0)
        sv = np.linalg.svd(M, compute_uv=False)
        ev = np.linalg.eigvalsh(G[h])
        assert np.allclose(np.sort(ev), np.sort(sv ** 2), atol=1e-10)
        assert abs(np.trace(G[h]) - 2 * N) < 1e-10
        assert np.allclose(G[h], G[h].T, atol=1e-14)
        assert ev.min() > -1e-10


def test_gram_is_additive_over_token_batches_and_rotates_with_the_channels():
    """Statistics collected over two batches add up; rotating every key and
    query by an orthogonal R conjugates the Gram: G(kR, qR) = R^T G R."""
    rng = np.random.default_rng(6)
    k = rng.standard_normal((3, 11, 2, 5))
    q = rng.standard_normal((3, 11, 2, 5))
    whole = oracle.channel_gram(k, q)
    parts = oracle.channel_gram(k[:, :4], q[:, :4]) + oracle.channel_gram(k[:, 4:], q[:, 4:])
    assert np.allclose(whole, parts, atol=1e-12)
    R, _ = np.linalg.qr(rng.standard_normal((5, 5)))
    rot = oracle.channel_gram(k @ R, q @ R)
    for h in range(2):
        assert np.allclose(rot[h], R.T @ whole[h] @ R, atol=1e-11)
    # a key channel that is zero everywhere gives a zero row and column
    k[..., 3] = 0.0
    q[..., 3] = 0.0
    Z = oracle.channel_gram(k, q)
    assert not Z[:, 3, :].any() and not Z[:, :, 3].any()


@pytest.mark.parametrize("seed", range(4))
def test_rho_is_the_volume_ratio_of_each_swap(seed):
    """Strong RRQR's test quantity: swapping kept column i with candidate j
    multiplies the volume of the kept columns by exactly rho_ij (brute force
    through determinants of Gram submatrices, no triangular factor)."""
    import scipy.linalg
    rng = np.random.default_rng(seed)
    n, k = 7, 3
    M = _structured(rng, 20, n)
    perm = rng.permutation(n)
    R = scipy.linalg.qr(M[:, perm], mode="r")[0][:n, :n]
    _, _, _, rho = oracle.rrqr_factors(R, k)
    base = _volume(M, perm[:k])
    for i in range(k):
        for j in range(n - k):
            cols = list(perm[:k])
            cols[i] = perm[k + j]
            assert np.isclose(_volume(M, cols) / base, rho[i, j], rtol=1e-9)


@pytest.mark.parametrize("seed", range(4))
@pytest.mark.parametrize("f", [1.0, 1.5, 2.0])
def test_result_is_a_local_volume_maximum_within_f(seed, f):
    """At the end no single swap can raise the kept volume by more than f
    (brute force), and the pages' bounds with c_f = sqrt(1 + f^2 k (n-k))
    hold."""
    import scipy.linalg
    rng = np.random.default_rng(10 + seed)
    n, k = 8, 3
    M = _structured(rng, 30, n)
    perm, rho_max, _ = oracle.drrqr(M, k, f=f)
    assert rho_max <= f
    base = _volume(M, perm[:k])
    for i in range(k):
        for j in range(k, n):
            cols = list(perm[:k])
            cols[i] = perm[j]
            assert _volume(M, cols) <= f * base * (1 + 1e-9)
    R = scipy.linalg.qr(M[:, perm], mode="r")[0][:n, :n]
    A, _, C, _ = oracle.rrqr_factors(R, k)
    sM = np.linalg.svd(M, compute_uv=False)
    sA = np.linalg.svd(A, compute_uv=False)
    cf = np.sqrt(1 + f * f * k * (n - k))
    assert np.all(sA >= sM[:k] / cf * (1 - 1e-9))
    assert np.linalg.norm(C, 2) <= cf * sM[k] * (1 + 1e-9)
    assert sA[0] / sA[-1] <= cf * sM[0] / sM[k - 1] * (1 + 1e-9)


def test_volume_against_the_exhaustive_maximum():
    """From the pages' bound sigma_i(A_k) >= sigma_i(M) / c_f: the kept volume
    is at least prod_{i<k} sigma_i(M) / c_f^k, and no k columns exceed
    prod_{i<k} sigma_i(M); checked against all C(n, k) subsets."""
    rng = np.random.default_rng(3)
    n, k, f = 6, 3, 1.0
    cf = np.sqrt(1 + f * f * k * (n - k))
    for _ in range(5):
        M = _structured(rng, 12, n)
        perm, _, _ = oracle.drrqr(M, k, f=f)
        top = np.prod(np.linalg.svd(M, compute_uv=False)[:k])
        best = max(_volume(M, c) for c in itertools.combinations(range(n), k))
        got = _volume(M, perm[:k])
        assert best <= top * (1 + 1e-9)
        assert got >= top / cf ** k


def test_unique_answers():
    """Orthogonal columns with distinct norms: the k longest.  Exactly k
    nonzero columns: those k."""
    rng = np.random.default_rng(5)
    Q, _ = np.linalg.qr(rng.standard_normal((40, 10)))
    norms = rng.permutation(np.arange(1, 11)).astype(float)
    perm, rho, swaps = oracle.drrqr(Q * norms, 4)
    assert set(perm[:4]) == set(np.argsort(-norms)[:4]) and swaps == 0
    M = np.zeros((30, 9))
    keep = [1, 4, 6, 8]
    M[:, keep] = rng.standard_normal((30, 4))
    M[:, [0, 2]] = 1e-3 * rng.standard_normal((30, 2))  # small but nonzero
    perm, _, _ = oracle.drrqr(M, 4)
    assert set(perm[:4]) == set(keep)


def test_swaps_fix_a_bad_greedy_start():
    """A case where the greedy pivoted-QR choice is not a local volume
    maximum within f = 1.01: the swap loop runs and ends at one."""
    rng = np.random.default_rng(7)
    found = False
    for _ in range(200):
        M = _structured(rng, 12, 8, rank=None)
        perm, rho, swaps = oracle.drrqr(M, 3, f=1.01)
        if swaps > 0:
            found = True
            assert rho <= 1.01
            break
    assert found
