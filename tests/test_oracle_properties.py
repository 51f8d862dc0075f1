"""Property tests of the oracles over random shapes and values (hypothesis):
identities that hold for every input, so that a slip anywhere in the
recurrence shows up on some draw.

- The update S <- S D (I - e k^T) + z k^T is linear in (v, S0) for fixed q, k
  and gates (GDN, KDA, GDN2 alike): outputs and final states add up.
- Running T1 tokens then T2 from the state reached equals running T1 + T2.
- The pruning prologue ignores a positive scale of its input row.
"""
import numpy as np
import pytest

import oracle

hyp = pytest.importorskip("hypothesis")
from hypothesis import given, settings  # noqa: E402
from hypothesis import strategies as st  # noqa: E402

SET = settings(max_examples=30, deadline=None)


def _draw(seed, B, T, H, K, V):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, T, H, K))
    k = rng.standard_normal((B, T, H, K))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    alpha = rng.uniform(0.2, 1.0, size=(B, T, H))
    beta = rng.uniform(0.0, 1.9, size=(B, T, H))
    return rng, q, k, alpha, beta


shapes = st.tuples(st.integers(0, 2 ** 31 - 1), st.integers(1, 2), st.integers(1, 9),
                   st.integers(1, 2), st.integers(1, 6), st.integers(1, 5))


@SET
@given(shapes)
def test_gdn_is_linear_in_values_and_start_state(sh):
    seed, B, T, H, K, V = sh
    rng, q, k, alpha, beta = _draw(seed, B, T, H, K, V)
    v1, v2 = rng.standard_normal((2, B, T, H, V))
    S1, S2 = rng.standard_normal((2, B, H, V, K))
    o1, T1 = oracle.recurrence(q, k, v1, alpha, beta, S0=S1, threads=1)
    o2, T2 = oracle.recurrence(q, k, v2, alpha, beta, S0=S2, threads=1)
    o3, T3 = oracle.recurrence(q, k, v1 + 2.0 * v2, alpha, beta, S0=S1 + 2.0 * S2, threads=1)
    assert np.allclose(o3, o1 + 2.0 * o2, atol=1e-9) and np.allclose(T3, T1 + 2.0 * T2, atol=1e-9)


@SET
@given(shapes, st.sampled_from(["kda", "gdn2"]))
def test_gated_rules_are_linear_in_values_and_start_state(sh, gate):
    seed, B, T, H, K, V = sh
    rng, q, k, _, beta = _draw(seed, B, T, H, K, V)
    alpha = rng.uniform(0.2, 1.0, size=(B, T, H, K))
    b = rng.uniform(0.0, 1.5, size=(B, T, H, K))
    w = rng.uniform(0.0, 1.5, size=(B, T, H, V))
    v1, v2 = rng.standard_normal((2, B, T, H, V))
    S1, S2 = rng.standard_normal((2, B, H, V, K))
    kw = dict(beta=beta, gate=gate) if gate == "kda" else dict(b=b, w=w, gate=gate)
    o1, T1 = oracle.recurrence_gated(q, k, v1, alpha, S0=S1, threads=1, **kw)
    o2, T2 = oracle.recurrence_gated(q, k, v2, alpha, S0=S2, threads=1, **kw)
    o3, T3 = oracle.recurrence_gated(q, k, v1 - v2, alpha, S0=S1 - S2, threads=1, **kw)
    assert np.allclose(o3, o1 - o2, atol=1e-9) and np.allclose(T3, T1 - T2, atol=1e-9)


@SET
@given(shapes, st.integers(0, 9))
def test_continuation_for_any_split(sh, cut):
    seed, B, T, H, K, V = sh
    rng, q, k, alpha, beta = _draw(seed, B, T, H, K, V)
    v = rng.standard_normal((B, T, H, V))
    c = min(cut, T)
    o, ST = oracle.recurrence(q, k, v, alpha, beta, threads=1)
    oa, Sa = oracle.recurrence(q[:, :c], k[:, :c], v[:, :c], alpha[:, :c], beta[:, :c],
                               threads=1)
    ob, Sb = oracle.recurrence(q[:, c:], k[:, c:], v[:, c:], alpha[:, c:], beta[:, c:], S0=Sa,
                               threads=1)
    assert np.allclose(np.concatenate([oa, ob], axis=1), o, atol=1e-10)
    assert np.allclose(Sb, ST, atol=1e-10)


@SET
@given(st.integers(0, 2 ** 31 - 1), st.floats(1e-3, 1e3))
def test_prologue_ignores_positive_scale(seed, c):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((3, 2, 16))
    idx = np.stack([rng.permutation(16)[:8] for _ in range(2)])
    assert np.allclose(oracle.gather_normalize(c * x, idx), oracle.gather_normalize(x, idx),
                       atol=1e-12)


@SET
@given(shapes)
def test_decay_acts_before_the_error(sh):
    """One step from S0 with alpha < 1: the error uses alpha S0 k, so the write
    along k is beta (v - alpha S0 k), visible as S_1 k - alpha S0 k (unit k)."""
    seed, B, _, H, K, V = sh
    rng, q, k, alpha, beta = _draw(seed, B, 1, H, K, V)
    v = rng.standard_normal((B, 1, H, V))
    S0 = rng.standard_normal((B, H, V, K))
    _, S1 = oracle.recurrence(q, k, v, alpha, beta, S0=S0, threads=1)
    kk = k[:, 0]
    a = alpha[:, 0][..., None]
    pred = a * np.einsum("bhvk,bhk->bhv", S0, kk)
    want = pred + beta[:, 0][..., None] * (v[:, 0] - pred)
    assert np.allclose(np.einsum("bhvk,bhk->bhv", S1, kk), want, atol=1e-10)
