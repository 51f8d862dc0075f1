"""The chunkwise form used by the GPU prefill equals the token-by-token oracle."""
import numpy as np
import pytest

import oracle
from chunk_ref import chunk_recurrence


@pytest.mark.parametrize("T,C", [(1, 64), (63, 64), (64, 64), (65, 64), (100, 16), (130, 64)])
def test_chunk_form_equals_recurrence(T, C):
    rng = np.random.default_rng(T * 7 + C)
    B, H, K, V = 1, 2, 8, 6
    q = rng.standard_normal((B, T, H, K)); q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k = rng.standard_normal((B, T, H, K)); k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, T, H, V))
    alpha = rng.uniform(0.2, 1.0, size=(B, T, H))
    beta = rng.uniform(0.0, 1.9, size=(B, T, H))
    S0 = rng.standard_normal((B, H, V, K))
    o, ST = oracle.recurrence(q, k, v, alpha, beta, S0=S0)
    oc, STc = chunk_recurrence(q, k, v, alpha, beta, S0=S0, C=C)
    np.testing.assert_allclose(oc, o, atol=1e-11, rtol=0)
    np.testing.assert_allclose(STc, ST, atol=1e-11, rtol=0)
