"""Pins of the KDA / GDN2 oracle ("Linear Attention Architectures" notes,
Secs. 2.5-2.6) against what the pages and the mathematics fix.

Every check takes an implementation ``run(gate, q, k, v, alpha, beta, b, w,
S0) -> (o, S_T)``.  The oracle must pass them all; three plausible mistakes,
planted in a float64 numpy re-statement here on the CPU (decay applied to the
value rows instead of the key channels, the write taken along the erase
direction e instead of the key, the erase read taken before the decay), must
each fail at least one of them.
"""
import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.filterwarnings("ignore")


def run_oracle(gate, q, k, v, alpha, beta, b, w, S0):
    return oracle.recurrence_gated(q, k, v, alpha, beta=beta, b=b, w=w, S0=S0, gate=gate,
                                   threads=1)


def make_mutant(decay_rows=False, write_along_e=False, read_before_decay=False):
    def run(gate, q, k, v, alpha, beta, b, w, S0):
        B, T, H, K = k.shape
        V = v.shape[-1]
        o = np.zeros((B, T, H, V))
        ST = np.zeros((B, H, V, K))
        for bb in range(B):
            for h in range(H):
                S = np.zeros((V, K)) if S0 is None else np.array(S0[bb, h], dtype=np.float64)
                for t in range(T):
                    kt, qt, vt, at = k[bb, t, h], q[bb, t, h], v[bb, t, h], alpha[bb, t, h]
                    if gate == "kda":
                        e, z = beta[bb, t, h] * kt, beta[bb, t, h] * vt
                    else:
                        e, z = b[bb, t, h] * kt, w[bb, t, h] * vt
                    read_old = S @ e
                    if decay_rows:
                        S = at[:V, None] * S if V <= K else S * at[None, :]
                    else:
                        S = S * at[None, :]
                    u = z - (read_old if read_before_decay else S @ e)
                    S = S + np.outer(u, e if write_along_e else kt)
                    o[bb, t, h] = S @ qt
                ST[bb, h] = S
        return o, ST
    return run


def _unit(x):
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def _problem(seed, B=1, T=9, H=2, K=6, V=5):
    rng = np.random.default_rng(seed)
    q = _unit(rng.standard_normal((B, T, H, K)))
    k = _unit(rng.standard_normal((B, T, H, K)))
    v = rng.standard_normal((B, T, H, V))
    alpha = rng.uniform(0.4, 1.0, size=(B, T, H, K))
    beta = rng.uniform(0.05, 1.2, size=(B, T, H))
    b = rng.uniform(0.0, 1.5, size=(B, T, H, K))
    w = rng.uniform(0.0, 1.5, size=(B, T, H, V))
    S0 = rng.standard_normal((B, H, V, K))
    return q, k, v, alpha, beta, b, w, S0


# ---- the checks -------------------------------------------------------------

def check_kda_scalar_decay_is_gdn(run):
    """Sec. 2.5: alpha_t = a_t 1 gives Gated DeltaNet (pinned on its own)."""
    q, k, v, alpha, beta, b, w, S0 = _problem(1)
    a = alpha[..., 0]
    o1, S1 = run("kda", q, k, v, np.repeat(a[..., None], k.shape[-1], -1), beta, None, None,
                 S0)
    o0, S0r = oracle.recurrence(q, k, v, a, beta, S0=S0, threads=1)
    return np.allclose(o1, o0, atol=1e-12) and np.allclose(S1, S0r, atol=1e-12)


def check_gdn2_equal_gates_is_kda(run):
    """Sec. 2.6: b = beta 1 and w = beta 1 give KDA back."""
    q, k, v, alpha, beta, b, w, S0 = _problem(2)
    K, V = k.shape[-1], v.shape[-1]
    o2, S2 = run("gdn2", q, k, v, alpha, None, np.repeat(beta[..., None], K, -1),
                 np.repeat(beta[..., None], V, -1), S0)
    o1, S1 = run_oracle("kda", q, k, v, alpha, beta, None, None, S0)
    return np.allclose(o2, o1, atol=1e-12) and np.allclose(S2, S1, atol=1e-12)


def check_decay_only_closed_form(run):
    """Nothing erased or written: S_t = S0 diag(prod_{s<=t} alpha_s), the
    decay acting on the key channels (columns), o_t = S_t q_t."""
    q, k, v, alpha, beta, b, w, S0 = _problem(3)
    ok = True
    for gate in ("kda", "gdn2"):
        o, ST = run(gate, q, k, v, alpha, np.zeros_like(beta), np.zeros_like(b),
                    np.zeros_like(w), S0)
        cum = np.cumprod(alpha, axis=1)  # [B, T, H, K]
        for t in range(k.shape[1]):
            St = S0 * cum[:, t][:, :, None, :]
            ok &= np.allclose(o[:, t], np.einsum("bhvk,bhk->bhv", St, q[:, t]), atol=1e-12)
        ok &= np.allclose(ST, S0 * cum[:, -1][:, :, None, :], atol=1e-12)
    return bool(ok)


def check_one_hot_keys_closed_form(run):
    """k_t = e_j: column j becomes alpha_j (1 - b_j) S[:, j] + w (.) v and every
    other column c is only decayed, alpha_c S[:, c]."""
    rng = np.random.default_rng(4)
    B, T, H, K, V = 1, 10, 1, 6, 5
    q, _, v, alpha, beta, b, w, S0 = _problem(4, B, T, H, K, V)
    js = rng.integers(0, K, size=T)
    k = np.zeros((B, T, H, K))
    k[0, np.arange(T), 0, js] = 1.0
    o, ST = run("gdn2", q, k, v, alpha, None, b, w, S0)
    S = S0[0, 0].copy()
    ok = True
    for t in range(T):
        j, a = js[t], alpha[0, t, 0]
        S = S * a[None, :]
        S[:, j] = (1.0 - b[0, t, 0, j]) * S[:, j] + w[0, t, 0] * v[0, t, 0]
        ok &= np.allclose(o[0, t, 0], S @ q[0, t, 0], atol=1e-12)
    return bool(ok and np.allclose(ST[0, 0], S, atol=1e-12))


def check_full_erase_writes_exactly(run):
    """b = 1 and a unit key: after the step S_t k_t = w (.) v_t, whatever the
    decayed state held along k_t."""
    q, k, v, alpha, beta, b, w, S0 = _problem(5, T=1)
    _, ST = run("gdn2", q, k, v, alpha, None, np.ones_like(b), w, S0)
    got = np.einsum("bhvk,bhk->bhv", ST, k[:, 0])
    return np.allclose(got, w[:, 0] * v[:, 0], atol=1e-12)


def check_channel_permutation(run):
    """Relabelling the key channels (k, q, alpha, b and the columns of S0 by
    the same permutation) leaves o unchanged and permutes the columns of S_T."""
    q, k, v, alpha, beta, b, w, S0 = _problem(6)
    perm = np.random.default_rng(7).permutation(k.shape[-1])
    ok = True
    for gate in ("kda", "gdn2"):
        o, ST = run(gate, q, k, v, alpha, beta, b, w, S0)
        op, STp = run(gate, q[..., perm], k[..., perm], v, alpha[..., perm], beta,
                      b[..., perm], w, S0[..., perm])
        ok &= np.allclose(op, o, atol=1e-12) and np.allclose(STp, ST[..., perm], atol=1e-12)
    return bool(ok)


def check_row_independence(run):
    """Value rows are independent systems: changing v and w of row 2 changes
    only row 2 of S_T and channel 2 of o."""
    q, k, v, alpha, beta, b, w, S0 = _problem(8)
    o, ST = run("gdn2", q, k, v, alpha, None, b, w, S0)
    v2, w2 = v.copy(), w.copy()
    v2[..., 2] += 1.0
    w2[..., 2] *= 0.5
    o2, ST2 = run("gdn2", q, k, v2, alpha, None, b, w2, S0)
    keep = [i for i in range(v.shape[-1]) if i != 2]
    return bool(np.array_equal(o[..., keep], o2[..., keep])
                and np.array_equal(ST[..., keep, :], ST2[..., keep, :])
                and not np.allclose(ST[..., 2, :], ST2[..., 2, :]))


CHECKS = [check_kda_scalar_decay_is_gdn, check_gdn2_equal_gates_is_kda,
          check_decay_only_closed_form, check_one_hot_keys_closed_form,
          check_full_erase_writes_exactly, check_channel_permutation,
          check_row_independence]


@pytest.mark.parametrize("check", CHECKS, ids=lambda c: c.__name__)
def test_oracle_passes(check):
    assert check(run_oracle)


def test_numpy_restatement_agrees_with_the_oracle():
    """The mutant harness without a mutation is the same rule (so that a
    failing mutant fails because of its mutation)."""
    q, k, v, alpha, beta, b, w, S0 = _problem(9)
    for gate in ("kda", "gdn2"):
        o1, S1 = make_mutant()(gate, q, k, v, alpha, beta, b, w, S0)
        o0, S0r = run_oracle(gate, q, k, v, alpha, beta, b, w, S0)
        assert np.allclose(o1, o0, atol=1e-12) and np.allclose(S1, S0r, atol=1e-12)


@pytest.mark.parametrize("mutation", ["decay_rows", "write_along_e", "read_before_decay"])
def test_planted_mistakes_are_caught(mutation):
    run = make_mutant(**{mutation: True})
    failed = [c.__name__ for c in CHECKS if not c(run)]
    assert failed, f"no pin catches {mutation}"
