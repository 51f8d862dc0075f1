"""Rank-r state truncation and the segmented prefill that applies it, on the
GPU through the C ABI, against the float64 oracle and constructed spectra."""
import numpy as np
import pytest

import oracle
from gpu_util import TOL, rel_err, to_dev, to_np
from gated_delta_rule_49_gb300 import binding, inputs

pytestmark = pytest.mark.gpu

VARIANTS = [(128, 128), (64, 128), (32, 32)]  # (K, V)


@pytest.fixture(autouse=True)
def _clear_device_status():
    binding.gdn_get_last_device_status()


def _orthonormal(rng, n, m):
    Q, R = np.linalg.qr(rng.standard_normal((n, m)))
    return Q * np.sign(np.diag(R))[None, :]


def _constructed(rng, BH, V, K, decay=0.93):
    """States A diag(sigma) B^T with distinct, geometrically spaced sigma."""
    n = min(V, K)
    sig = 3.0 * decay ** np.arange(n)
    S, A, Bs = [], [], []
    for _ in range(BH):
        a, b = _orthonormal(rng, V, n), _orthonormal(rng, K, n)
        S.append((a * sig) @ b.T)
        A.append(a)
        Bs.append(b)
    return np.stack(S).astype(np.float32), np.stack(A), np.stack(Bs), sig


@pytest.mark.parametrize("K,V", VARIANTS)
@pytest.mark.parametrize("r", [1, 4, 12, 24])
def test_truncate_constructed_spectrum(K, V, r):
    import torch
    rng = np.random.default_rng(r * 7 + K)
    S, A, Bs, sig = _constructed(rng, 6, V, K)
    dS = torch.from_numpy(S).cuda()
    sigma = binding.state_truncate(dS, r, want_sigma=True)
    want = np.einsum("bvr,r,bkr->bvk", A[..., :r], sig[:r], Bs[..., :r])
    assert rel_err(to_np(dS), want) <= 1e-4
    assert rel_err(to_np(sigma), np.broadcast_to(sig, (6, len(sig)))) <= 1e-5
    assert binding.gdn_get_last_device_status() == binding.GDN_OK


@pytest.mark.parametrize("K,V", VARIANTS)
@pytest.mark.parametrize("r", [1, 4, 12, 24])
def test_truncate_without_sigma_clustered_tail(K, V, r):
    """r well-separated leading values over a tail of many nearly equal tiny
    ones (the near-degenerate cluster a low-rank state ends in): without
    sigma the result is the best rank-r approximation, and the sweeps
    converge."""
    import torch
    rng = np.random.default_rng(r * 11 + K)
    n = min(V, K)
    S, want = [], []
    for _ in range(6):
        a, b = _orthonormal(rng, V, n), _orthonormal(rng, K, n)
        sig = np.concatenate([3.0 * 0.8 ** np.arange(r),
                              1e-3 * (1.0 + 1e-4 * rng.standard_normal(n - r))])
        S.append((a * sig) @ b.T)
        want.append((a[:, :r] * sig[:r]) @ b[:, :r].T)
    dS = torch.from_numpy(np.stack(S).astype(np.float32)).cuda()
    binding.state_truncate(dS, r)
    assert rel_err(to_np(dS), np.stack(want)) <= 1e-4
    assert binding.gdn_get_last_device_status() == binding.GDN_OK


@pytest.mark.parametrize("K,V", VARIANTS)
def test_truncate_prefill_states_against_oracle(K, V):
    """Final states of a short run (decaying, gapless-looking spectra): where
    the gap at r is clear the truncation matches the oracle's; everywhere the
    result has rank <= r and the discarded energy is the optimum."""
    import torch
    p = inputs.make_tiny(seed=K, B=2, H=4, T=200, K=K, V=V, dtype="fp32")
    _, ST = oracle.recurrence(p.q, p.k, p.v, p.alpha, p.beta)
    ST = ST.astype(np.float32)
    sv = np.linalg.svd(ST.astype(np.float64), compute_uv=False)
    for r in (1, 4, 12):
        dS = torch.from_numpy(ST.copy()).cuda()
        binding.state_truncate(dS, r)
        got = to_np(dS)
        ref = oracle.truncate_state(ST, r)
        for b in range(2):
            for h in range(4):
                s = sv[b, h]
                disc = np.sum(s[r:] ** 2)
                err = np.sum((got[b, h] - ST[b, h].astype(np.float64)) ** 2)
                assert err <= disc + 1e-5 * np.sum(s ** 2)
                assert np.linalg.svd(got[b, h], compute_uv=False)[r] <= 1e-4 * s[0]
                if (s[r - 1] - s[r]) > 0.05 * s[0]:
                    assert rel_err(got[b, h], ref[b, h]) <= 1e-3


def test_truncate_zero_state_full_rank_and_stable_rank():
    import torch
    Z = torch.zeros((3, 128, 128), device="cuda")
    sig = binding.state_truncate(Z, 4, want_sigma=True)
    assert torch.count_nonzero(Z) == 0 and torch.count_nonzero(sig) == 0
    assert binding.gdn_get_last_device_status() == binding.GDN_OK
    rng = np.random.default_rng(2)
    S = rng.standard_normal((5, 128, 64)).astype(np.float32)
    dS = torch.from_numpy(S).cuda()
    sig = to_np(binding.state_truncate(dS, 64, want_sigma=True))  # r = min(V, K): no cut
    assert np.array_equal(to_np(dS), S)
    ref = np.linalg.svd(S.astype(np.float64), compute_uv=False)
    assert rel_err(sig, ref) <= 1e-5
    # stable rank from the singular values agrees with the power iteration
    _, _, er = binding.state_rank(dS, max_iter=2000, tol=0.0)
    er_svd = (sig ** 2).sum(-1) / sig[:, 0] ** 2
    assert np.allclose(to_np(er), er_svd, rtol=1e-4)


def _subspace_problem(seed, B, T, H, K, V, d, eta, dtype):
    """Values near a per-head d-dimensional subspace (noise eta per channel).
    The state's column space lies in the span of the values, so every carried
    state has d dominant singular values and a tail of order eta (sigma_{d+1}
    / sigma_d <= 0.25 at every boundary for eta = 0.05): rank-d truncation is
    well conditioned, bf16 rounding cannot swap the kept subspace, and it
    still changes the outputs by more than 5x the tolerance."""
    rng = np.random.default_rng(seed)
    Qv = np.stack([_orthonormal(rng, V, d) for _ in range(H)])  # [H, V, d]
    v = np.einsum("hvd,bthd->bthv", Qv, rng.standard_normal((B, T, H, d)))
    v = v + eta * rng.standard_normal((B, T, H, V))
    k = rng.standard_normal((B, T, H, K))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    q = rng.standard_normal((B, T, H, K))
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    alpha = rng.uniform(0.97, 1.0, size=(B, T, H)).astype(np.float32)
    beta = rng.uniform(0.2, 0.8, size=(B, T, H)).astype(np.float32)
    rd = inputs.round_to_bf16 if dtype == "bf16" else (lambda x: x.astype(np.float32))
    return rd(q), rd(k), rd(v), alpha, beta


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("K,V", VARIANTS)
@pytest.mark.parametrize("seg_len", [64, 100])
def test_prefill_truncated_matches_oracle(dtype, K, V, seg_len):
    import torch
    B, T, H, d = 2, 300, 2, 4
    q, k, v, alpha, beta = _subspace_problem(seg_len + K, B, T, H, K, V, d, 0.05, dtype)
    o, ST = binding.prefill_truncated(to_dev(q, dtype), to_dev(k, dtype), to_dev(v, dtype),
                                      torch.from_numpy(alpha).cuda(),
                                      torch.from_numpy(beta).cuda(), seg_len=seg_len, r=d)
    o_ref, S_ref = oracle.recurrence_truncated(q, k, v, alpha, beta, seg_len=seg_len, r=d)
    assert rel_err(to_np(o), o_ref) <= TOL[dtype]
    assert rel_err(to_np(ST), S_ref) <= TOL[dtype]
    o_plain, _ = oracle.recurrence(q, k, v, alpha, beta)
    assert rel_err(o_plain, o_ref) > 5 * TOL[dtype]  # the truncation did change the outputs
    assert binding.gdn_get_last_device_status() == binding.GDN_OK


@pytest.mark.parametrize("K", [128, 64])
def test_prefill_truncated_windows_equal_contiguous_copies(K):
    """The segmented driver reads windows of the [B, T, H, *] tensors in place
    (token stride T): the same result, bit for bit, as gdn_prefill on
    contiguous copies of each window followed by gdn_state_truncate."""
    import torch
    B, T, H, seg, r = 3, 200, 2, 64, 6
    p = inputs.make_prefill(seed=1, B=B, T=T, H=H, K=128, V=128,
                            pruned_K=None if K == 128 else 64)
    d = {n: to_dev(getattr(p, n), "bf16") for n in ("q", "k", "v")}
    al, be = torch.from_numpy(p.alpha).cuda(), torch.from_numpy(p.beta).cuda()
    o, ST = binding.prefill_truncated(d["q"], d["k"], d["v"], al, be, seg_len=seg, r=r)
    S = None
    outs = []
    for t0 in range(0, T, seg):
        sl = slice(t0, min(T, t0 + seg))
        ow, S = binding.prefill(d["q"][:, sl].contiguous(), d["k"][:, sl].contiguous(),
                                d["v"][:, sl].contiguous(), al[:, sl].contiguous(),
                                be[:, sl].contiguous(), S)
        outs.append(ow)
        if t0 + seg < T:
            binding.state_truncate(S, r)
    assert torch.equal(o, torch.cat(outs, dim=1))
    assert torch.equal(ST, S)
