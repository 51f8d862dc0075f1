"""GPU parity: every entry point against the float64 oracle on the same seeded
inputs, element by element, within the stated tolerances
(max |gpu - ref| / max |ref| <= 1e-2 for bf16 inputs with an fp32 state,
<= 1e-4 all-fp32), plus the pages' invariants re-checked on the GPU path."""
import numpy as np
import pytest

import oracle
from gpu_util import TOL, rel_err, run_decode, run_prefill, problem_to_dev, to_np
from gated_delta_rule_49_gb300 import binding, inputs

pytestmark = pytest.mark.gpu

VARIANTS = [(32, 32), (64, 128), (128, 128)]


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from gated_delta_rule_49_gb300 import build
    build.build()
    binding.load()


def small_problem(K, V, T, dtype, B=2, H=3, seed=0, with_S0=True, alpha_lo=0.6):
    rng = np.random.default_rng(seed + 1000 * K + T)
    rnd = (lambda x: inputs.round_to_bf16(x)) if dtype == "bf16" else (lambda x: x.astype(np.float32))
    q = rng.standard_normal((B, T, H, K)); q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k = rng.standard_normal((B, T, H, K)); k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, T, H, V))
    alpha = rng.uniform(alpha_lo, 1.0, size=(B, T, H)).astype(np.float32)
    beta = rng.uniform(0.0, 1.0, size=(B, T, H)).astype(np.float32)
    S0 = (0.3 * rng.standard_normal((B, H, V, K))).astype(np.float32) if with_S0 else None
    return inputs.Problem("small", dtype, rnd(q), rnd(k), rnd(v), alpha, beta, S0)


def oracle_of(p):
    return oracle.recurrence(p.q, p.k, p.v, p.alpha, p.beta, S0=p.S0)


def check(p, o, ST, tol=None):
    o_ref, S_ref = oracle_of(p)
    tol = TOL[p.dtype] if tol is None else tol
    eo, es = rel_err(o, o_ref), rel_err(ST, S_ref)
    assert eo <= tol and es <= tol, (eo, es)
    return eo, es


# ---------------------------------------------------------------- prefill
def test_tiny_workload_fp32():
    """256 tokens, one head, d = 32, all fp32: o, S_T and er within 1e-4."""
    p = inputs.make_tiny()
    o, ST = run_prefill(p)
    check(p, o, ST)
    _, _, er_ref = oracle.stable_rank(oracle_of(p)[1])
    import torch
    _, _, er = binding.state_rank(torch.from_numpy(ST).cuda())
    assert rel_err(to_np(er), er_ref) <= 1e-4


@pytest.mark.parametrize("K,V", VARIANTS)
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("T", [1, 63, 64, 65, 130, 320])
def test_prefill_small(K, V, dtype, T):
    p = small_problem(K, V, T, dtype)
    o, ST = run_prefill(p)
    check(p, o, ST)


@pytest.mark.parametrize("K,V", VARIANTS)
def test_prefill_zero_initial_state(K, V):
    p = small_problem(K, V, 200, "bf16", with_S0=False)
    o, ST = run_prefill(p)
    check(p, o, ST)


def test_prefill_poison_canary():
    """Outputs pre-filled with NaN: every element must be written."""
    import torch
    p = small_problem(128, 128, 77, "bf16")
    d = problem_to_dev(p)
    B, T, H, K, V = p.shape
    o = torch.full((B, T, H, V), float("nan"), dtype=torch.bfloat16, device="cuda")
    ST = torch.full((B, H, V, K), float("nan"), device="cuda")
    binding.gdn_prefill(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["S0"], o, ST, B, T, H,
                        K, V, binding.GDN_BF16)
    assert not torch.isnan(o.float()).any() and not torch.isnan(ST).any()
    check(p, to_np(o), to_np(ST))


def test_prefill_empty_and_in_place():
    import torch
    p = small_problem(64, 128, 90, "fp32")
    d = problem_to_dev(p)
    B, T, H, K, V = p.shape
    # T = 0: S_T = S0
    ST = torch.empty((B, H, V, K), device="cuda")
    binding.gdn_prefill(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["S0"], None, ST, B, 0,
                        H, K, V, binding.GDN_FP32)
    assert torch.equal(ST, d["S0"])
    binding.gdn_prefill(None, None, None, None, None, None, None, ST, B, 0, H, K, V,
                        binding.GDN_FP32)
    assert torch.count_nonzero(ST) == 0
    # S_T aliasing S0: in-place continuation
    S = d["S0"].clone()
    o = torch.empty((B, T, H, V), device="cuda")
    binding.gdn_prefill(d["q"], d["k"], d["v"], d["alpha"], d["beta"], S, o, S, B, T, H, K, V,
                        binding.GDN_FP32)
    check(p, to_np(o), to_np(S))
    assert binding.gdn_get_last_device_status() == binding.GDN_OK


@pytest.mark.parametrize("K,V", VARIANTS)
def test_prefill_continuation(K, V):
    """prefill(T1) then prefill(T2, S0 = S_T1) equals prefill(T1 + T2)."""
    import torch
    p = small_problem(K, V, 200, "bf16")
    d = problem_to_dev(p)
    o, ST = binding.prefill(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["S0"])
    a = slice(0, 77)
    b = slice(77, 200)
    sub = {n: d[n][:, a].contiguous() for n in ("q", "k", "v", "alpha", "beta")}
    o1, S1 = binding.prefill(sub["q"], sub["k"], sub["v"], sub["alpha"], sub["beta"], d["S0"])
    sub = {n: d[n][:, b].contiguous() for n in ("q", "k", "v", "alpha", "beta")}
    o2, S2 = binding.prefill(sub["q"], sub["k"], sub["v"], sub["alpha"], sub["beta"], S1)
    assert rel_err(to_np(torch.cat([o1, o2], 1)), to_np(o)) <= 1e-2
    assert rel_err(to_np(S2), to_np(ST)) <= 1e-2


def test_prefill_beta_one_unit_key_write():
    """beta = 1 with unit keys: after the last token S_T k_T = v_T (fp32 mode)."""
    p = small_problem(128, 128, 65, "fp32")
    p.beta[:, -1] = 1.0
    k = p.k.astype(np.float64)
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    p.k[:] = k.astype(np.float32)
    _, ST = run_prefill(p)
    kT = p.k[:, -1].astype(np.float64)                      # [B,H,K]
    got = np.einsum("bhvk,bhk->bhv", ST.astype(np.float64), kT)
    assert rel_err(got, p.v[:, -1]) <= 1e-4


def test_prefill_decay_only():
    """beta = 0: S_T = (prod alpha) S0 and o_t = (prod_{s<=t} alpha_s) S0 q_t."""
    p = small_problem(64, 128, 100, "fp32", alpha_lo=0.95)
    p.beta[:] = 0.0
    o, ST = run_prefill(p)
    cum = np.cumprod(p.alpha.astype(np.float64), axis=1)         # [B,T,H]
    S0 = p.S0.astype(np.float64)
    assert rel_err(ST, cum[:, -1, :, None, None] * S0) <= 1e-4
    want = cum[..., None] * np.einsum("bhvk,bthk->bthv", S0, p.q.astype(np.float64))
    assert rel_err(o, want) <= 1e-4


def test_prefill_orthogonal_invariance():
    """k' = T k, q' = T q, S0' = S0 T^T: same o, S_T' = S_T T^T (fp32 mode)."""
    p = small_problem(128, 128, 96, "fp32")
    Tm = np.linalg.qr(np.random.default_rng(5).standard_normal((128, 128)))[0]
    o, ST = run_prefill(p)
    p2 = inputs.Problem("rot", "fp32", (p.q @ Tm.T).astype(np.float32),
                        (p.k @ Tm.T).astype(np.float32), p.v, p.alpha, p.beta,
                        (p.S0 @ Tm.T).astype(np.float32))
    o2, ST2 = run_prefill(p2)
    assert rel_err(o2, o) <= 1e-4
    assert rel_err(ST2, ST @ Tm.T) <= 1e-4


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_pruned_equals_zeroed_channels(dtype):
    """The (64, 128) variant on gathered channels equals the (128, 128)
    variant with the dropped q/k channels and S0 columns zeroed."""
    p = small_problem(128, 128, 150, dtype)
    rng = np.random.default_rng(9)
    B, T, H, K, V = p.shape
    idx = np.stack([np.sort(rng.permutation(K)[:64]) for _ in range(H)])
    mask = np.zeros((H, K), np.float32)
    mask[np.arange(H)[:, None], idx] = 1.0
    hh = np.arange(H)[:, None]
    pz = inputs.Problem("z", dtype, p.q * mask[None, None], p.k * mask[None, None], p.v, p.alpha,
                        p.beta, p.S0 * mask[None, :, None, :])
    pp = inputs.Problem("p", dtype, np.ascontiguousarray(p.q[:, :, hh, idx]),
                        np.ascontiguousarray(p.k[:, :, hh, idx]), p.v, p.alpha, p.beta,
                        np.ascontiguousarray(np.take_along_axis(p.S0, idx[None, :, None, :], -1)))
    oz, Sz = run_prefill(pz)
    op, Sp = run_prefill(pp)
    tol = TOL[dtype]
    assert rel_err(op, oz) <= tol
    assert rel_err(Sp, np.take_along_axis(Sz, idx[None, :, None, :], -1)) <= tol
    assert rel_err(Sz * (1 - mask[None, :, None, :]), np.zeros_like(Sz)) <= tol


def test_row_independence_on_gpu():
    """Perturbing v[..., i] changes only row i of S_T and o[..., i]."""
    p = small_problem(128, 128, 70, "fp32")
    o, ST = run_prefill(p)
    v2 = p.v.copy()
    v2[..., 5] += 1.0
    p2 = inputs.Problem("r", "fp32", p.q, p.k, v2, p.alpha, p.beta, p.S0)
    o2, ST2 = run_prefill(p2)
    others = [i for i in range(128) if i != 5]
    np.testing.assert_array_equal(o2[..., others], o[..., others])
    np.testing.assert_array_equal(ST2[:, :, others], ST[:, :, others])


# ---------------------------------------------------------------- decode
@pytest.mark.parametrize("K,V", VARIANTS)
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_decode_small(K, V, dtype):
    p = small_problem(K, V, 40, dtype, B=3, H=5)
    o, S = run_decode(p)
    check(p, o, S)


@pytest.mark.parametrize("K", [128, 64])
def test_decode_equals_prefill(K):
    """decode x n equals prefill over the same n tokens."""
    p = small_problem(K, 128, 96, "bf16")
    od, Sd = run_decode(p)
    op, Sp = run_prefill(p)
    assert rel_err(od, op) <= 1e-2 and rel_err(Sd, Sp) <= 1e-2


# ---------------------------------------------------------------- stable rank
def test_state_rank_against_svd():
    import torch
    rng = np.random.default_rng(3)
    mats = [rng.standard_normal((128, 128)),
            rng.standard_normal((128, 4)) @ rng.standard_normal((4, 128)),
            inputs.low_stable_rank_state(rng, 1, 1, 128, 128)[0, 0],
            rng.standard_normal((128, 64)), rng.standard_normal((32, 32))]
    for M in mats:
        M = M.astype(np.float32)
        f2, s1, er = binding.state_rank(torch.from_numpy(M[None]).cuda(), max_iter=2000, tol=0.0)
        rf, rs, re = oracle.stable_rank(M.astype(np.float64))
        assert rel_err(to_np(f2), [rf]) <= 1e-4
        assert rel_err(to_np(s1), [rs]) <= 1e-4
        assert rel_err(to_np(er), [re]) <= 1e-4


def test_state_rank_worked_example_and_bounds():
    """diag(1, 0.01) zero-padded in 32 x 32 gives er = 1.0001; c I gives er = d;
    a rank-one state gives er = 1; the zero state gives 0 and the warning."""
    import torch
    from load import load
    g = load("diag_stable_rank.txt")
    Z = np.zeros((4, 32, 32), np.float32)
    Z[0, :2, :2] = np.array(g["S"], np.float32)
    Z[1] = 2.5 * np.eye(32)
    Z[2] = np.outer(np.arange(1, 33), np.linspace(-1, 1, 32))
    f2, s1, er = binding.state_rank(torch.from_numpy(Z).cuda(), max_iter=1000, tol=0.0)
    er = to_np(er)
    assert abs(er[0] - g["er"]) <= 1e-4 * g["er"]
    assert abs(er[0] / 2 - g["u"]) <= 1e-4 * g["u"]  # u = er / min(d_v, d_k) of the 2 x 2 state
    assert abs(er[1] - 32.0) <= 1e-4 * 32
    assert abs(er[2] - 1.0) <= 1e-4
    assert er[3] == 0 and to_np(s1)[3] == 0 and to_np(f2)[3] == 0
    assert binding.gdn_get_last_device_status() == binding.GDN_WARN_ZERO_STATE
    assert binding.gdn_get_last_device_status() == binding.GDN_OK  # read clears it


# ---------------------------------------------------------------- full-size workloads
def _sampled_check(p, o, ST, seqs):
    """Oracle on a few (b, h) sequences of a full-size run."""
    for b, h in seqs:
        sub = inputs.take_sequences(p, [b], [h])
        o_ref, S_ref = oracle_of(sub)
        eo = rel_err(o[b:b + 1, :, h:h + 1], o_ref)
        es = rel_err(ST[b:b + 1, h:h + 1], S_ref)
        assert eo <= TOL[p.dtype] and es <= TOL[p.dtype], ((b, h), eo, es)


@pytest.mark.slow
def test_full_prefill_workload_sampled():
    """B=8, T=4096, H=16, d = 128, bf16: sampled sequences vs the oracle,
    including the heads with the longest and shortest decay horizons."""
    p = inputs.make_prefill()
    o, ST = run_prefill(p)
    hor = -1.0 / np.log(p.alpha.astype(np.float64)).mean(axis=(0, 1))
    seqs = [(0, int(hor.argmax())), (7, int(hor.argmin())), (3, 5), (5, 11)]
    _sampled_check(p, o, ST, seqs)


@pytest.mark.slow
def test_full_pruned_workload_sampled():
    p = inputs.make_prefill(pruned_K=64)
    o, ST = run_prefill(p)
    _sampled_check(p, o, ST, [(0, 0), (4, 9), (7, 15)])


@pytest.mark.slow
def test_full_long_context_sampled():
    """B=1, T=65536, H=16, alpha in [0.9995, 0.9999], keys in a narrow cone:
    two heads against the oracle, and the per-head stable rank of S_T."""
    import torch
    p = inputs.make_long()
    o, ST = run_prefill(p)
    _sampled_check(p, o, ST, [(0, 0), (0, 13)])
    _, _, er = binding.state_rank(torch.from_numpy(ST).cuda(), max_iter=2000, tol=0.0)
    _, _, er_ref = oracle.stable_rank(ST.astype(np.float64))
    assert rel_err(to_np(er), er_ref) <= 1e-2


@pytest.mark.slow
@pytest.mark.parametrize("K", [128, 64])
@pytest.mark.parametrize("B", [64, 1])
def test_full_decode_workload_sampled(K, B):
    """1024 decode steps from a low-stable-rank state; sampled heads vs the
    oracle, and er of the final states."""
    import torch
    p = inputs.make_decode(B=B, pruned_K=None if K == 128 else 64)
    d = problem_to_dev(p)
    S = d["S0"].clone()
    steps = p.k.shape[1]
    q = d["q"].transpose(0, 1).contiguous()
    k = d["k"].transpose(0, 1).contiguous()
    v = d["v"].transpose(0, 1).contiguous()
    al = d["alpha"].transpose(0, 1).contiguous()
    be = d["beta"].transpose(0, 1).contiguous()
    outs = torch.empty_like(v)
    for t in range(steps):
        binding.decode_step(q[t], k[t], v[t], al[t], be[t], S, o=outs[t])
    o = to_np(outs.transpose(0, 1))
    ST = to_np(S)
    seqs = [(0, 0), (B - 1, 15), (B // 2, 7)]
    _sampled_check(p, o, ST, seqs)
    _, _, er = binding.state_rank(S, max_iter=2000, tol=0.0)
    _, _, er_ref = oracle.stable_rank(ST.astype(np.float64))
    assert rel_err(to_np(er), er_ref) <= 1e-2
