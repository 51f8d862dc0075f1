"""Channel-gated rules (KDA, GDN2, and the scalar gate through the same
kernels) on the GPU, through the C ABI, against the float64 oracle."""
import numpy as np
import pytest

import oracle
from gpu_util import TOL, rel_err, to_dev, to_np
from gated_delta_rule_49_gb300 import binding, inputs

pytestmark = pytest.mark.gpu

VARIANTS = [(128, 128), (64, 128), (32, 32)]


@pytest.fixture(autouse=True)
def _clear_device_status():
    binding.gdn_get_last_device_status()


def _f32(x):
    import torch
    return None if x is None else torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).cuda()


def _run_prefill(p, want_o=True, want_state=True, S0=None):
    d = p.dtype
    return binding.prefill_gated(to_dev(p.q, d), to_dev(p.k, d), to_dev(p.v, d), _f32(p.alpha),
                                 beta=_f32(p.beta), b=_f32(p.b), w=_f32(p.w),
                                 S0=_f32(p.S0) if S0 is None else S0, gate=p.gate,
                                 want_o=want_o, want_state=want_state)


def _oracle(p):
    return oracle.recurrence_gated(p.q, p.k, p.v, p.alpha, beta=p.beta, b=p.b, w=p.w, S0=p.S0,
                                   gate=p.gate)


@pytest.mark.parametrize("gate", ["kda", "gdn2"])
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("K,V", VARIANTS)
@pytest.mark.parametrize("T", [1, 15, 16, 17, 100])
def test_prefill_gated_matches_oracle(gate, dtype, K, V, T):
    p = inputs.make_channel_gated(seed=T, B=2, T=T, H=3, K=K, V=V, dtype=dtype, gate=gate,
                                  with_S0=(T % 2 == 1))
    o, ST = _run_prefill(p)
    o_ref, S_ref = _oracle(p)
    assert rel_err(to_np(o), o_ref) <= TOL[dtype]
    assert rel_err(to_np(ST), S_ref) <= TOL[dtype]


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_scalar_gate_matches_oracle_and_chunked_prefill(dtype):
    """The scalar gate through the token-by-token kernel equals the oracle's
    Gated DeltaNet and the chunked prefill (two independent GPU paths)."""
    import torch
    p = inputs.make_tiny(seed=3, B=2, H=2, T=130, K=128, V=128, dtype=dtype)
    q, k, v = to_dev(p.q, dtype), to_dev(p.k, dtype), to_dev(p.v, dtype)
    al, be = _f32(p.alpha), _f32(p.beta)
    og, Sg = binding.prefill_gated(q, k, v, al, beta=be, gate="gdn")
    oc, Sc = binding.prefill(q, k, v, al, be)
    o_ref, S_ref = oracle.recurrence(p.q, p.k, p.v, p.alpha, p.beta)
    assert rel_err(to_np(og), o_ref) <= TOL[dtype] and rel_err(to_np(Sg), S_ref) <= TOL[dtype]
    assert rel_err(to_np(og), to_np(oc)) <= 2 * TOL[dtype]
    assert torch.isfinite(Sg).all()


def test_decay_only_and_full_erase_on_gpu():
    """Nothing written (b = w = 0): S_T = S0 diag(prod alpha).  b = 1 and unit
    keys: after one step S k = w (.) v."""
    import torch
    p = inputs.make_channel_gated(seed=5, B=1, T=40, H=2, K=64, V=128, dtype="fp32",
                                  gate="gdn2", with_S0=True)
    p.b[:] = 0.0
    p.w[:] = 0.0
    _, ST = _run_prefill(p, want_o=False)
    ref = p.S0.astype(np.float64) * np.prod(p.alpha.astype(np.float64), axis=1)[:, :, None, :]
    assert rel_err(to_np(ST), ref) <= 1e-5
    p1 = inputs.make_channel_gated(seed=6, B=2, T=1, H=2, K=64, V=128, dtype="fp32",
                                   gate="gdn2", with_S0=True)
    p1.b[:] = 1.0
    _, ST1 = _run_prefill(p1, want_o=False)
    got = np.einsum("bhvk,bhk->bhv", to_np(ST1), p1.k[:, 0])
    assert rel_err(got, p1.w[:, 0] * p1.v[:, 0]) <= 1e-5


def test_prefill_gated_null_outputs_zero_length_and_in_place():
    import torch
    p = inputs.make_channel_gated(seed=7, B=1, T=33, H=2, K=128, V=128, gate="kda",
                                  with_S0=True)
    o_ref, S_ref = _oracle(p)
    o, ST = _run_prefill(p, want_state=False)
    assert ST is None and rel_err(to_np(o), o_ref) <= TOL["bf16"]
    o, ST = _run_prefill(p, want_o=False)
    assert o is None and rel_err(to_np(ST), S_ref) <= TOL["bf16"]
    # in place: S_T aliases S0
    S = _f32(p.S0)
    B, T, H, K = p.k.shape
    o = torch.empty((B, T, H, 128), dtype=torch.bfloat16, device="cuda")
    binding.gdn_prefill_gated(to_dev(p.q, "bf16"), to_dev(p.k, "bf16"), to_dev(p.v, "bf16"),
                              _f32(p.alpha), _f32(p.beta), None, None, S, o, S, B, T, H, K, 128,
                              binding.GDN_GATE_KDA, binding.GDN_BF16)
    assert rel_err(to_np(S), S_ref) <= TOL["bf16"]
    # T = 0 copies S0
    S2 = torch.empty_like(S)
    binding.gdn_prefill_gated(None, None, None, None, _f32(p.beta), None, None, _f32(p.S0), None,
                              S2, B, 0, H, K, 128, binding.GDN_GATE_KDA, binding.GDN_BF16)
    assert np.array_equal(to_np(S2), p.S0)


@pytest.mark.parametrize("gate", ["gdn", "kda", "gdn2"])
@pytest.mark.parametrize("K,V", VARIANTS)
def test_decode_gated_matches_oracle_and_prefill(gate, K, V):
    import torch
    steps = 9
    if gate == "gdn":
        p = inputs.make_tiny(seed=K, B=3, H=2, T=steps, K=K, V=V, dtype="bf16")
        S0 = (0.2 * np.random.default_rng(1).standard_normal((3, 2, V, K))).astype(np.float32)
        o_ref, S_ref = oracle.recurrence(p.q, p.k, p.v, p.alpha, p.beta, S0=S0)
        alpha, beta, bg, wg = p.alpha, p.beta, None, None
    else:
        p = inputs.make_channel_gated(seed=K + 1, B=3, T=steps, H=2, K=K, V=V, gate=gate,
                                      with_S0=True)
        S0 = p.S0
        o_ref, S_ref = _oracle(p)
        alpha, beta, bg, wg = p.alpha, p.beta, p.b, p.w
    B, H = 3, 2
    S = _f32(S0)
    outs = []
    for t in range(steps):
        o = torch.empty((B, H, V), dtype=torch.bfloat16, device="cuda")
        sl = lambda x: None if x is None else _f32(x[:, t])  # noqa: E731
        binding.gdn_decode_step_gated(to_dev(np.ascontiguousarray(p.q[:, t]), "bf16"),
                                      to_dev(np.ascontiguousarray(p.k[:, t]), "bf16"),
                                      to_dev(np.ascontiguousarray(p.v[:, t]), "bf16"),
                                      sl(alpha), sl(beta), sl(bg), sl(wg), S, o, B, H, K, V,
                                      binding.GATES[gate], binding.GDN_BF16)
        outs.append(to_np(o))
    o_gpu = np.stack(outs, axis=1)
    assert rel_err(o_gpu, o_ref) <= TOL["bf16"] and rel_err(to_np(S), S_ref) <= TOL["bf16"]


@pytest.mark.slow
@pytest.mark.parametrize("gate", ["kda", "gdn2"])
def test_gated_full_size_sampled(gate):
    """The prefill workload's shapes (B=8, T=4096, H=16, d_k=d_v=128, bf16)
    under each gate: sampled sequences, including the heads with the
    fastest- and slowest-decaying channel centres, against the oracle."""
    p = inputs.make_channel_gated(gate=gate)
    o, ST = _run_prefill(p)
    o, ST = to_np(o), to_np(ST)
    la = np.log(p.alpha[0, :256].astype(np.float64)).mean(axis=(0, 2))  # per head
    for b, h in [(0, int(la.argmin())), (7, int(la.argmax())), (3, 5)]:
        sub = inputs.take_gated_sequences(p, [b], [h])
        o_ref, S_ref = _oracle(sub)
        assert rel_err(o[b:b + 1, :, h:h + 1], o_ref) <= TOL["bf16"]
        assert rel_err(ST[b:b + 1, h:h + 1], S_ref) <= TOL["bf16"]
