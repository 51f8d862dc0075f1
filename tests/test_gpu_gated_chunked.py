"""The chunkwise tensor-core prefill of KDA and GDN2 (gdn_prefill_gated_chunked)
on the GPU, through the C ABI, against the float64 oracle and the
token-by-token GPU kernel."""
import numpy as np
import pytest

import oracle
from gpu_util import TOL, rel_err, to_dev, to_np
from gated_delta_rule_49_gb300 import binding, inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clear_device_status():
    binding.gdn_get_last_device_status()


def _f32(x):
    import torch
    return None if x is None else torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).cuda()


def _run(p, want_o=True, want_state=True, poison=True):
    import torch
    B, T, H, K = p.k.shape
    V = p.v.shape[-1]
    gate = binding.GATES[p.gate]
    need = binding.gdn_prefill_gated_chunked_workspace_size(B, T, H, K, V, gate, binding.GDN_BF16)
    assert need > 0
    # a poisoned workspace: every byte the state pass reads must have been written
    ws = torch.full((need,), 0xFF if poison else 0, dtype=torch.uint8, device="cuda")
    o = (torch.full((B, T, H, V), float("nan"), dtype=torch.bfloat16, device="cuda")
         if want_o else None)
    ST = torch.full((B, H, V, K), float("nan"), device="cuda") if want_state else None
    binding.gdn_prefill_gated_chunked(to_dev(p.q, "bf16"), to_dev(p.k, "bf16"),
                                      to_dev(p.v, "bf16"), _f32(p.alpha), _f32(p.beta),
                                      _f32(p.b), _f32(p.w), _f32(p.S0), o, ST, B, T, H, K, V,
                                      gate, binding.GDN_BF16, ws, need)
    import torch as _t
    _t.cuda.synchronize()
    assert binding.gdn_get_last_device_status() == binding.GDN_OK
    return (None if o is None else to_np(o)), (None if ST is None else to_np(ST))


def _oracle(p):
    return oracle.recurrence_gated(p.q, p.k, p.v, p.alpha, beta=p.beta, b=p.b, w=p.w, S0=p.S0,
                                   gate=p.gate)


@pytest.mark.parametrize("gate", ["kda", "gdn2"])
@pytest.mark.parametrize("B,T,H,S0", [(2, 300, 3, True), (1, 64, 1, False), (3, 1, 2, True),
                                      (2, 129, 4, False), (1, 577, 2, True)])
def test_gated_chunked_matches_oracle(gate, B, T, H, S0):
    """Whole chunks, a single token, and ragged tails, with and without S0,
    element by element against the float64 oracle at the bf16 bound."""
    p = inputs.make_channel_gated(seed=T + H, B=B, T=T, H=H, K=128, V=128, gate=gate,
                                  with_S0=S0)
    o, ST = _run(p)
    o_ref, S_ref = _oracle(p)
    assert not np.isnan(o).any() and not np.isnan(ST).any()
    assert rel_err(o, o_ref) <= TOL["bf16"], rel_err(o, o_ref)
    assert rel_err(ST, S_ref) <= TOL["bf16"], rel_err(ST, S_ref)


@pytest.mark.parametrize("gate", ["kda", "gdn2"])
def test_gated_chunked_agrees_with_token_kernel(gate):
    """Two independent GPU paths (chunkwise tensor-core, token-by-token CUDA
    core) on the same inputs agree to the bf16 operand rounding."""
    p = inputs.make_channel_gated(seed=11, B=2, T=1000, H=4, K=128, V=128, gate=gate,
                                  with_S0=True)
    o, ST = _run(p)
    ot, STt = binding.prefill_gated(to_dev(p.q, "bf16"), to_dev(p.k, "bf16"), to_dev(p.v, "bf16"),
                                    _f32(p.alpha), beta=_f32(p.beta), b=_f32(p.b), w=_f32(p.w),
                                    S0=_f32(p.S0), gate=gate)
    assert rel_err(o, to_np(ot)) <= TOL["bf16"] and rel_err(ST, to_np(STt)) <= TOL["bf16"]


@pytest.mark.parametrize("want_o,want_S", [(True, False), (False, True)])
def test_gated_chunked_outputs_or_state_alone(want_o, want_S):
    p = inputs.make_channel_gated(seed=4, B=2, T=200, H=3, K=128, V=128, gate="kda")
    o, ST = _run(p, want_o=want_o, want_state=want_S)
    o_ref, S_ref = _oracle(p)
    if want_o:
        assert rel_err(o, o_ref) <= TOL["bf16"]
    if want_S:
        assert rel_err(ST, S_ref) <= TOL["bf16"]


def test_gated_chunked_in_place_and_repeatable():
    """S_T may alias S0; repeated calls give identical bytes."""
    import torch
    p = inputs.make_channel_gated(seed=8, B=2, T=333, H=2, K=128, V=128, gate="gdn2",
                                  with_S0=True)
    B, T, H, K = p.k.shape
    gate = binding.GATES["gdn2"]
    need = binding.gdn_prefill_gated_chunked_workspace_size(B, T, H, K, 128, gate, binding.GDN_BF16)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    args = (to_dev(p.q, "bf16"), to_dev(p.k, "bf16"), to_dev(p.v, "bf16"), _f32(p.alpha), None,
            _f32(p.b), _f32(p.w))
    firsts = None
    for _ in range(3):
        S = _f32(p.S0)
        o = torch.empty((B, T, H, 128), dtype=torch.bfloat16, device="cuda")
        binding.gdn_prefill_gated_chunked(*args, S, o, S, B, T, H, K, 128, gate,
                                          binding.GDN_BF16, ws, need)
        cur = (o.view(torch.int16).clone(), S.view(torch.int32).clone())
        if firsts is None:
            firsts = cur
        else:
            assert torch.equal(cur[0], firsts[0]) and torch.equal(cur[1], firsts[1])
    _, S_ref = _oracle(p)
    assert rel_err(to_np(firsts[1].view(torch.float32)), S_ref) <= TOL["bf16"]


def test_gdn2_chunked_graph_capture_and_single_calls():
    """GDN2 forks its write-content kernel onto a second stream and joins it
    back: eager calls, a single call after an idle GPU, and a CUDA graph
    replay of the call give identical bytes."""
    import torch
    p = inputs.make_channel_gated(seed=9, B=2, T=333, H=3, K=128, V=128, gate="gdn2",
                                  with_S0=True)
    B, T, H, K = p.k.shape
    gate = binding.GATES["gdn2"]
    need = binding.gdn_prefill_gated_chunked_workspace_size(B, T, H, K, 128, gate, binding.GDN_BF16)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    q, k, v = to_dev(p.q, "bf16"), to_dev(p.k, "bf16"), to_dev(p.v, "bf16")
    al, bg, wg, S0 = _f32(p.alpha), _f32(p.b), _f32(p.w), _f32(p.S0)
    o = torch.empty((B, T, H, 128), dtype=torch.bfloat16, device="cuda")
    ST = torch.empty((B, H, 128, K), device="cuda")

    def call():
        binding.gdn_prefill_gated_chunked(q, k, v, al, None, bg, wg, S0, o, ST, B, T, H, K, 128,
                                          gate, binding.GDN_BF16, ws, need)

    call()
    torch.cuda.synchronize()
    ref = (o.view(torch.int16).clone(), ST.view(torch.int32).clone())
    o_ref, S_ref = _oracle(p)
    assert rel_err(to_np(o), o_ref) <= TOL["bf16"] and rel_err(to_np(ST), S_ref) <= TOL["bf16"]
    for _ in range(3):  # single calls, the GPU idle in between
        o.zero_()
        ST.zero_()
        torch.cuda.synchronize()
        call()
        torch.cuda.synchronize()
        assert torch.equal(o.view(torch.int16), ref[0]) and torch.equal(ST.view(torch.int32), ref[1])
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        call()  # warm-up on the capturing stream
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call()
    o.zero_()
    ST.zero_()
    torch.cuda.synchronize()
    graph.replay()
    torch.cuda.synchronize()
    assert binding.gdn_get_last_device_status() == binding.GDN_OK
    assert torch.equal(o.view(torch.int16), ref[0]) and torch.equal(ST.view(torch.int32), ref[1])


def test_gated_chunked_rejects():
    """Unsupported shapes and gates, a short workspace: errors, no launch."""
    import torch
    p = inputs.make_channel_gated(seed=2, B=1, T=70, H=1, K=128, V=128, gate="kda")
    q, k, v = to_dev(p.q, "bf16"), to_dev(p.k, "bf16"), to_dev(p.v, "bf16")
    al, be = _f32(p.alpha), _f32(p.beta)
    o = torch.empty((1, 70, 1, 128), dtype=torch.bfloat16, device="cuda")
    need = binding.gdn_prefill_gated_chunked_workspace_size(1, 70, 1, 128, 128,
                                                            binding.GDN_GATE_KDA, binding.GDN_BF16)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    with pytest.raises(binding.GDNError) as e:
        binding.gdn_prefill_gated_chunked(q, k, v, al, be, None, None, None, o, None, 1, 70, 1,
                                          128, 128, binding.GDN_GATE_KDA, binding.GDN_BF16, ws,
                                          need - 16)
    assert e.value.status == binding.GDN_ERR_WORKSPACE
    with pytest.raises(binding.GDNError) as e:
        binding.gdn_prefill_gated_chunked(q, k, v, al[..., 0].contiguous(), be, None, None, None,
                                          o, None, 1, 70, 1, 128, 128, binding.GDN_GATE_SCALAR,
                                          binding.GDN_BF16, ws, need)
    assert e.value.status == binding.GDN_ERR_UNSUPPORTED


@pytest.mark.slow
@pytest.mark.parametrize("gate", ["kda", "gdn2"])
def test_gated_chunked_full_size_sampled(gate):
    """The gated prefill workload (B=8, T=4096, H=16, d_k=d_v=128, bf16):
    sampled sequences, including the heads with the fastest- and
    slowest-decaying channel centres, against the oracle."""
    p = inputs.make_channel_gated(gate=gate)
    o, ST = _run(p, poison=False)
    la = np.log(p.alpha[0, :256].astype(np.float64)).mean(axis=(0, 2))  # per head
    for b, h in [(0, int(la.argmin())), (7, int(la.argmax())), (3, 5)]:
        sub = inputs.take_gated_sequences(p, [b], [h])
        o_ref, S_ref = _oracle(sub)
        assert rel_err(o[b:b + 1, :, h:h + 1], o_ref) <= TOL["bf16"]
        assert rel_err(ST[b:b + 1, h:h + 1], S_ref) <= TOL["bf16"]
