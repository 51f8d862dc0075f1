"""The two-pass form of the tensor-core prefill (a key-side pass over every
chunk of every sequence, then the state recurrence loading its operands) is
the same arithmetic as the one-pass form, split across two kernels: outputs
and final states must be bit-identical, in the one-CTA-per-sequence mode and
in the segment-parallel mode, with and without a start state, and with a
ragged last chunk.  Both forms are held to the oracle elsewhere (the parity
tests call the convenience wrapper, which takes the two-pass form, and the
C-ABI tests with the minimum workspace, which take the one-pass form)."""
import numpy as np
import pytest

import oracle
from gpu_util import TOL, problem_to_dev, rel_err, to_np
from gated_delta_rule_49_gb300 import binding, inputs

pytestmark = pytest.mark.gpu


def run_both(p, S0=True):
    import torch
    B, T, H, K, V = p.shape
    d = problem_to_dev(p)
    s0 = d["S0"] if S0 else None
    need = binding.gdn_prefill_workspace_size(B, T, H, K, V, binding.GDN_BF16)
    two = binding.gdn_prefill_two_pass_workspace_size(B, T, H, K, V, binding.GDN_BF16)
    assert two > need
    chunks = (T + 63) // 64
    assert two - (need + 255) // 256 * 256 == B * H * chunks * 24576
    outs = []
    for ws_bytes in (need, two):
        o = torch.full((B, T, H, V), float("nan"), dtype=torch.bfloat16, device="cuda")
        ST = torch.full((B, H, V, K), float("nan"), device="cuda")
        ws = torch.full((max(ws_bytes, 1),), 0xFF, dtype=torch.uint8, device="cuda")
        binding.gdn_prefill(d["q"], d["k"], d["v"], d["alpha"], d["beta"], s0, o, ST, B, T, H, K,
                            V, binding.GDN_BF16, ws if ws_bytes else None, ws_bytes)
        torch.cuda.synchronize()
        assert binding.gdn_get_last_device_status() == binding.GDN_OK
        outs.append((o.view(torch.int16).cpu().numpy(), ST.cpu().numpy()))
    return outs


@pytest.mark.parametrize("K", [128, 64])
@pytest.mark.parametrize("B,T,H", [(2, 300, 3), (1, 64, 1), (3, 1, 2), (4, 577, 8)])
def test_two_pass_bit_identical_whole_sequences(K, B, T, H):
    p = inputs.make_prefill(B=B, T=T, H=H, K=K, seed=T + K, with_S0=True)
    (o1, s1), (o2, s2) = run_both(p)
    assert np.array_equal(o1, o2)
    assert np.array_equal(s1.view(np.int32), s2.view(np.int32))
    o_ref, S_ref = oracle.recurrence(p.q, p.k, p.v, p.alpha, p.beta, S0=p.S0)
    import torch
    o_f = torch.from_numpy(o2).view(torch.bfloat16).float().numpy()
    assert rel_err(o_f, o_ref) <= TOL["bf16"] and rel_err(s2, S_ref) <= TOL["bf16"]


@pytest.mark.parametrize("K", [128, 64])
@pytest.mark.parametrize("T,S0", [(4133, True), (2048, False)])
def test_two_pass_bit_identical_segmented(K, T, S0):
    from test_gpu_segments import long_problem
    p = long_problem(K, T, with_S0=S0)
    B, T_, H, K_, V = p.shape
    assert binding.gdn_prefill_workspace_size(B, T, H, K, V, binding.GDN_BF16) > 0
    (o1, s1), (o2, s2) = run_both(p, S0=S0)
    assert np.array_equal(o1, o2)
    assert np.array_equal(s1.view(np.int32), s2.view(np.int32))


def test_two_pass_sizes():
    # no two-pass form for float32 or the (32, 32) variant
    assert binding.gdn_prefill_two_pass_workspace_size(2, 300, 3, 128, 128, binding.GDN_FP32) == 0
    assert binding.gdn_prefill_two_pass_workspace_size(2, 300, 3, 32, 32, binding.GDN_BF16) == 0
    assert binding.gdn_prefill_two_pass_workspace_size(8, 4096, 16, 128, 128,
                                                       binding.GDN_BF16) == 8 * 16 * 64 * 24576


def test_two_pass_repeated_calls_stay_identical():
    # the start of every sequence races the key group against the state
    # group's first loads; many CTAs and repeated calls exercise the handoff
    import torch
    B, T, H, K, V = 8, 1024, 16, 128, 128
    p = inputs.make_prefill(B=B, T=T, H=H, K=K, seed=5)
    d = problem_to_dev(p)
    need = binding.gdn_prefill_two_pass_workspace_size(B, T, H, K, V, binding.GDN_BF16)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    o = torch.empty((B, T, H, V), dtype=torch.bfloat16, device="cuda")
    ST = torch.empty((B, H, V, K), device="cuda")
    first = None
    for _ in range(30):
        binding.gdn_prefill(d["q"], d["k"], d["v"], d["alpha"], d["beta"], None, o, ST, B, T, H,
                            K, V, binding.GDN_BF16, ws, need)
        assert binding.gdn_get_last_device_status() == binding.GDN_OK
        cur = (o.view(torch.int16).clone(), ST.view(torch.int32).clone())
        if first is None:
            first = cur
        else:
            assert torch.equal(cur[0], first[0]) and torch.equal(cur[1], first[1])
