"""The two-pass form of the tensor-core prefill (a key-side pass over every
chunk of every sequence, then the state recurrence loading its operands) is
the one-pass form's arithmetic split across two kernels.  Every product that
feeds the state is the same instruction on the same operands, so the final
states must be bit-identical; the output product is computed transposed
there, which may round an output differently in its last bf16 bit (another
accumulation order inside one product), so outputs must agree to one bf16
ulp.  Checked with and without a start state, with a ragged last chunk, and
with outputs or the final state alone; repeated calls must be bit-identical.
In the segment-parallel mode the two-pass form takes another route than the
one-pass form's second pass (the outputs as o0 + S_start x, the end state
from the combine), so there the forms agree to a tolerance.  Both forms are
also held to the oracle."""
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
    xbuf = 0 if need == 0 else -(-B * T * H * 128 * 2 // 256) * 256  # segments' X buffer
    assert two - (need + 255) // 256 * 256 == B * H * chunks * 16384 + xbuf
    outs = []
    # segmented: also the two-pass form without the X buffer (its second
    # pass reruns the segments like the one-pass form: bit-identical states)
    for ws_bytes in ((need, two - xbuf, two) if xbuf else (need, two)):
        o = torch.full((B, T, H, V), float("nan"), dtype=torch.bfloat16, device="cuda")
        ST = torch.full((B, H, V, K), float("nan"), device="cuda")
        ws = torch.full((max(ws_bytes, 1),), 0xFF, dtype=torch.uint8, device="cuda")
        binding.gdn_prefill(d["q"], d["k"], d["v"], d["alpha"], d["beta"], s0, o, ST, B, T, H, K,
                            V, binding.GDN_BF16, ws if ws_bytes else None, ws_bytes)
        torch.cuda.synchronize()
        assert binding.gdn_get_last_device_status() == binding.GDN_OK
        outs.append((o.float().cpu().numpy(), ST.cpu().numpy()))
    if xbuf:
        assert_same(outs[0], outs[1])
    return outs[0], outs[-1]


def assert_same(one, two):
    (o1, s1), (o2, s2) = one, two
    # the states take the same operands through the same products
    assert np.array_equal(s1.view(np.int32), s2.view(np.int32))
    assert not np.isnan(o2).any()
    # o: the two forms sum q_t . k_s in different orders (a tensor-memory
    # product in one, warp-level MMAs in the other) before P is rounded to
    # bf16, so an entry of P may land one bf16 step (2^-8 relative) apart,
    # and the transposed product accumulates in another order; both stay
    # far inside one part in 10^3 of o (the parity bar is 10^-2)
    assert rel_err(o2, o1) <= 1e-3, rel_err(o2, o1)
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.maximum(np.abs(o1), np.abs(o2)), 1e-30))) - 7)
    assert np.mean(np.abs(o1 - o2) > ulp) <= 1e-2


@pytest.mark.parametrize("K", [128, 64])
@pytest.mark.parametrize("B,T,H", [(2, 300, 3), (1, 64, 1), (3, 1, 2), (4, 577, 8)])
def test_two_pass_bit_identical_whole_sequences(K, B, T, H):
    p = inputs.make_prefill(B=B, T=T, H=H, K=K, seed=T + K, with_S0=True)
    one, two = run_both(p)
    assert_same(one, two)
    o_ref, S_ref = oracle.recurrence(p.q, p.k, p.v, p.alpha, p.beta, S0=p.S0)
    for o_, S_ in (one, two):
        assert rel_err(o_, o_ref) <= TOL["bf16"] and rel_err(S_, S_ref) <= TOL["bf16"]


@pytest.mark.parametrize("K", [128, 64])
@pytest.mark.parametrize("T,S0", [(4133, True), (2048, False)])
def test_two_pass_bit_identical_segmented(K, T, S0):
    from test_gpu_segments import long_problem
    p = long_problem(K, T, with_S0=S0)
    B, T_, H, K_, V = p.shape
    assert binding.gdn_prefill_workspace_size(B, T, H, K, V, binding.GDN_BF16) > 0
    one, two = run_both(p, S0=S0)
    # o: the one-pass form rounds each output to bf16 once; the two-pass form
    # rounds o0 and then o0 + S_start x (and x itself), so they may land two
    # bf16 steps apart at the largest outputs (2 * 2^-8 of the scale).  S_T:
    # the combine's affine chain instead of the rerun's bf16-operand products
    assert not np.isnan(two[0]).any() and not np.isnan(two[1]).any()
    assert rel_err(two[0], one[0]) <= 8e-3, rel_err(two[0], one[0])
    assert rel_err(two[1], one[1]) <= 5e-3, rel_err(two[1], one[1])
    o_ref, S_ref = oracle.recurrence(p.q, p.k, p.v, p.alpha, p.beta, S0=p.S0)
    for o_, S_ in (one, two):
        assert rel_err(o_, o_ref) <= TOL["bf16"] and rel_err(S_, S_ref) <= TOL["bf16"]


def test_two_pass_sizes():
    # no two-pass form for float32 or the (32, 32) variant
    assert binding.gdn_prefill_two_pass_workspace_size(2, 300, 3, 128, 128, binding.GDN_FP32) == 0
    assert binding.gdn_prefill_two_pass_workspace_size(2, 300, 3, 32, 32, binding.GDN_BF16) == 0
    assert binding.gdn_prefill_two_pass_workspace_size(8, 4096, 16, 128, 128,
                                                       binding.GDN_BF16) == 8 * 16 * 64 * 16384


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
        cur = (o.view(torch.int16).clone(), ST.view(torch.int32).clone())  # deterministic
        if first is None:
            first = cur
        else:
            assert torch.equal(cur[0], first[0]) and torch.equal(cur[1], first[1])


def test_one_pass_repeated_calls_stay_identical():
    # the one-pass form (no workspace): the key group runs up to two chunks
    # ahead of the state group in every CTA; repeated calls over many CTAs
    # give identical bytes
    import torch
    B, T, H, K, V = 8, 1024, 16, 128, 128
    p = inputs.make_prefill(B=B, T=T, H=H, K=K, seed=6)
    d = problem_to_dev(p)
    o = torch.empty((B, T, H, V), dtype=torch.bfloat16, device="cuda")
    ST = torch.empty((B, H, V, K), device="cuda")
    first = None
    for _ in range(10):
        binding.gdn_prefill(d["q"], d["k"], d["v"], d["alpha"], d["beta"], None, o, ST, B, T, H,
                            K, V, binding.GDN_BF16, None, 0)
        assert binding.gdn_get_last_device_status() == binding.GDN_OK
        cur = (o.view(torch.int16).clone(), ST.view(torch.int32).clone())
        if first is None:
            first = cur
        else:
            assert torch.equal(cur[0], first[0]) and torch.equal(cur[1], first[1])


@pytest.mark.parametrize("want_o,want_S", [(True, False), (False, True)])
def test_two_pass_outputs_or_state_alone(want_o, want_S):
    import torch
    B, T, H, K, V = 2, 333, 4, 128, 128
    p = inputs.make_prefill(B=B, T=T, H=H, K=K, seed=9)
    d = problem_to_dev(p)
    need = binding.gdn_prefill_two_pass_workspace_size(B, T, H, K, V, binding.GDN_BF16)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    o = torch.full((B, T, H, V), float("nan"), dtype=torch.bfloat16, device="cuda") if want_o else None
    ST = torch.full((B, H, V, K), float("nan"), device="cuda") if want_S else None
    binding.gdn_prefill(d["q"], d["k"], d["v"], d["alpha"], d["beta"], None, o, ST, B, T, H, K, V,
                        binding.GDN_BF16, ws, need)
    assert binding.gdn_get_last_device_status() == binding.GDN_OK
    o_ref, S_ref = oracle.recurrence(p.q, p.k, p.v, p.alpha, p.beta)
    if want_o:
        assert rel_err(to_np(o), o_ref) <= TOL["bf16"]
    if want_S:
        assert rel_err(to_np(ST), S_ref) <= TOL["bf16"]


@pytest.mark.parametrize("B,T,H", [(2, 300, 3), (1, 4133, 2)])
def test_two_pass_in_place_continuation(B, T, H):
    # S_T may alias S0: each CTA reads its start state before writing the end
    # state (whole sequences), or the start states are read by the first
    # segment pass and the end state written by the last (segment-parallel)
    import torch
    K, V = 128, 128
    p = inputs.make_prefill(B=B, T=T, H=H, K=K, seed=11, with_S0=True)
    d = problem_to_dev(p)
    need = binding.gdn_prefill_workspace_size(B, T, H, K, V, binding.GDN_BF16)
    two = binding.gdn_prefill_two_pass_workspace_size(B, T, H, K, V, binding.GDN_BF16)
    res = []
    for wsb in (need, two):
        S = d["S0"].clone()
        o = torch.empty((B, T, H, V), dtype=torch.bfloat16, device="cuda")
        ws = torch.empty(max(wsb, 1), dtype=torch.uint8, device="cuda")
        binding.gdn_prefill(d["q"], d["k"], d["v"], d["alpha"], d["beta"], S, o, S, B, T, H, K,
                            V, binding.GDN_BF16, ws if wsb else None, wsb)
        assert binding.gdn_get_last_device_status() == binding.GDN_OK
        res.append(S.cpu().numpy())
    if need == 0:
        assert np.array_equal(res[0].view(np.int32), res[1].view(np.int32))
    else:  # segmented: the end state from the combine, not from a rerun
        assert rel_err(res[1], res[0]) <= 5e-3, rel_err(res[1], res[0])
    _, S_ref = oracle.recurrence(p.q, p.k, p.v, p.alpha, p.beta, S0=p.S0)
    assert rel_err(res[1], S_ref) <= TOL["bf16"]


@pytest.mark.parametrize("K", [128, 64])
def test_two_pass_segmented_state_alone(K):
    # without outputs the segmented two-pass form needs no second pass: the
    # combine chains the segments' maps on to the end state
    import torch
    B, T, H, V = 1, 4133, 2, 128
    p = inputs.make_prefill(B=B, T=T, H=H, K=K, seed=13, with_S0=True)
    d = problem_to_dev(p)
    need = binding.gdn_prefill_workspace_size(B, T, H, K, V, binding.GDN_BF16)
    two = binding.gdn_prefill_two_pass_workspace_size(B, T, H, K, V, binding.GDN_BF16)
    assert need > 0
    res = []
    for wsb in (need, two):
        ST = torch.full((B, H, V, K), float("nan"), device="cuda")
        ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
        binding.gdn_prefill(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["S0"], None, ST, B, T,
                            H, K, V, binding.GDN_BF16, ws, wsb)
        assert binding.gdn_get_last_device_status() == binding.GDN_OK
        res.append(to_np(ST))
    assert rel_err(res[1], res[0]) <= 5e-3, rel_err(res[1], res[0])
    _, S_ref = oracle.recurrence(p.q, p.k, p.v, p.alpha, p.beta, S0=p.S0)
    assert rel_err(res[1], S_ref) <= TOL["bf16"]
