"""The pruned prefill from full-width q/k (gdn_prefill_gathered): the pruning
prologue runs inside the key-side pass of the two-pass prefill.  Its gathered
q', k' use the standalone prologue's arithmetic and the rest is the two-pass
prefill, so the results must be bit-identical to gdn_gather_normalize followed
by gdn_prefill with its two-pass workspace; both are held to the float64
oracle on the oracle's own prologue ("On State Reduction" notes, Sec. 2.6 and
Alg. 1)."""
import numpy as np
import pytest

import oracle
from gpu_util import TOL, rel_err, to_dev, to_np
from gated_delta_rule_49_gb300 import binding, inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clear_device_status():
    binding.gdn_get_last_device_status()


def _problem(B, T, H, seed, S0=True):
    rng = np.random.default_rng(seed)
    qf = rng.standard_normal((B, T, H, 128)) * rng.uniform(0.5, 2.0, size=(B, T, H, 1))
    kf = rng.standard_normal((B, T, H, 128)) * rng.uniform(0.5, 2.0, size=(B, T, H, 1))
    v = rng.standard_normal((B, T, H, 128))
    al = rng.uniform(0.9, 1.0, size=(B, T, H)).astype(np.float32)
    be = rng.uniform(0.0, 1.0, size=(B, T, H)).astype(np.float32)
    s0 = (0.3 * rng.standard_normal((B, H, 128, 64))).astype(np.float32) if S0 else None
    idx = np.stack([np.sort(rng.permutation(128)[:64]) for _ in range(H)]).astype(np.int32)
    r = inputs.round_to_bf16
    return r(qf), r(kf), r(v), al, be, s0, idx


def _run_both(qf, kf, v, al, be, s0, idx):
    import torch
    B, T, H, _ = kf.shape
    K, V = 64, 128
    dq, dk, dv = to_dev(qf, "bf16"), to_dev(kf, "bf16"), to_dev(v, "bf16")
    da, db = torch.from_numpy(al).cuda(), torch.from_numpy(be).cuda()
    ds0 = None if s0 is None else torch.from_numpy(s0).cuda()
    didx = torch.from_numpy(idx).cuda()
    # fused: the prologue inside the key-side pass
    need = binding.gdn_prefill_gathered_workspace_size(B, T, H, 128, K, V, binding.GDN_BF16)
    ws = torch.full((need,), 0xFF, dtype=torch.uint8, device="cuda")
    o1 = torch.full((B, T, H, V), float("nan"), dtype=torch.bfloat16, device="cuda")
    S1 = torch.full((B, H, V, K), float("nan"), device="cuda")
    binding.gdn_prefill_gathered(dq, dk, didx, 128, dv, da, db, ds0, o1, S1, B, T, H, K, V,
                                 binding.GDN_BF16, ws, need)
    torch.cuda.synchronize()
    assert binding.gdn_get_last_device_status() == binding.GDN_OK
    # unfused: the standalone prologue, then the two-pass prefill
    q = binding.gather_normalize(dq, didx)
    k = binding.gather_normalize(dk, didx)
    two = binding.gdn_prefill_two_pass_workspace_size(B, T, H, K, V, binding.GDN_BF16)
    ws2 = torch.empty(two, dtype=torch.uint8, device="cuda")
    o2 = torch.empty((B, T, H, V), dtype=torch.bfloat16, device="cuda")
    S2 = torch.empty((B, H, V, K), device="cuda")
    binding.gdn_prefill(q, k, dv, da, db, ds0, o2, S2, B, T, H, K, V, binding.GDN_BF16, ws2, two)
    torch.cuda.synchronize()
    assert binding.gdn_get_last_device_status() == binding.GDN_OK
    return (o1, S1), (o2, S2)


@pytest.mark.parametrize("B,T,H,S0", [(2, 300, 3, True), (1, 64, 1, False), (3, 1, 2, True),
                                      (4, 577, 8, False)])
def test_gathered_prefill_bit_identical_to_prologue_then_prefill(B, T, H, S0):
    import torch
    p = _problem(B, T, H, seed=T + H, S0=S0)
    (o1, S1), (o2, S2) = _run_both(*p)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(S1.view(torch.int32), S2.view(torch.int32))
    qf, kf, v, al, be, s0, idx = p
    qn = inputs.round_to_bf16(oracle.gather_normalize(qf, idx))
    kn = inputs.round_to_bf16(oracle.gather_normalize(kf, idx))
    o_ref, S_ref = oracle.recurrence(qn, kn, v, al, be, S0=s0)
    assert rel_err(to_np(o1), o_ref) <= TOL["bf16"]
    assert rel_err(to_np(S1), S_ref) <= TOL["bf16"]


def test_gathered_prefill_segment_parallel():
    """Few long sequences take the segment-parallel state pass; the gathered
    q', k' come from the same workspace."""
    import torch
    B, T, H = 1, 4133, 2
    assert binding.gdn_prefill_workspace_size(B, T, H, 64, 128, binding.GDN_BF16) > 0
    p = _problem(B, T, H, seed=5)
    (o1, S1), (o2, S2) = _run_both(*p)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(S1.view(torch.int32), S2.view(torch.int32))
    qf, kf, v, al, be, s0, idx = p
    qn = inputs.round_to_bf16(oracle.gather_normalize(qf, idx))
    kn = inputs.round_to_bf16(oracle.gather_normalize(kf, idx))
    o_ref, S_ref = oracle.recurrence(qn, kn, v, al, be, S0=s0)
    assert rel_err(to_np(o1), o_ref) <= TOL["bf16"]
    assert rel_err(to_np(S1), S_ref) <= TOL["bf16"]


def test_gathered_prefill_bad_index_is_reported_not_read():
    import torch
    qf, kf, v, al, be, s0, idx = _problem(1, 100, 2, seed=9)
    idx[1, 7] = 128  # out of range
    B, T, H = 1, 100, 2
    need = binding.gdn_prefill_gathered_workspace_size(B, T, H, 128, 64, 128, binding.GDN_BF16)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    o = torch.empty((B, T, H, 128), dtype=torch.bfloat16, device="cuda")
    S = torch.empty((B, H, 128, 64), device="cuda")
    binding.gdn_prefill_gathered(to_dev(qf, "bf16"), to_dev(kf, "bf16"),
                                 torch.from_numpy(idx).cuda(), 128, to_dev(v, "bf16"),
                                 torch.from_numpy(al).cuda(), torch.from_numpy(be).cuda(),
                                 torch.from_numpy(s0).cuda(), o, S, B, T, H, 64, 128,
                                 binding.GDN_BF16, ws, need)
    assert binding.gdn_get_last_device_status() == binding.GDN_ERR_DEVICE_BOUNDS
    # head 0 is untouched by the bad index
    qn = inputs.round_to_bf16(oracle.gather_normalize(qf[:, :, :1], idx[:1]))
    kn = inputs.round_to_bf16(oracle.gather_normalize(kf[:, :, :1], idx[:1]))
    o_ref, S_ref = oracle.recurrence(qn, kn, v[:, :, :1], al[:, :, :1], be[:, :, :1], S0=s0[:, :1])
    assert rel_err(to_np(o)[:, :, :1], o_ref) <= TOL["bf16"]
    assert rel_err(to_np(S)[:, :1], S_ref) <= TOL["bf16"]
    assert binding.gdn_get_last_device_status() == binding.GDN_OK


@pytest.mark.slow
def test_pruned_workload_gathered():
    """The prefill workload's full-width bf16 q/k, pruned to the workload's 64
    kept channels per head inside the prefill: sampled sequences (shortest and
    longest decay horizons) against the oracle on its own prologue."""
    import torch
    p = inputs.make_prefill()
    pp = inputs.make_prefill(pruned_K=64)
    idx = pp.meta["kept_channels"]
    o, ST = binding.prefill_gathered(to_dev(p.q, "bf16"), to_dev(p.k, "bf16"),
                                     torch.from_numpy(idx).cuda(), to_dev(p.v, "bf16"),
                                     torch.from_numpy(p.alpha).cuda(),
                                     torch.from_numpy(p.beta).cuda())
    assert binding.gdn_get_last_device_status() == binding.GDN_OK
    o, ST = to_np(o), to_np(ST)
    hor = -1.0 / np.log(p.alpha.astype(np.float64)).mean(axis=(0, 1))
    for b, h in [(0, int(np.argmin(hor))), (5, int(np.argmax(hor))), (7, 9)]:
        sub = inputs.take_sequences(p, [b], [h])
        qn = inputs.round_to_bf16(oracle.gather_normalize(sub.q, idx[h:h + 1]))
        kn = inputs.round_to_bf16(oracle.gather_normalize(sub.k, idx[h:h + 1]))
        o_ref, S_ref = oracle.recurrence(qn, kn, sub.v, sub.alpha, sub.beta)
        assert rel_err(o[b:b + 1, :, h:h + 1], o_ref) <= TOL["bf16"]
        assert rel_err(ST[b:b + 1, h:h + 1], S_ref) <= TOL["bf16"]
