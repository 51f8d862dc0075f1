"""Long sequences on few heads run segment-parallel (a first pass for each
segment's zero-start end state and transition matrix, a combine, a second
pass from the true start states).  Results must match the oracle exactly as
the one-CTA-per-sequence path does."""
import numpy as np
import pytest

import oracle
from gpu_util import TOL, problem_to_dev, rel_err, to_np
from gated_delta_rule_49_gb300 import binding, inputs

pytestmark = pytest.mark.gpu


def long_problem(K, T, seed=0, B=1, H=2, with_S0=True):
    rng = np.random.default_rng(seed + T + K)
    q = rng.standard_normal((B, T, H, K)); q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k = rng.standard_normal((B, T, H, K)); k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, T, H, 128))
    alpha = rng.uniform(0.97, 1.0, size=(B, T, H)).astype(np.float32)
    beta = rng.uniform(0.0, 1.0, size=(B, T, H)).astype(np.float32)
    S0 = (0.3 * rng.standard_normal((B, H, 128, K))).astype(np.float32) if with_S0 else None
    r = inputs.round_to_bf16
    return inputs.Problem("long-small", "bf16", r(q), r(k), r(v), alpha, beta, S0)


@pytest.mark.parametrize("K", [128, 64])
@pytest.mark.parametrize("T", [4096, 4133])
def test_segmented_prefill_matches_oracle(K, T):
    import torch
    p = long_problem(K, T)
    B, T_, H, K_, V = p.shape
    ws_bytes = binding.gdn_prefill_workspace_size(B, T, H, K, V, binding.GDN_BF16)
    assert ws_bytes > 0, "this shape should take the segment-parallel path"
    d = problem_to_dev(p)
    o = torch.full((B, T, H, V), float("nan"), dtype=torch.bfloat16, device="cuda")
    S = d["S0"].clone()  # in place: S_T overwrites S0
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    binding.gdn_prefill(d["q"], d["k"], d["v"], d["alpha"], d["beta"], S, o, S, B, T, H, K, V,
                        binding.GDN_BF16, ws, ws_bytes)
    assert binding.gdn_get_last_device_status() == binding.GDN_OK
    o_ref, S_ref = oracle.recurrence(p.q, p.k, p.v, p.alpha, p.beta, S0=p.S0)
    eo, es = rel_err(to_np(o), o_ref), rel_err(to_np(S), S_ref)
    assert eo <= TOL["bf16"] and es <= TOL["bf16"], (eo, es)


def test_segmented_zero_state_and_missing_workspace():
    import torch
    p = long_problem(128, 2048, with_S0=False)
    B, T, H, K, V = p.shape
    ws_bytes = binding.gdn_prefill_workspace_size(B, T, H, K, V, binding.GDN_BF16)
    assert ws_bytes > 0
    d = problem_to_dev(p)
    o = torch.empty((B, T, H, V), dtype=torch.bfloat16, device="cuda")
    ST = torch.empty((B, H, V, K), device="cuda")
    with pytest.raises(binding.GDNError) as e:
        binding.gdn_prefill(d["q"], d["k"], d["v"], d["alpha"], d["beta"], None, o, ST, B, T, H,
                            K, V, binding.GDN_BF16, None, 0)
    assert e.value.status == binding.GDN_ERR_WORKSPACE
    o2, ST2 = binding.prefill(d["q"], d["k"], d["v"], d["alpha"], d["beta"])
    o_ref, S_ref = oracle.recurrence(p.q, p.k, p.v, p.alpha, p.beta)
    assert rel_err(to_np(o2), o_ref) <= TOL["bf16"] and rel_err(to_np(ST2), S_ref) <= TOL["bf16"]
