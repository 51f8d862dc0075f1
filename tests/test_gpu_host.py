"""gdn_prefill_host: the prefill on host buffers, pipelined over token
windows, against gdn_prefill on device copies and against the oracle."""
import numpy as np
import pytest

import oracle
from gpu_util import TOL, rel_err, to_dev, to_np
from gated_delta_rule_49_gb300 import binding, inputs

pytestmark = pytest.mark.gpu


def _host(x, dtype, pin=True):
    import torch
    x = np.ascontiguousarray(x, dtype=np.float32)
    if dtype == "bf16":
        t = torch.from_numpy(inputs.bf16_bits(x).view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(x.copy())
    return t.pin_memory() if pin else t


def _run_host(p, window, S0=None, want_o=True, want_state=True, pin=True):
    import torch
    B, T, H, K = p.k.shape
    V = p.v.shape[-1]
    dt = binding.GDN_BF16 if p.dtype == "bf16" else binding.GDN_FP32
    q, k, v = (_host(getattr(p, n), p.dtype, pin) for n in ("q", "k", "v"))
    al, be = _host(p.alpha, "fp32", pin), _host(p.beta, "fp32", pin)
    s0 = None if S0 is None else _host(S0, "fp32", pin)
    tdt = torch.bfloat16 if p.dtype == "bf16" else torch.float32
    o = torch.empty((B, T, H, V), dtype=tdt)
    ST = torch.empty((B, H, V, K), dtype=torch.float32)
    if pin:
        o, ST = o.pin_memory(), ST.pin_memory()
    need = binding.gdn_prefill_host_workspace_size(B, T, H, K, V, dt, window)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    binding.gdn_prefill_host(q, k, v, al, be, s0, o if want_o else None,
                             ST if want_state else None, B, T, H, K, V, dt, window, ws, need)
    torch.cuda.synchronize()
    return (o.float().numpy() if want_o else None), (ST.numpy() if want_state else None)


@pytest.mark.parametrize("K,V,dtype", [(128, 128, "bf16"), (64, 128, "bf16"), (32, 32, "fp32")])
@pytest.mark.parametrize("window", [128, 512])
def test_aligned_windows_equal_the_device_prefill(K, V, dtype, window):
    """Windows that are multiples of 64 keep the chunk boundaries of one
    whole-sequence prefill: identical outputs and final state.  (T = 900 is
    15 chunks, below the length at which a prefill of so few sequences would
    run segment-parallel, which rounds differently.)"""
    import torch
    p = inputs.make_tiny(seed=window + K, B=2, H=3, T=900, K=K, V=V, dtype=dtype)
    S0 = (0.2 * np.random.default_rng(1).standard_normal((2, 3, V, K))).astype(np.float32)
    assert binding.gdn_prefill_workspace_size(2, 900, 3, K, V, 0) == 0  # whole-sequence mode
    o_h, S_h = _run_host(p, window, S0=S0)
    d = {n: to_dev(getattr(p, n), dtype) for n in ("q", "k", "v")}
    o_d, S_d = binding.prefill(d["q"], d["k"], d["v"], torch.from_numpy(p.alpha).cuda(),
                               torch.from_numpy(p.beta).cuda(), torch.from_numpy(S0).cuda())
    assert np.array_equal(o_h, to_np(o_d)) and np.array_equal(S_h, to_np(S_d))


@pytest.mark.parametrize("window", [100, 1, 777])
def test_ragged_windows_match_the_oracle(window):
    p = inputs.make_tiny(seed=window, B=2, H=2, T=300, K=128, V=128, dtype="bf16")
    o_h, S_h = _run_host(p, window)
    o_ref, S_ref = oracle.recurrence(p.q, p.k, p.v, p.alpha, p.beta)
    assert rel_err(o_h, o_ref) <= TOL["bf16"] and rel_err(S_h, S_ref) <= TOL["bf16"]


def test_null_outputs_zero_length_and_pageable_memory():
    p = inputs.make_tiny(seed=5, B=2, H=2, T=200, K=64, V=128, dtype="bf16")
    S0 = (0.1 * np.random.default_rng(2).standard_normal((2, 2, 128, 64))).astype(np.float32)
    o_ref, S_ref = oracle.recurrence(p.q, p.k, p.v, p.alpha, p.beta, S0=S0)
    _, S_h = _run_host(p, 64, S0=S0, want_o=False)
    assert rel_err(S_h, S_ref) <= TOL["bf16"]
    o_h, _ = _run_host(p, 64, S0=S0, want_state=False, pin=False)  # pageable host memory
    assert rel_err(o_h, o_ref) <= TOL["bf16"]
    p0 = inputs.make_tiny(seed=6, B=2, H=2, T=0, K=64, V=128, dtype="bf16")
    _, S_e = _run_host(p0, 64, S0=S0, want_o=False)
    assert np.array_equal(S_e, S0)
    _, S_z = _run_host(p0, 64, want_o=False)
    assert not np.any(S_z)
