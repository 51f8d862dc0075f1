"""Pruning prologue on the GPU: the gather + renormalise kernel and the decode
step that fuses it, against the float64 oracle on the same inputs."""
import numpy as np
import pytest

import oracle
from gpu_util import TOL, rel_err, to_dev, to_np
from gated_delta_rule_49_gb300 import binding, inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clear_device_status():
    binding.gdn_get_last_device_status()  # read-and-clear whatever earlier tests left


def _full_width(B, T, H, K, dtype, seed):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((B, T, H, K)) * rng.uniform(0.5, 2.0, size=(B, T, H, 1))
    return inputs.round_to_bf16(x) if dtype == "bf16" else x.astype(np.float32)


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("K_in,K_out", [(128, 64), (128, 32), (100, 64), (1024, 64), (36, 32)])
def test_gather_normalize_matches_oracle(dtype, K_in, K_out):
    """Row widths that take the staged kernel (row bytes a multiple of 16, one
    to 28 rows per warp tile) and the row-wise one (bf16 rows of 100 channels);
    808 rows leave a ragged last tile."""
    import torch
    B, T, H = 2, 101, 4
    x = _full_width(B, T, H, K_in, dtype, 7 + K_out)
    rng = np.random.default_rng(3)
    idx = np.stack([rng.permutation(K_in)[:K_out] for _ in range(H)]).astype(np.int32)
    y = binding.gather_normalize(to_dev(x, dtype), torch.from_numpy(idx).cuda())
    ref = oracle.gather_normalize(x, idx)
    tol = TOL["bf16"] if dtype == "bf16" else 1e-5
    assert rel_err(to_np(y), ref) <= tol
    assert binding.gdn_get_last_device_status() == binding.GDN_OK


@pytest.mark.parametrize("dtype,K_in", [("fp32", 64), ("bf16", 100)])
def test_gather_normalize_bad_index_is_reported_not_read(dtype, K_in):
    """Staged (fp32, 256-byte rows) and row-wise (bf16, 200-byte rows) kernels."""
    import torch
    x = _full_width(1, 8, 2, K_in, dtype, 1)
    idx = np.tile(np.arange(32, dtype=np.int32), (2, 1))
    idx[1, 5] = K_in  # out of range
    y = binding.gather_normalize(to_dev(x, dtype), torch.from_numpy(idx).cuda())
    assert binding.gdn_get_last_device_status() == binding.GDN_ERR_DEVICE_BOUNDS
    good = oracle.gather_normalize(x[:, :, :1], idx[:1])
    tol = TOL["bf16"] if dtype == "bf16" else 1e-5
    assert rel_err(to_np(y)[:, :, :1], good) <= tol
    assert np.all(to_np(y)[:, :, 1, 5] == 0.0)
    assert binding.gdn_get_last_device_status() == binding.GDN_OK


@pytest.mark.parametrize("K", [64, 32])
def test_decode_gathered_matches_oracle(K):
    """Full-width q/k of width 128 pruned to K kept channels inside the step."""
    import torch
    B, H, V, K_in, steps = 3, 4, 128 if K == 64 else 32, 128, 12
    rng = np.random.default_rng(K)
    qf = _full_width(B, steps, H, K_in, "bf16", 11)
    kf = _full_width(B, steps, H, K_in, "bf16", 12)
    v = inputs.round_to_bf16(rng.standard_normal((B, steps, H, V)))
    al = rng.uniform(0.7, 1.0, size=(B, steps, H)).astype(np.float32)
    be = rng.uniform(0.0, 1.0, size=(B, steps, H)).astype(np.float32)
    S0 = (0.3 * rng.standard_normal((B, H, V, K))).astype(np.float32)
    idx = np.stack([np.sort(rng.permutation(K_in)[:K]) for _ in range(H)]).astype(np.int32)
    didx = torch.from_numpy(idx).cuda()
    S = torch.from_numpy(S0).cuda()
    outs = []
    for t in range(steps):
        o = torch.empty((B, H, V), dtype=torch.bfloat16, device="cuda")
        binding.gdn_decode_step_gathered(
            to_dev(np.ascontiguousarray(qf[:, t]), "bf16"), to_dev(np.ascontiguousarray(kf[:, t]), "bf16"),
            didx, K_in, to_dev(np.ascontiguousarray(v[:, t]), "bf16"),
            torch.from_numpy(np.ascontiguousarray(al[:, t])).cuda(),
            torch.from_numpy(np.ascontiguousarray(be[:, t])).cuda(), S, o, B, H, K, V,
            binding.GDN_BF16)
        outs.append(to_np(o))
    o_gpu = np.stack(outs, axis=1)
    qn = oracle.gather_normalize(qf, idx)
    kn = oracle.gather_normalize(kf, idx)
    o_ref, S_ref = oracle.recurrence(qn, kn, v, al, be, S0=S0)
    assert rel_err(o_gpu, o_ref) <= TOL["bf16"] and rel_err(to_np(S), S_ref) <= TOL["bf16"]
    assert binding.gdn_get_last_device_status() == binding.GDN_OK


@pytest.mark.slow
def test_pruned_workload_through_the_prologue():
    """Full-width bf16 q/k of the prefill workload, pruned to 64 kept channels
    per head by the prologue kernel, then the d_k' = 64 prefill: sampled
    sequences against the oracle on the oracle's own prologue, whose output is
    rounded to bf16 as the prologue kernel stores it."""
    import torch
    p = inputs.make_prefill()
    pp = inputs.make_prefill(pruned_K=64)
    idx = pp.meta["kept_channels"]
    didx = torch.from_numpy(idx).cuda()
    q = binding.gather_normalize(to_dev(p.q, "bf16"), didx)
    k = binding.gather_normalize(to_dev(p.k, "bf16"), didx)
    v = to_dev(p.v, "bf16")
    al = torch.from_numpy(p.alpha).cuda()
    be = torch.from_numpy(p.beta).cuda()
    o, ST = binding.prefill(q, k, v, al, be)
    o, ST = to_np(o), to_np(ST)
    for b, h in [(0, 3), (6, 12)]:
        sub = inputs.take_sequences(p, [b], [h])
        qn = inputs.round_to_bf16(oracle.gather_normalize(sub.q, idx[h:h + 1]))
        kn = inputs.round_to_bf16(oracle.gather_normalize(sub.k, idx[h:h + 1]))
        o_ref, S_ref = oracle.recurrence(qn, kn, sub.v, sub.alpha, sub.beta)
        assert rel_err(o[b:b + 1, :, h:h + 1], o_ref) <= TOL["bf16"]
        assert rel_err(ST[b:b + 1, h:h + 1], S_ref) <= TOL["bf16"]
