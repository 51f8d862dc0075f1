"""gdn_prefill_noalloc: the prefill for callers that cannot allocate device
memory (a component that only gets device pointers from the framework that
owns the GPU's memory, or a server that must not call cudaMalloc after
start-up).  Its scratch is a fixed array inside the library; its results must
match gdn_prefill given a caller-allocated workspace, call after call, since
every call reuses the same array.

This file is named so that pytest collects it last."""
import ctypes

import numpy as np
import pytest

from gated_delta_rule_49_gb300 import binding, build, inputs

pytestmark = pytest.mark.gpu

TOL_BF16 = 1e-2  # max |x - ref| / max |ref|, the bf16 parity bar of the other tests


def _problem(K, T, seed):
    rng = np.random.default_rng(seed)
    B, H, V = 1, 2, 128
    q = rng.standard_normal((B, T, H, K)); q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k = rng.standard_normal((B, T, H, K)); k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, T, H, V))
    alpha = rng.uniform(0.97, 1.0, size=(B, T, H)).astype(np.float32)
    beta = rng.uniform(0.0, 1.0, size=(B, T, H)).astype(np.float32)
    S0 = (0.3 * rng.standard_normal((B, H, V, K))).astype(np.float32)
    r = inputs.round_to_bf16
    return r(q), r(k), r(v), alpha, beta, S0


def _rel(a, b):
    a = a.double().cpu().numpy()
    b = b.double().cpu().numpy()
    return float(np.abs(a - b).max() / np.abs(b).max())


def test_noalloc_matches_workspace_prefill_twice():
    import torch
    assert torch.cuda.is_available()
    build.build()
    lib = binding.load()

    def dev(x, bf):
        x = np.ascontiguousarray(x, np.float32)
        if bf:
            return torch.from_numpy(inputs.bf16_bits(x).view(np.int16)).view(torch.bfloat16).cuda()
        return torch.from_numpy(x).cuda()

    for call, (K, T, seed) in enumerate([(128, 4096, 1), (64, 4133, 2)]):
        q, k, v, alpha, beta, S0 = _problem(K, T, seed)
        B, H, V = 1, 2, 128
        need = binding.gdn_prefill_workspace_size(B, T, H, K, V, binding.GDN_BF16)
        # this shape takes the segment-parallel path, so the scratch is used
        assert 0 < need <= binding.gdn_prefill_noalloc_max_workspace()
        dq, dk, dv = dev(q, True), dev(k, True), dev(v, True)
        da, db, dS0 = dev(alpha, False), dev(beta, False), dev(S0, False)

        # existing entry point with a caller-allocated workspace
        o_ref = torch.empty((B, T, H, V), dtype=torch.bfloat16, device="cuda")
        S_ref = torch.empty((B, H, V, K), device="cuda")
        ws = torch.empty(need, dtype=torch.uint8, device="cuda")
        binding.gdn_prefill(dq, dk, dv, da, db, dS0, o_ref, S_ref, B, T, H, K, V,
                            binding.GDN_BF16, ws, need)

        # the no-allocation entry point, called directly through the C ABI
        o = torch.full((B, T, H, V), float("nan"), dtype=torch.bfloat16, device="cuda")
        S = torch.full((B, H, V, K), float("nan"), device="cuda")
        stream = torch.cuda.current_stream().cuda_stream
        rc = lib.gdn_prefill_noalloc(dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), da.data_ptr(),
                                     db.data_ptr(), dS0.data_ptr(), o.data_ptr(), S.data_ptr(),
                                     B, T, H, K, V, binding.GDN_BF16, ctypes.c_void_p(stream))
        assert rc == binding.GDN_OK, binding.status_string(rc)
        assert binding.gdn_get_last_device_status() == binding.GDN_OK
        assert not torch.isnan(o.float()).any() and not torch.isnan(S).any()
        assert _rel(o.float(), o_ref.float()) <= TOL_BF16, call
        assert _rel(S, S_ref) <= TOL_BF16, call


def rejected_shape():
    """A problem whose segment-parallel scratch exceeds the array on this
    device: few long sequences, more heads until the scratch no longer fits
    (the segment count depends on the SM count, so the shape is searched)."""
    cap = binding.gdn_prefill_noalloc_max_workspace()
    for T in (65536, 262144):
        for H in range(1, 129):
            need = binding.gdn_prefill_workspace_size(1, T, H, 128, 128, binding.GDN_BF16)
            if need > cap:
                return 1, T, H, need
    return None


def test_noalloc_rejects_problems_beyond_its_scratch():
    import torch
    assert torch.cuda.is_available()
    lib = binding.load()
    found = rejected_shape()
    assert found is not None, "no shape needs more scratch than the array holds"
    B, T, H, need = found
    K, V = 128, 128
    assert need > binding.gdn_prefill_noalloc_max_workspace()
    fake = 0x10000  # never dereferenced: the size check returns before any launch
    rc = lib.gdn_prefill_noalloc(fake, fake, fake, fake, fake, None, fake, fake, B, T, H, K, V,
                                 binding.GDN_BF16, None)
    assert rc == binding.GDN_ERR_WORKSPACE
    # nothing was launched: the device status word is clean
    assert binding.gdn_get_last_device_status() == binding.GDN_OK
