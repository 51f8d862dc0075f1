"""Failure detection on the GPU without a fault: a bounded wait that runs out
reports GDN_ERR_TIMEOUT through the device status word, and the context stays
usable afterwards."""
import numpy as np
import pytest

import oracle
from gpu_util import rel_err, run_prefill
from gated_delta_rule_49_gb300 import binding, inputs

pytestmark = pytest.mark.gpu


def test_wait_timeout_is_reported_and_context_survives():
    import torch
    assert torch.cuda.is_available()
    binding.load()
    assert binding.gdn_get_last_device_status() == binding.GDN_OK
    binding.gdn_selftest_wait_timeout(2_000_000)  # ~1 ms of SM clocks
    assert binding.gdn_get_last_device_status() == binding.GDN_ERR_TIMEOUT
    assert binding.gdn_get_last_device_status() == binding.GDN_OK  # read clears it
    # the device still computes correctly
    p = inputs.make_prefill(B=1, T=70, H=2)
    o, ST = run_prefill(p)
    o_ref, S_ref = oracle.recurrence(p.q, p.k, p.v, p.alpha, p.beta)
    assert rel_err(o, o_ref) <= 1e-2 and rel_err(ST, S_ref) <= 1e-2
