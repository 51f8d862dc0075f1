"""Gated delta-rule recurrence on one GB300 GPU (sm_103a).

The compute lives in ``libgdn.so`` (C ABI in ``include/gdn.h``); this package
holds its ctypes binding, the in-tree build script and the seeded input
generator.  Importing the package does not load the library; the first call
does, and raises if the library has not been built.
"""
from .binding import (  # noqa: F401
    EXPORTS,
    GDN_BF16,
    GDN_FP32,
    GDNError,
    decode_step,
    gdn_decode_step,
    gdn_decode_step_gathered,
    gdn_gather_normalize,
    gather_normalize,
    gdn_get_last_device_status,
    gdn_prefill,
    gdn_prefill_gated,
    gdn_prefill_gated_chunked,
    gdn_prefill_gated_chunked_workspace_size,
    prefill_gated_chunked,
    gdn_prefill_gathered,
    prefill_gathered,
    gdn_decode_step_gated,
    prefill_gated,
    prefill_truncated,
    channel_gram,
    drrqr_select,
    state_truncate,
    gdn_state_truncate,
    gdn_prefill_truncated,
    gdn_prefill_workspace_size,
    gdn_prefill_two_pass_workspace_size,
    gdn_selftest_wait_timeout,
    gdn_state_rank,
    gdn_status_string,
    gdn_version,
    prefill,
    state_rank,
)
