"""Chunked gated delta rule (Gated DeltaNet) operator for NVIDIA GB300.

The operator runs in hand-written sm_103a CUDA kernels behind the C ABI of
include/gdn.h (built into ``_build/libgdn.so``); this package holds the build
script, the thin ctypes binding and the seeded synthetic workloads.
"""

from .gdn import (  # noqa: F401
    GdnError,
    chunk_gated_delta_rule,
    chunk_gated_delta_rule_bwd,
    chunk_gated_delta_rule_fwd,
    gdn_chunk_bwd,
    gdn_chunk_bwd_workspace_size,
    gdn_chunk_fwd,
    gdn_chunk_fwd_workspace_size,
    gdn_get_last_device_error,
    gdn_status_string,
)
