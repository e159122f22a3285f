"""Gated delta-rule (GDN / KDA) chunked forward and decode for GB300 (sm_103a).

The arithmetic lives in the CUDA library built from ``csrc/`` (see
``build_lib.py``); this package holds its ctypes binding and the seeded
synthetic input generators.
"""
from .api import (  # noqa: F401
    gdn_check_device_error, gdn_chunk_fwd, gdn_chunk_segment_count, gdn_chunk_fwd_host, gdn_chunk_fwd_noalloc,
    gdn_chunk_state_bwd, gdn_chunk_state_fwd,
    gdn_chunk_host_workspace_bytes, gdn_decode,
    gdn_noalloc_scratch_bytes, kda_chunk_fwd,
)
from ._lib import GateKind, GdnError, Status  # noqa: F401
