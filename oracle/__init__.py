"""fp64 CPU oracle for the gated delta rule (test infrastructure only).

This package is test infrastructure.  Only the test-suite, the smoke check in
``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import it; the
CUDA library and its Python binding never do, and it imports nothing from them.

Modules
-------
``recurrence``  the method written out token by token (the definition).
``brute``       the closed-form product of the per-token transition matrices.
``chunked``     an independent fp64 chunked (WY) rewrite for any chunk length.
"""
from .recurrence import (  # noqa: F401
    gdn_recurrent,
    kda_recurrent,
    decode_gates,
    l2_normalize,
    softplus,
    gdn_decode,
    raw_gate_from_chunk_cumsum,
    sequence_bounds,
)
