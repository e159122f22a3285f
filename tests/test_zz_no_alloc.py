"""The no-allocation chunked forward against the regular one.

``gdn_chunk_fwd_noalloc`` serves callers that cannot give the library a
workspace (a host runtime that owns a fixed device-memory budget and forbids
its plugins to allocate, or a latency-critical loop that must not hit
cudaMalloc's implicit synchronisation).  It runs the same kernels on a fixed
device array owned by the library.  This file is collected last so that a run
stopping at the first failure has already run every other test; it also
passes when run on its own in a fresh process.
"""
import ctypes

import pytest
import torch

import gated_delta_rule_kk_gb300 as gdn
from gated_delta_rule_kk_gb300 import _lib, synth
from gated_delta_rule_kk_gb300._lib import GdnChunkArgs, Status

from _util import to_dev

pytestmark = pytest.mark.gpu


def _regular(d):
    return gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], scale=d["scale"],
                             initial_state=d["h0"], cu_seqlens=d["cu_seqlens"])


def _noalloc(d):
    return gdn.gdn_chunk_fwd_noalloc(d["q"], d["k"], d["v"], d["g"], d["beta"], scale=d["scale"],
                                     initial_state=d["h0"], cu_seqlens=d["cu_seqlens"])


@pytest.mark.parametrize("lengths", [None, [70, 1, 200]])
def test_noalloc_matches_regular_entry_point_twice(lengths):
    if lengths is None:
        inp = synth.prefill_inputs(91, 2, 300, 4, 2, 128, 128, h0_std=0.1)
    else:
        inp = synth.prefill_inputs(92, 1, sum(lengths), 4, 2, 128, 128, h0_std=0.1,
                                   lengths=lengths)
    d = to_dev(inp)
    o_ref, ht_ref = _regular(d)
    assert gdn.gdn_check_device_error() == Status.OK
    for call in range(2):
        o, ht = _noalloc(d)
        assert gdn.gdn_check_device_error() == Status.OK
        # the same kernels on the same inputs: bit for bit the regular results
        assert torch.equal(o, o_ref), f"o differs on call {call}"
        assert torch.equal(ht, ht_ref), f"ht differs on call {call}"


def test_noalloc_rejects_problems_beyond_the_fixed_array():
    lib = _lib.load()
    limit = gdn.gdn_noalloc_scratch_bytes()
    # a problem whose workspace needs more than the fixed array
    a = GdnChunkArgs(dtype=1, q=0x10000, k=0x10000, v=0x10000, g=0x10000, beta=0x10000,
                     o=0x10000, B=64, T=8192, H=16, Hg=16, K=128, V=128, N=64, chunk_size=64)
    need = ctypes.c_size_t(0)
    assert lib.gdn_chunk_workspace_size(ctypes.byref(a), ctypes.byref(need)) == Status.OK
    assert need.value > limit
    st = lib.gdn_chunk_fwd_noalloc(ctypes.byref(a), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == Status.WORKSPACE
    assert b"32 MiB" in lib.gdn_last_error_message()
