"""The bounded-wait failure path on the GPU, made to run out on purpose.

Every kernel that waits on an asynchronous copy or tensor-core operation
polls its mbarrier a bounded number of times and records GDN_ERR_TIMEOUT
instead of hanging.  gdn_self_test_wait runs that same wait on a barrier
nothing arrives on (no copy or MMA in flight), with a poll limit of one, so
the timeout is reached at once; the context stays usable afterwards.
"""
import ctypes

import pytest
import torch

import gated_delta_rule_kk_gb300 as gdn
from gated_delta_rule_kk_gb300 import _lib, synth
from gated_delta_rule_kk_gb300._lib import Status

pytestmark = pytest.mark.gpu


def _self_test(arrive, polls):
    lib = _lib.load()
    st = lib.gdn_self_test_wait(arrive, polls,
                                ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == Status.OK
    return gdn.gdn_check_device_error()


def test_wait_that_runs_out_records_timeout_and_the_context_stays_usable():
    assert gdn.gdn_check_device_error() == Status.OK
    assert _self_test(0, 1) == Status.TIMEOUT
    assert _self_test(0, 64) == Status.TIMEOUT
    assert gdn.gdn_check_device_error() == Status.OK  # reading cleared it
    # a completed phase passes on the first poll
    assert _self_test(1, 1) == Status.OK
    # the library still computes afterwards
    inp = synth.prefill_inputs(71, 1, 100, 2, 1, 128, 128, dtype=torch.bfloat16)
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    o, ht = gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"])
    assert gdn.gdn_check_device_error() == Status.OK
    assert torch.isfinite(o.float()).all() and torch.isfinite(ht).all()
