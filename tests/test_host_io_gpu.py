"""gdn_chunk_fwd_host: the chunked forward end to end from host buffers.

The host entry point cuts the problem into pieces (time ranges handing the
fp32 state on, or ranges of whole sequences) and overlaps their copies with
the kernels.  Its results must equal those of gdn_chunk_fwd on device copies
of the same inputs bit for bit, for each way of cutting; one small case is
also held against the oracle directly.
"""
import ctypes

import numpy as np
import pytest
import torch

import gated_delta_rule_kk_gb300 as gdn
from gated_delta_rule_kk_gb300 import _lib, synth
from gated_delta_rule_kk_gb300._lib import GdnChunkArgs, Status
from oracle import recurrence as R

from _util import TOL_F32, assert_close, to_dev

pytestmark = pytest.mark.gpu


def _device(inp, h0=True):
    d = to_dev(inp)
    o, ht = gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], scale=d["scale"],
                              initial_state=d["h0"] if h0 else None, cu_seqlens=d["cu_seqlens"],
                              g_is_cumsum=d["g_is_cumsum"], segments=1)
    torch.cuda.synchronize()
    assert gdn.gdn_check_device_error() == Status.OK
    return o.cpu(), ht.cpu()


def _host(inp, pin=True, h0=True, want_ht=True):
    def p(t):
        return None if t is None else (t.pin_memory() if pin else t.clone())
    o, ht = gdn.gdn_chunk_fwd_host(p(inp["q"]), p(inp["k"]), p(inp["v"]), p(inp["g"]),
                                   p(inp["beta"]), scale=inp["scale"],
                                   initial_state=p(inp["h0"]) if h0 else None,
                                   cu_seqlens=p(inp["cu_seqlens"]),
                                   g_is_cumsum=inp["g_is_cumsum"], output_final_state=want_ht)
    torch.cuda.synchronize()
    assert gdn.gdn_check_device_error() == Status.OK
    return o, ht


def _same(a, b, what):
    assert a.shape == b.shape and a.dtype == b.dtype, what
    diff = (a.float() - b.float()).abs().max().item() if a.numel() else 0.0
    assert torch.equal(a, b), f"{what}: host path differs from device path (max {diff:.3e})"


CASES = {
    # B=2, T=4096: four time pieces (34, 17, 9, 4 chunks), state handed on
    "time_cut_bench_shape": lambda: synth.prefill_inputs(61, 2, 4096, 16, 16, 128, 128, h0_std=0.1),
    # T=2100 = 32 full chunks + a ragged tail of 52 tokens: three time pieces
    "time_cut_ragged": lambda: synth.prefill_inputs(62, 1, 2100, 4, 2, 128, 64, h0_std=0.1),
    # 16 short sequences: four pieces of four whole sequences
    "batch_cut": lambda: synth.prefill_inputs(63, 16, 512, 8, 4, 128, 128, h0_std=0.1),
    # packed sequences, pieces at sequence ends
    "varlen": synth.varlen_gqa,
    # the fp32 CUDA-core path with a time cut (K=64, V=48)
    "time_cut_fp32": lambda: synth.prefill_inputs(64, 1, 2200, 2, 1, 64, 48,
                                                  dtype=torch.float32, h0_std=0.1),
}


@pytest.mark.parametrize("name", list(CASES))
def test_host_equals_device_path(name):
    inp = CASES[name]()
    o_d, ht_d = _device(inp)
    o_h, ht_h = _host(inp)
    _same(o_h, o_d, f"{name} o")
    _same(ht_h, ht_d, f"{name} ht")


def test_no_initial_state_no_final_state_and_pageable_buffers():
    inp = synth.prefill_inputs(65, 2, 2048, 4, 4, 128, 128, h0_std=0.1)
    o_d, _ = _device(inp, h0=False)
    o_h, ht_h = _host(inp, pin=False, h0=False, want_ht=False)
    assert ht_h is None
    _same(o_h, o_d, "o")


def test_host_path_against_oracle():
    inp = synth.prefill_inputs(66, 1, 2176, 2, 1, 32, 16, dtype=torch.float32, h0_std=0.2)
    o, ht = _host(inp)
    o_ref, ht_ref = R.gdn_recurrent(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                                    scale=inp["scale"], h0=inp["h0"])
    assert_close(o, o_ref, TOL_F32, "o")
    assert_close(ht, ht_ref, TOL_F32, "ht")


def test_repeated_calls_reuse_the_workspace():
    inp = synth.prefill_inputs(67, 2, 3072, 4, 2, 128, 128, h0_std=0.1)
    pin = {k: (v.pin_memory() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    ws = torch.empty(gdn.gdn_chunk_host_workspace_bytes(pin["q"], pin["v"]), dtype=torch.uint8,
                     device="cuda")
    outs = []
    for _ in range(3):
        o, ht = gdn.gdn_chunk_fwd_host(pin["q"], pin["k"], pin["v"], pin["g"], pin["beta"],
                                       scale=pin["scale"], initial_state=pin["h0"], workspace=ws)
        outs.append((o, ht))
    torch.cuda.synchronize()
    o_d, ht_d = _device(inp)
    for o, ht in outs:
        _same(o, o_d, "o")
        _same(ht, ht_d, "ht")


def test_device_pointers_are_rejected():
    inp = synth.prefill_inputs(68, 1, 128, 2, 2, 128, 128)
    d = to_dev(inp)
    lib = _lib.load()
    host_o = torch.empty((1, 128, 2, 128), dtype=torch.bfloat16)
    ws = torch.empty(1 << 24, dtype=torch.uint8, device="cuda")
    vp = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    a = GdnChunkArgs(dtype=1, q=vp(d["q"]), k=vp(inp["k"]), v=vp(inp["v"]), g=vp(inp["g"]),
                     beta=vp(inp["beta"]), o=vp(host_o), B=1, T=128, H=2, Hg=2, K=128, V=128,
                     N=1, chunk_size=64, workspace=vp(ws), workspace_bytes=ws.numel())
    assert lib.gdn_chunk_fwd_host(ctypes.byref(a), None) == Status.INVALID_ARG
    assert "host memory" in lib.gdn_last_error_message().decode()
    a.q = vp(inp["q"])
    a.workspace = vp(host_o)
    assert lib.gdn_chunk_fwd_host(ctypes.byref(a), None) in (Status.WORKSPACE, Status.MISALIGNED)
    a.workspace = vp(ws)
    assert lib.gdn_chunk_fwd_host(ctypes.byref(a), None) == Status.OK
    torch.cuda.synchronize()
    o_d, _ = gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], segments=1)
    _same(host_o, o_d.cpu(), "o")


def test_fp32_output_from_host_buffers_equals_device_entry_point():
    """o in fp32 (twice the bytes per row of bf16 o) through time pieces."""
    inp = synth.prefill_inputs(97, 2, 1500, 2, 1, 128, 128, h0_std=0.1)
    d = to_dev(inp)
    o_d, ht_d = gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], scale=d["scale"],
                                  initial_state=d["h0"], out_dtype=torch.float32, segments=1)
    o_h, ht_h = gdn.gdn_chunk_fwd_host(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                                       scale=inp["scale"], initial_state=inp["h0"],
                                       out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert o_h.dtype == torch.float32
    assert torch.equal(o_h, o_d.cpu())
    assert torch.equal(ht_h, ht_d.cpu())
