"""Decode step (T = 1..4) on the GPU against the fp64 oracle."""
import numpy as np
import pytest
import torch

from gated_delta_rule_kk_gb300 import Status, gdn_check_device_error, gdn_decode
from gated_delta_rule_kk_gb300 import synth
from oracle import recurrence as R

from _fullsize import decode_all_entries
from _util import TOL_BF16, assert_close, to_dev

pytestmark = pytest.mark.gpu


def run_gpu(inp, **kw):
    """o and the updated states in fp32 (the values the bound applies to), plus
    the bf16 pool after the call.  A second call with the default bf16 o must
    give that o rounded to nearest even, and the pool must hold the fp32
    states rounded the same way, bit for bit."""
    d = to_dev(inp)
    B, T, H, K = d["q"].shape
    HV, V = d["v"].shape[2], d["v"].shape[3]
    args = (d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"], d["dt_bias"])
    kw = dict(slot_indices=d["slot_indices"], scale=d["scale"], **kw)
    state = d["state"].clone()
    st32 = torch.full((B, HV, V, K), float("nan"), device="cuda")
    o = gdn_decode(*args, state, out_dtype=torch.float32, new_state_f32=st32, **kw)
    state16 = d["state"].clone()
    o16 = gdn_decode(*args, state16, **kw)
    assert torch.equal(o16, o.to(torch.bfloat16)), "bf16 o is not the RNE of the fp32 o"
    assert torch.equal(state16, state)
    slots = (torch.arange(B, device="cuda") if d["slot_indices"] is None
             else d["slot_indices"].long())
    ok = (slots >= 0) & (slots < state.shape[0])
    assert torch.equal(state[slots[ok]], st32[ok].to(torch.bfloat16)), \
        "the pool does not hold the RNE of the fp32 states"
    return o, st32, state


def oracle_for(inp, batch, **kw):
    """Oracle on the batch entries `batch`, with only their slots of the pool."""
    slots = inp["slot_indices"]
    slots = np.arange(inp["dims"]["B"]) if slots is None else slots.numpy()
    sel = list(batch)
    return R.gdn_decode(inp["q"][sel], inp["k"][sel], inp["v"][sel], inp["a"][sel],
                        inp["b"][sel], inp["A_log"], inp["dt_bias"],
                        inp["state"][torch.as_tensor(np.asarray(slots)[sel])], None,
                        scale=inp["scale"], **kw)


@pytest.mark.parametrize("T", [1, 2, 3, 4])
def test_small_batch(T):
    inp = synth.decode_inputs(300 + T, 6, T, 2, 4, 128, 128)
    o, st32, _ = run_gpu(inp)
    assert gdn_check_device_error() == Status.OK
    o_ref, st_ref = oracle_for(inp, range(6))
    assert_close(o, o_ref, TOL_BF16, "o")
    assert_close(st32, st_ref, TOL_BF16, "state")


@pytest.mark.parametrize("T", [2, 4])
def test_permuted_slots_pool_larger_than_batch(T):
    slots = [5, 0, 3]
    inp = synth.decode_inputs(311, 3, T, 1, 2, 128, 128, pool=7, slots=slots)
    o, st32, pool = run_gpu(inp)
    assert gdn_check_device_error() == Status.OK
    o_ref, st_ref = oracle_for(inp, range(3))
    assert_close(o, o_ref, TOL_BF16, "o")
    assert_close(st32, st_ref, TOL_BF16, "state")
    untouched = [1, 2, 4, 6]
    assert torch.equal(pool[untouched].cpu(), inp["state"][untouched])


def test_without_l2norm_and_custom_gate_params():
    inp = synth.decode_inputs(312, 4, 3, 2, 2, 128, 128)
    inp["q"] = (inp["q"].float() * 0.05).bfloat16()
    inp["k"] = (inp["k"].float() * 0.05).bfloat16()
    kw = dict(use_qk_l2norm=False, softplus_beta=2.0, softplus_threshold=1.0)
    o, st32, _ = run_gpu(inp, **kw)
    o_ref, st_ref = oracle_for(inp, range(4), use_qk_l2norm=False, softplus_beta=2.0,
                               softplus_threshold=1.0)
    assert_close(o, o_ref, TOL_BF16, "o")
    assert_close(st32, st_ref, TOL_BF16, "state")


@pytest.mark.parametrize("T", [1, 3, 4])
def test_bad_slot_is_reported_and_skipped(T):
    inp = synth.decode_inputs(313, 3, T, 1, 1, 128, 128, pool=3, slots=[0, 9, 2])
    o, st32, pool = run_gpu(inp)
    assert gdn_check_device_error() == Status.BAD_SLOT
    assert torch.count_nonzero(o[1]).item() == 0
    o_ref, st_ref = oracle_for(dict(inp, slot_indices=torch.tensor([0, 0, 2], dtype=torch.int32)),
                               [0, 2])
    assert_close(o[[0, 2]], o_ref, TOL_BF16, "o")
    assert_close(st32[[0, 2]], st_ref, TOL_BF16, "state")
    assert torch.equal(pool[1].cpu(), inp["state"][1])


def test_chained_single_token_calls():
    """Four one-token calls through the bf16 pool against the oracle chained the
    same way (its state rounded to bf16 between calls, as the pool stores it).
    Outputs are taken in fp32, and the last call's updated states too."""
    inp = synth.decode_inputs(314, 4, 4, 2, 4, 128, 128)
    d = to_dev(inp)
    st = d["state"].clone()
    st32 = torch.empty((4, 4, 128, 128), device="cuda")
    outs = []
    for t in range(4):
        sl = slice(t, t + 1)
        outs.append(gdn_decode(d["q"][:, sl].contiguous(), d["k"][:, sl].contiguous(),
                               d["v"][:, sl].contiguous(), d["a"][:, sl].contiguous(),
                               d["b"][:, sl].contiguous(), d["A_log"], d["dt_bias"], st,
                               out_dtype=torch.float32,
                               new_state_f32=st32 if t == 3 else None))
    ref_state = inp["state"].clone()
    ref_outs = []
    for t in range(4):
        sl = slice(t, t + 1)
        o_t, ns = R.gdn_decode(inp["q"][:, sl], inp["k"][:, sl], inp["v"][:, sl], inp["a"][:, sl],
                               inp["b"][:, sl], inp["A_log"], inp["dt_bias"], ref_state, None,
                               scale=inp["scale"])
        ref_outs.append(o_t)
        ref_state = torch.from_numpy(ns).to(torch.bfloat16)
    assert gdn_check_device_error() == Status.OK
    assert_close(torch.cat(outs, dim=1), np.concatenate(ref_outs, axis=1), TOL_BF16, "chained o")
    assert_close(st32, ns, TOL_BF16, "chained state")
    assert torch.equal(st, st32.to(torch.bfloat16))


@pytest.mark.parametrize("T", [1, 2, 3, 4])
def test_decode_workload_all_entries(T):
    """B=pool=256, H=16, HV=32, K=V=128: all 8192 (batch entry, value head) states."""
    inp = synth.decode(T)
    o, st32, _ = run_gpu(inp)
    assert gdn_check_device_error() == Status.OK
    o_ref, st_ref = decode_all_entries(inp)
    assert_close(o, o_ref, TOL_BF16, "o")
    assert_close(st32, st_ref, TOL_BF16, "state")


@pytest.mark.parametrize("T", [2, 4])
def test_strong_decay(T):
    """Gates from e^-3 down to exact fp32 zero: the kernel keeps the state as a
    running scale times the registers and folds the scale back in before it
    underflows; both branches must agree with the oracle."""
    inp = synth.decode_inputs(315 + T, 5, T, 2, 4, 128, 128)
    inp["A_log"] = torch.tensor([5.0, 4.0, 3.0, 0.0], dtype=torch.float32)
    inp["dt_bias"] = torch.tensor([1.0, 1.0, 0.5, 0.0], dtype=torch.float32)
    o, st32, _ = run_gpu(inp)
    assert gdn_check_device_error() == Status.OK
    o_ref, st_ref = oracle_for(inp, range(5))
    assert_close(o, o_ref, TOL_BF16, "o")
    assert_close(st32, st_ref, TOL_BF16, "state")
