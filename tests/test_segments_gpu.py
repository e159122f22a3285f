"""The segment-parallel state pass (`segments`) on the tensor-core path.

Every sequence is cut into S runs of equal chunk counts that are processed at
once (from zero and on the identity, giving each run's affine map), combined
in order and run again from their true starts.  The results must meet the
bound against the oracle and agree with the one-chain-per-sequence pass.
"""
import numpy as np
import pytest
import torch

from gated_delta_rule_kk_gb300 import Status, gdn_check_device_error, gdn_chunk_fwd, kda_chunk_fwd
from gated_delta_rule_kk_gb300 import synth
from oracle import recurrence as R

from _util import TOL_BF16, assert_close, to_dev

pytestmark = pytest.mark.gpu


def _run(fn, d, segments, **kw):
    o, ht = fn(d["q"], d["k"], d["v"], d["g"], d["beta"], scale=d["scale"],
               initial_state=d["h0"], cu_seqlens=d["cu_seqlens"], g_is_cumsum=d["g_is_cumsum"],
               out_dtype=torch.float32, segments=segments, **kw)
    assert gdn_check_device_error() == Status.OK
    return o, ht


@pytest.mark.parametrize("segments", [2, 3, 5, 16])
def test_gdn_segments_match_oracle_and_one_chain(segments):
    # 16 chunks (the last one ragged) per sequence, two sequences, grouped heads
    inp = synth.prefill_inputs(120 + segments, 2, 1000, 2, 1, 128, 128, h0_std=0.1)
    d = to_dev(inp)
    o, ht = _run(gdn_chunk_fwd, d, segments)
    o1, ht1 = _run(gdn_chunk_fwd, d, 1)
    o_ref, ht_ref = R.gdn_recurrent(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                                    scale=inp["scale"], h0=inp["h0"])
    assert_close(o, o_ref, TOL_BF16, f"o ({segments} segments)")
    assert_close(ht, ht_ref, TOL_BF16, f"ht ({segments} segments)")
    assert_close(o, o1.cpu().double().numpy(), TOL_BF16, "o vs one chain")


def test_gdn_segments_long_memory():
    """Gates near zero keep the state for the whole sequence, so every
    segment's map and the combine carry it: T = 2048 in 8 segments."""
    inp = synth.prefill_inputs(130, 1, 2048, 1, 1, 128, 128, h0_std=0.1)
    inp["g"] = torch.full(inp["g"].shape, -0.002)
    d = to_dev(inp)
    o, ht = _run(gdn_chunk_fwd, d, 8)
    o_ref, ht_ref = R.gdn_recurrent(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                                    scale=inp["scale"], h0=inp["h0"])
    assert_close(o, o_ref, TOL_BF16, "o")
    assert_close(ht, ht_ref, TOL_BF16, "ht")


def test_gdn_segments_packed_sequences_with_empty_and_short_ones():
    lengths = [70, 0, 400, 1, 700, 130]
    inp = synth.prefill_inputs(131, 1, sum(lengths), 4, 2, 128, 64, lengths=lengths)
    inp["h0"] = 0.1 * torch.randn(len(lengths), 4, 128, 64, generator=torch.Generator().manual_seed(9))
    d = to_dev(inp)
    o, ht = _run(gdn_chunk_fwd, d, 4)
    o_ref, ht_ref = R.gdn_recurrent(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                                    scale=inp["scale"], h0=inp["h0"], cu_seqlens=inp["cu_seqlens"])
    assert_close(o, o_ref, TOL_BF16, "o")
    assert_close(ht, ht_ref, TOL_BF16, "ht")
    for n in (i for i, x in enumerate(lengths) if x == 0):
        assert torch.equal(ht[n].cpu(), inp["h0"][n])


def test_kda_segments():
    inp = synth.prefill_inputs(132, 1, 900, 2, 2, 128, 128, h0_std=0.1, per_channel=True)
    d = to_dev(inp)
    o, ht = _run(kda_chunk_fwd, d, 4)
    o_ref, ht_ref = R.kda_recurrent(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                                    scale=inp["scale"], h0=inp["h0"])
    assert_close(o, o_ref, TOL_BF16, "o")
    assert_close(ht, ht_ref, TOL_BF16, "ht")


def test_segments_with_state_v_first():
    inp = synth.prefill_inputs(133, 1, 700, 2, 2, 128, 96, h0_std=0.1)
    d = to_dev(inp)
    o1, ht1 = _run(gdn_chunk_fwd, d, 3)
    d2 = dict(d, h0=d["h0"].transpose(-1, -2).contiguous())
    o2, ht2 = _run(gdn_chunk_fwd, d2, 3, state_v_first=True)
    assert torch.equal(o1, o2)
    assert torch.equal(ht2, ht1.transpose(-1, -2))


def test_automatic_choice_on_few_long_chains():
    """One sequence and one head (4 chains of 32 columns) of 64 chunks: the
    library takes the segment-parallel pass by itself."""
    inp = synth.prefill_inputs(134, 1, 4096, 1, 1, 128, 128, h0_std=0.1)
    d = to_dev(inp)
    o, ht = _run(gdn_chunk_fwd, d, 0)
    o1, ht1 = _run(gdn_chunk_fwd, d, 1)
    o_ref, ht_ref = R.gdn_recurrent(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                                    scale=inp["scale"], h0=inp["h0"])
    assert_close(o, o_ref, TOL_BF16, "o")
    assert_close(ht, ht_ref, TOL_BF16, "ht")
    assert not torch.equal(o, o1)  # a different summation order: it did take the segments
