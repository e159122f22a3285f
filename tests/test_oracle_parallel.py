"""The oracle's worker-pool runner returns exactly what the direct calls return."""
import numpy as np
import torch

from gated_delta_rule_kk_gb300 import synth
from oracle import recurrence as R

from _fullsize import decode_all_entries, prefill_all_chains


def test_prefill_chains_on_workers_equal_the_direct_call():
    lengths = [70, 0, 130, 5]
    inp = synth.prefill_inputs(41, 1, sum(lengths), 4, 2, 8, 6, dtype=torch.bfloat16,
                               h0_std=0.1, lengths=lengths)
    o, ht = prefill_all_chains(inp, workers=3)
    o_ref, ht_ref = R.gdn_recurrent(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                                    scale=inp["scale"], h0=inp["h0"], cu_seqlens=inp["cu_seqlens"])
    np.testing.assert_array_equal(o, o_ref)
    np.testing.assert_array_equal(ht, ht_ref)
    kin = synth.prefill_inputs(42, 2, 100, 2, 1, 8, 4, dtype=torch.float32, per_channel=True)
    o, ht = prefill_all_chains(kin, kda=True, workers=2)
    o_ref, ht_ref = R.kda_recurrent(kin["q"], kin["k"], kin["v"], kin["g"], kin["beta"],
                                    scale=kin["scale"], g_is_cumsum=True)
    np.testing.assert_array_equal(o, o_ref)
    np.testing.assert_array_equal(ht, ht_ref)


def test_decode_slices_on_workers_equal_the_direct_call():
    inp = synth.decode_inputs(43, 7, 3, 1, 2, 8, 8, pool=9, slots=[8, 0, 3, 1, 2, 5, 6])
    o, st = decode_all_entries(inp, slice_len=3, workers=2)
    o_ref, st_ref = R.gdn_decode(inp["q"], inp["k"], inp["v"], inp["a"], inp["b"], inp["A_log"],
                                 inp["dt_bias"], inp["state"], inp["slot_indices"],
                                 scale=inp["scale"])
    np.testing.assert_array_equal(o, o_ref)
    np.testing.assert_array_equal(st, st_ref)
