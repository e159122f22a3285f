"""gdn_chunk_state_fwd (gated linear-attention chunk state pass) against the oracle.

Every gate kind on fp32 and bf16 inputs, ragged tails and a partial value
tile, packed sequences with empty ones, bf16 chunk states, no outputs but the
final state, an empty batch, a bad cu_seqlens reported on the device, and the
benchmarked shape on sampled chains.
The kernel computes in fp32 from the inputs as stored, so the fp32 bound
(1e-4 RMS) applies to both input dtypes.  Chunk states requested in bf16 are
checked twice: bit for bit as the round-to-nearest-even of the fp32 states of
the same call made with fp32 states (which meet the fp32 bound), and raw
against the bf16 bound.
"""
import pytest
import torch

import gated_delta_rule_kk_gb300 as gdn
from gated_delta_rule_kk_gb300 import Status, synth
from oracle import state_pass as SP

from _util import TOL_BF16, TOL_F32, assert_close

pytestmark = pytest.mark.gpu

GATES = [None, "g", "g_gamma", "gk", "gv"]


def _dev(x):
    return None if x is None else x.cuda()


def run(inp, states_dtype=torch.float32, output_states=True, split_size=None):
    hs, ht = gdn.gdn_chunk_state_fwd(
        inp["k"].cuda(), inp["v"].cuda(), gate=inp["gate"], gate_values=_dev(inp["gate_values"]),
        initial_state=_dev(inp["h0"]), cu_seqlens=_dev(inp["cu_seqlens"]),
        states_dtype=states_dtype, output_states=output_states, split_size=split_size)
    torch.cuda.synchronize()
    assert gdn.gdn_check_device_error() == Status.OK
    return hs, ht


def oracle(inp, split_size=None):
    return SP.chunk_state_pass(inp["k"], inp["v"], inp["gate"], inp["gate_values"], h0=inp["h0"],
                               cu_seqlens=inp["cu_seqlens"], split_size=split_size)


@pytest.mark.parametrize("gate", GATES)
def test_fp32_every_gate(gate):
    # T = 150: two full chunks and a 22-token tail; V = 48: one full and one half tile
    inp = synth.state_pass_inputs(70, 2, 150, 3, 32, 48, gate, dtype=torch.float32, h0_std=0.3)
    hs, ht = run(inp)
    hs_ref, ht_ref = oracle(inp)
    assert tuple(hs.shape) == hs_ref.shape
    assert_close(hs, hs_ref, TOL_F32, f"hs ({gate})")
    assert_close(ht, ht_ref, TOL_F32, f"ht ({gate})")


@pytest.mark.parametrize("gate", GATES)
def test_bf16_inputs_full_width(gate):
    inp = synth.state_pass_inputs(71, 1, 300, 2, 128, 128, gate, h0_std=0.1)
    hs, ht = run(inp)
    hs_ref, ht_ref = oracle(inp)
    assert_close(hs, hs_ref, TOL_F32, f"hs ({gate})")
    assert_close(ht, ht_ref, TOL_F32, f"ht ({gate})")


@pytest.mark.parametrize("gate", ["g", "gk", "gv"])
def test_tensor_core_path_partial_tile_and_bf16_states(gate):
    # K = 128 bf16 (tensor-core kernel), V = 48: one full and one half 32-column
    # tile; T = 190: two full chunks and a 62-token tail; chunk states in bf16
    inp = synth.state_pass_inputs(75, 2, 190, 3, 128, 48, gate, h0_std=0.2)
    hs, ht = run(inp, states_dtype=torch.bfloat16)
    hs_ref, ht_ref = oracle(inp)
    assert hs.dtype == torch.bfloat16
    hs32, ht32 = run(inp)
    assert torch.equal(hs, hs32.to(torch.bfloat16)), "bf16 states are not the RNE of fp32 ones"
    assert torch.equal(ht32, ht)
    assert_close(hs32, hs_ref, TOL_F32, f"hs fp32 ({gate})")
    assert_close(ht, ht_ref, TOL_F32, f"ht ({gate})")
    assert_close(hs, hs_ref, TOL_BF16, f"hs bf16 ({gate})")


def test_bf16_chunk_states_and_no_states():
    inp = synth.state_pass_inputs(72, 2, 200, 2, 64, 64, "g", h0_std=0.2)
    hs, ht = run(inp, states_dtype=torch.bfloat16)
    hs_ref, ht_ref = oracle(inp)
    assert hs.dtype == torch.bfloat16
    hs32, _ = run(inp)
    assert torch.equal(hs, hs32.to(torch.bfloat16))
    assert_close(hs32, hs_ref, TOL_F32, "hs (fp32)")
    assert_close(hs, hs_ref, TOL_BF16, "hs (bf16)")
    assert_close(ht, ht_ref, TOL_F32, "ht")
    none, ht2 = run(inp, output_states=False)
    assert none is None
    assert torch.equal(ht2, ht)


def test_packed_sequences_with_empty_ones():
    lengths = [70, 0, 130, 1, 64]
    inp = synth.state_pass_inputs(73, 1, sum(lengths), 2, 32, 32, "gk", dtype=torch.float32,
                                  lengths=lengths, h0_std=0.5)
    hs, ht = run(inp)
    hs_ref, ht_ref = oracle(inp)
    assert hs.shape[0] == 2 + 0 + 3 + 1 + 1
    assert_close(hs, hs_ref, TOL_F32, "hs")
    assert_close(ht, ht_ref, TOL_F32, "ht")
    assert torch.equal(ht[1].cpu(), inp["h0"][1])  # the empty sequence keeps its state


@pytest.mark.parametrize("gate", ["g", "gk", "gv"])
def test_tensor_core_path_packed_sequences(gate):
    """bf16 with K = 128 (the tcgen05 kernel), packed sequences with empty
    ones: the TMA tiles of a sequence's last chunk hold the next sequence's
    rows, which must take no part."""
    lengths = [70, 0, 130, 1, 64]
    inp = synth.state_pass_inputs(80, 1, sum(lengths), 2, 128, 64, gate, lengths=lengths,
                                  h0_std=0.3)
    hs, ht = run(inp)
    hs_ref, ht_ref = oracle(inp)
    assert hs.shape[0] == 2 + 0 + 3 + 1 + 1
    assert_close(hs, hs_ref, TOL_F32, f"hs ({gate})")
    assert_close(ht, ht_ref, TOL_F32, f"ht ({gate})")
    assert torch.equal(ht[1].cpu(), inp["h0"][1])


@pytest.mark.parametrize("factor", [40.0, -0.5])
@pytest.mark.parametrize("gate", ["gk", "gv", "g"])
def test_tensor_core_path_strong_and_positive_gates(gate, factor):
    """The chunk-local cumulative gates scaled: by 40 (about -2 per token, so
    the in-chunk factors span e^0 .. far below fp32's range) and by -0.5
    (growing states, factors above one)."""
    inp = synth.state_pass_inputs(81, 2, 150, 2, 128, 64, gate, h0_std=0.3)
    inp["gate_values"] = inp["gate_values"] * factor
    hs, ht = run(inp)
    hs_ref, ht_ref = oracle(inp)
    assert_close(hs, hs_ref, TOL_F32, f"hs ({gate}, x{factor})")
    assert_close(ht, ht_ref, TOL_F32, f"ht ({gate}, x{factor})")


@pytest.mark.parametrize("V", [32, 96])
@pytest.mark.parametrize("gate", ["g", "g_gamma", "gk", "gv", None])
def test_tensor_core_path_one_and_three_value_tiles(gate, V):
    """bf16 with K = 128 (the tcgen05 kernel) at V = 32 and 96: one and three
    32-column value tiles per head; T = 150 leaves a 22-token tail."""
    inp = synth.state_pass_inputs(82, 2, 150, 2, 128, V, gate, h0_std=0.3)
    hs, ht = run(inp)
    hs_ref, ht_ref = oracle(inp)
    assert_close(hs, hs_ref, TOL_F32, f"hs ({gate}, V={V})")
    assert_close(ht, ht_ref, TOL_F32, f"ht ({gate}, V={V})")


def test_empty_batch_returns_the_initial_state():
    inp = synth.state_pass_inputs(74, 2, 0, 2, 32, 32, "g", dtype=torch.float32, h0_std=1.0)
    hs, ht = run(inp)
    assert hs.shape[0] == 0
    assert torch.equal(ht.cpu(), inp["h0"])


def test_bad_seqlens_is_reported():
    k = torch.randn(1, 100, 2, 32, device="cuda")
    v = torch.randn(1, 100, 2, 32, device="cuda")
    cu = torch.tensor([0, 60, 40, 100], dtype=torch.int32, device="cuda")
    gdn.gdn_chunk_state_fwd(k, v, cu_seqlens=cu, num_chunks=8)
    torch.cuda.synchronize()
    assert gdn.gdn_check_device_error() == Status.BAD_SEQLENS
    assert gdn.gdn_check_device_error() == Status.OK  # reading clears it


def _head_slice(inp, b, h):
    """The inputs of one (sequence, head) chain of a fixed-length batch."""
    gv = inp["gate_values"]
    if gv is not None:
        gv = gv[h:h + 1] if inp["gate"] == "g_gamma" else gv[b:b + 1, :, h:h + 1]
    return {"k": inp["k"][b:b + 1, :, h:h + 1], "v": inp["v"][b:b + 1, :, h:h + 1],
            "gate": inp["gate"], "gate_values": gv,
            "h0": None if inp["h0"] is None else inp["h0"][b:b + 1, h:h + 1],
            "cu_seqlens": None}


@pytest.mark.parametrize("gate", ["g", "gk", "gv"])
def test_benchmark_workload_sampled(gate):
    # the benchmarked shape and launch (B=2, T=4096, H=16, K=V=128, bf16, fp32
    # chunk states); the oracle runs three sampled (sequence, head) chains
    inp = synth.state_pass_inputs(5, 2, 4096, 16, 128, 128, gate, h0_std=0.1)
    hs, ht = run(inp)
    nt = 4096 // 64
    for b, h in ((0, 0), (1, 7), (1, 15)):
        hs_ref, ht_ref = oracle(_head_slice(inp, b, h))
        what = f"({gate}) seq {b} head {h}"
        assert_close(hs[b * nt:(b + 1) * nt, h], hs_ref[:, 0], TOL_F32, f"hs {what}")
        assert_close(ht[b, h], ht_ref[0, 0], TOL_F32, f"ht {what}")


@pytest.mark.parametrize("T", [1, 64, 65])
@pytest.mark.parametrize("gate", ["g", "gk"])
def test_tensor_core_path_chunk_boundaries(T, gate):
    # one token, exactly one chunk, one chunk and one token (both variants of
    # the tensor-core kernel: k from the ring, and k~ staged for gk)
    inp = synth.state_pass_inputs(76, 2, T, 2, 128, 64, gate, h0_std=0.3)
    hs, ht = run(inp)
    hs_ref, ht_ref = oracle(inp)
    assert tuple(hs.shape) == hs_ref.shape
    assert_close(hs, hs_ref, TOL_F32, f"hs ({gate}, T={T})")
    assert_close(ht, ht_ref, TOL_F32, f"ht ({gate}, T={T})")


@pytest.mark.parametrize("split", [128, 192])
@pytest.mark.parametrize("K,dtype", [(128, torch.bfloat16), (32, torch.float32)])
def test_split_size(split, K, dtype):
    # states stored every split / 64 chunks, fixed-length and packed sequences,
    # tensor-core (K = 128 bf16) and exact kernels
    inp = synth.state_pass_inputs(77, 2, 333, 2, K, 64, "g", dtype=dtype, h0_std=0.3)
    hs, ht = run(inp, split_size=split)
    hs_ref, ht_ref = oracle(inp, split_size=split)
    assert tuple(hs.shape) == hs_ref.shape
    assert_close(hs, hs_ref, TOL_F32, f"hs (split {split})")
    assert_close(ht, ht_ref, TOL_F32, f"ht (split {split})")
    lengths = [200, 0, 64, 260]
    inp = synth.state_pass_inputs(78, 1, sum(lengths), 2, K, 64, "gv", dtype=dtype,
                                  lengths=lengths, h0_std=0.3)
    hs, ht = run(inp, split_size=split)
    hs_ref, ht_ref = oracle(inp, split_size=split)
    assert tuple(hs.shape) == hs_ref.shape
    assert_close(hs, hs_ref, TOL_F32, f"hs packed (split {split})")
    assert_close(ht, ht_ref, TOL_F32, f"ht packed (split {split})")


@pytest.mark.parametrize("K,dtype,states_dtype", [(128, torch.bfloat16, torch.float32),
                                                  (128, torch.bfloat16, torch.bfloat16),
                                                  (32, torch.float32, torch.float32)])
def test_state_v_first(K, dtype, states_dtype):
    # every state [V, K]: h0 in, hs and ht out (a partial value tile, a split)
    inp = synth.state_pass_inputs(79, 2, 200, 2, K, 48, "gk", dtype=dtype, h0_std=0.3)
    hs_ref, ht_ref = oracle(inp, split_size=128)
    hs, ht = gdn.gdn_chunk_state_fwd(
        inp["k"].cuda(), inp["v"].cuda(), gate="gk", gate_values=inp["gate_values"].cuda(),
        initial_state=inp["h0"].transpose(-1, -2).contiguous().cuda(), split_size=128,
        states_dtype=states_dtype, state_v_first=True)
    torch.cuda.synchronize()
    assert gdn.gdn_check_device_error() == Status.OK
    assert tuple(hs.shape) == (4, 2, 48, K) and tuple(ht.shape) == (2, 2, 48, K)
    if states_dtype == torch.bfloat16:
        hs32, _ = gdn.gdn_chunk_state_fwd(
            inp["k"].cuda(), inp["v"].cuda(), gate="gk", gate_values=inp["gate_values"].cuda(),
            initial_state=inp["h0"].transpose(-1, -2).contiguous().cuda(), split_size=128,
            state_v_first=True)
        assert torch.equal(hs, hs32.to(torch.bfloat16))
        assert_close(hs32, hs_ref.swapaxes(-1, -2), TOL_F32, "hs [V, K] fp32")
        assert_close(hs, hs_ref.swapaxes(-1, -2), TOL_BF16, "hs [V, K] bf16")
    else:
        assert_close(hs, hs_ref.swapaxes(-1, -2), TOL_F32, "hs [V, K]")
    assert_close(ht, ht_ref.swapaxes(-1, -2), TOL_F32, "ht [V, K]")
