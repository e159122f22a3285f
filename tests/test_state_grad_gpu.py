"""gdn_chunk_state_bwd (backward state pass, the dh recurrence) against the oracle.

Every gate kind on fp32 and bf16 inputs with ragged tails and a partial value
tile, grouped query heads sharing a gate head, packed sequences with empty
ones, bf16 chunk gradients, the default and an explicit scale, an empty
batch, and the benchmarked shape on sampled chains.  Like the forward pass the kernel computes in fp32 from the inputs as
stored, so the fp32 bound (1e-4 RMS) applies to both input dtypes.
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


def run(inp, states_dtype=torch.float32, output_states=True, scale="inp", split_size=None):
    dh, dh0 = gdn.gdn_chunk_state_bwd(
        inp["q"].cuda(), inp["do"].cuda(), gate=inp["gate"], gate_values=_dev(inp["gate_values"]),
        dht=_dev(inp["dht"]), cu_seqlens=_dev(inp["cu_seqlens"]),
        scale=inp["scale"] if scale == "inp" else scale, states_dtype=states_dtype,
        output_states=output_states, split_size=split_size)
    torch.cuda.synchronize()
    assert gdn.gdn_check_device_error() == Status.OK
    return dh, dh0


def oracle(inp, scale="inp", split_size=None):
    return SP.chunk_state_grad(inp["q"], inp["do"], inp["gate"], inp["gate_values"],
                               dht=inp["dht"], cu_seqlens=inp["cu_seqlens"],
                               scale=inp["scale"] if scale == "inp" else scale,
                               split_size=split_size)


@pytest.mark.parametrize("gate", GATES)
def test_fp32_every_gate(gate):
    # T = 150: two full chunks and a 22-token tail; V = 48: one full and one half tile
    inp = synth.state_grad_inputs(80, 2, 150, 3, 3, 32, 48, gate, dtype=torch.float32,
                                  dht_std=0.3)
    dh, dh0 = run(inp)
    dh_ref, dh0_ref = oracle(inp)
    assert tuple(dh.shape) == dh_ref.shape
    assert_close(dh, dh_ref, TOL_F32, f"dh ({gate})")
    assert_close(dh0, dh0_ref, TOL_F32, f"dh0 ({gate})")


@pytest.mark.parametrize("gate", GATES)
def test_bf16_inputs_full_width_grouped_heads(gate):
    # K = 128 bf16 takes the tensor-core kernel; 4 query heads over 2 gate heads
    inp = synth.state_grad_inputs(81, 1, 300, 4, 2, 128, 128, gate, dht_std=0.1)
    dh, dh0 = run(inp)
    dh_ref, dh0_ref = oracle(inp)
    assert_close(dh, dh_ref, TOL_F32, f"dh ({gate})")
    assert_close(dh0, dh0_ref, TOL_F32, f"dh0 ({gate})")


def test_fp32_grouped_heads_and_default_scale():
    inp = synth.state_grad_inputs(82, 2, 100, 6, 2, 64, 32, "gk", dtype=torch.float32,
                                  dht_std=0.2)
    dh, dh0 = run(inp, scale=None)
    dh_ref, dh0_ref = oracle(inp, scale=None)
    assert_close(dh, dh_ref, TOL_F32, "dh")
    assert_close(dh0, dh0_ref, TOL_F32, "dh0")
    dh2, _ = run(inp, scale=0.37)
    dh2_ref, _ = oracle(inp, scale=0.37)
    assert_close(dh2, dh2_ref, TOL_F32, "dh (scale 0.37)")


@pytest.mark.parametrize("gate", ["g_gamma", "gk"])
def test_tensor_core_path_partial_tile_and_bf16_gradients(gate):
    # K = 128 bf16 (tensor-core kernel), V = 48, T = 190, 6 query heads over 3
    # gate heads, chunk gradients in bf16
    inp = synth.state_grad_inputs(86, 2, 190, 6, 3, 128, 48, gate, dht_std=0.2)
    dh, dh0 = run(inp, states_dtype=torch.bfloat16)
    dh_ref, dh0_ref = oracle(inp)
    assert dh.dtype == torch.bfloat16
    # bf16 chunk gradients: bit for bit the RNE of the fp32 ones of the same call
    dh32, _ = run(inp)
    assert torch.equal(dh, dh32.to(torch.bfloat16))
    assert_close(dh32, dh_ref, TOL_F32, f"dh fp32 ({gate})")
    assert_close(dh, dh_ref, TOL_BF16, f"dh bf16 ({gate})")
    assert_close(dh0, dh0_ref, TOL_F32, f"dh0 ({gate})")


def test_bf16_chunk_gradients_and_no_chunk_output():
    inp = synth.state_grad_inputs(83, 2, 200, 2, 2, 64, 64, "g", dht_std=0.2)
    dh, dh0 = run(inp, states_dtype=torch.bfloat16)
    dh_ref, dh0_ref = oracle(inp)
    assert dh.dtype == torch.bfloat16
    dh32, _ = run(inp)
    assert torch.equal(dh, dh32.to(torch.bfloat16))
    assert_close(dh32, dh_ref, TOL_F32, "dh (fp32)")
    assert_close(dh, dh_ref, TOL_BF16, "dh (bf16)")
    assert_close(dh0, dh0_ref, TOL_F32, "dh0")
    none, dh0b = run(inp, output_states=False)
    assert none is None
    assert torch.equal(dh0b, dh0)


@pytest.mark.parametrize("K,dtype", [(32, torch.float32), (128, torch.bfloat16)])
def test_packed_sequences_with_empty_ones(K, dtype):
    lengths = [70, 0, 130, 1, 64]
    inp = synth.state_grad_inputs(84, 1, sum(lengths), 4, 2, K, 32, "gv", dtype=dtype,
                                  lengths=lengths, dht_std=0.5)
    dh, dh0 = run(inp)
    dh_ref, dh0_ref = oracle(inp)
    assert dh.shape[0] == 2 + 0 + 3 + 1 + 1
    assert_close(dh, dh_ref, TOL_F32, "dh")
    assert_close(dh0, dh0_ref, TOL_F32, "dh0")
    assert torch.equal(dh0[1].cpu(), inp["dht"][1])  # the empty sequence passes dht through


@pytest.mark.parametrize("gate", ["gk", "g"])
def test_tensor_core_path_packed_sequences(gate):
    """bf16 with K = 128 (the tcgen05 kernel, run backwards), packed sequences
    with empty ones and grouped query heads."""
    lengths = [70, 0, 130, 1, 64]
    inp = synth.state_grad_inputs(86, 1, sum(lengths), 4, 2, 128, 64, gate, lengths=lengths,
                                  dht_std=0.3)
    dh, dh0 = run(inp)
    dh_ref, dh0_ref = oracle(inp)
    assert_close(dh, dh_ref, TOL_F32, f"dh ({gate})")
    assert_close(dh0, dh0_ref, TOL_F32, f"dh0 ({gate})")
    assert torch.equal(dh0[1].cpu(), inp["dht"][1])


@pytest.mark.parametrize("factor", [40.0, -0.5])
def test_tensor_core_path_strong_and_positive_gk(factor):
    """The chunk-local cumulative per-key gates scaled by 40 (factors far below
    fp32's range inside a chunk) and by -0.5 (factors above one)."""
    inp = synth.state_grad_inputs(87, 2, 150, 2, 2, 128, 64, "gk", dht_std=0.3)
    inp["gate_values"] = inp["gate_values"] * factor
    dh, dh0 = run(inp)
    dh_ref, dh0_ref = oracle(inp)
    assert_close(dh, dh_ref, TOL_F32, f"dh (gk, x{factor})")
    assert_close(dh0, dh0_ref, TOL_F32, f"dh0 (gk, x{factor})")


@pytest.mark.parametrize("V", [32, 96])
@pytest.mark.parametrize("gate", ["g", "gk", "gv"])
def test_tensor_core_path_one_and_three_value_tiles(gate, V):
    """The tcgen05 kernel run backwards at V = 32 and 96 (one and three value
    tiles), grouped query heads."""
    inp = synth.state_grad_inputs(88, 2, 150, 4, 2, 128, V, gate, dht_std=0.3)
    dh, dh0 = run(inp)
    dh_ref, dh0_ref = oracle(inp)
    assert_close(dh, dh_ref, TOL_F32, f"dh ({gate}, V={V})")
    assert_close(dh0, dh0_ref, TOL_F32, f"dh0 ({gate}, V={V})")


def test_empty_batch_returns_dht():
    inp = synth.state_grad_inputs(85, 2, 0, 2, 2, 32, 32, "g", dtype=torch.float32, dht_std=1.0)
    dh, dh0 = run(inp)
    assert dh.shape[0] == 0
    assert torch.equal(dh0.cpu(), inp["dht"])


@pytest.mark.parametrize("gate", ["g", "gk", "gv"])
def test_benchmark_workload_sampled(gate):
    # the benchmarked shape and launch (B=2, T=4096, HQ=H=16, K=V=128, bf16,
    # fp32 chunk gradients); the oracle runs three sampled (sequence, head) chains
    inp = synth.state_grad_inputs(6, 2, 4096, 16, 16, 128, 128, gate, dht_std=0.1)
    dh, dh0 = run(inp)
    nt = 4096 // 64
    for b, h in ((0, 0), (1, 7), (1, 15)):
        one = {"q": inp["q"][b:b + 1, :, h:h + 1], "do": inp["do"][b:b + 1, :, h:h + 1],
               "gate": gate, "gate_values": inp["gate_values"][b:b + 1, :, h:h + 1],
               "dht": inp["dht"][b:b + 1, h:h + 1],
               "cu_seqlens": None, "scale": inp["scale"]}
        dh_ref, dh0_ref = oracle(one)
        what = f"({gate}) seq {b} head {h}"
        assert_close(dh[b * nt:(b + 1) * nt, h], dh_ref[:, 0], TOL_F32, f"dh {what}")
        assert_close(dh0[b, h], dh0_ref[0, 0], TOL_F32, f"dh0 {what}")


@pytest.mark.parametrize("T", [1, 64, 65])
@pytest.mark.parametrize("gate", ["g", "gk"])
def test_tensor_core_path_chunk_boundaries(T, gate):
    inp = synth.state_grad_inputs(87, 2, T, 2, 2, 128, 64, gate, dht_std=0.3)
    dh, dh0 = run(inp)
    dh_ref, dh0_ref = oracle(inp)
    assert tuple(dh.shape) == dh_ref.shape
    assert_close(dh, dh_ref, TOL_F32, f"dh ({gate}, T={T})")
    assert_close(dh0, dh0_ref, TOL_F32, f"dh0 ({gate}, T={T})")


@pytest.mark.parametrize("split", [128, 192])
@pytest.mark.parametrize("K,dtype", [(128, torch.bfloat16), (32, torch.float32)])
def test_split_size(split, K, dtype):
    inp = synth.state_grad_inputs(88, 2, 333, 2, 2, K, 64, "gk", dtype=dtype, dht_std=0.3)
    dh, dh0 = run(inp, split_size=split)
    dh_ref, dh0_ref = oracle(inp, split_size=split)
    assert tuple(dh.shape) == dh_ref.shape
    assert_close(dh, dh_ref, TOL_F32, f"dh (split {split})")
    assert_close(dh0, dh0_ref, TOL_F32, f"dh0 (split {split})")
    lengths = [200, 0, 64, 260]
    inp = synth.state_grad_inputs(89, 1, sum(lengths), 2, 2, K, 64, "g", dtype=dtype,
                                  lengths=lengths, dht_std=0.3)
    dh, dh0 = run(inp, split_size=split)
    dh_ref, dh0_ref = oracle(inp, split_size=split)
    assert tuple(dh.shape) == dh_ref.shape
    assert_close(dh, dh_ref, TOL_F32, f"dh packed (split {split})")
    assert_close(dh0, dh0_ref, TOL_F32, f"dh0 packed (split {split})")


@pytest.mark.parametrize("K,dtype", [(128, torch.bfloat16), (32, torch.float32)])
def test_state_v_first(K, dtype):
    inp = synth.state_grad_inputs(90, 2, 200, 4, 2, K, 48, "gv", dtype=dtype, dht_std=0.3)
    dh_ref, dh0_ref = oracle(inp)
    dh, dh0 = gdn.gdn_chunk_state_bwd(
        inp["q"].cuda(), inp["do"].cuda(), gate="gv", gate_values=inp["gate_values"].cuda(),
        dht=inp["dht"].transpose(-1, -2).contiguous().cuda(), scale=inp["scale"],
        state_v_first=True)
    torch.cuda.synchronize()
    assert gdn.gdn_check_device_error() == Status.OK
    assert tuple(dh.shape) == (8, 4, 48, K)
    assert_close(dh, dh_ref.swapaxes(-1, -2), TOL_F32, "dh [V, K]")
    assert_close(dh0, dh0_ref.swapaxes(-1, -2), TOL_F32, "dh0 [V, K]")
