"""GDN chunked forward on the GPU against the fp64 oracle (through the C ABI)."""
import numpy as np
import pytest
import torch

from gated_delta_rule_kk_gb300 import Status, gdn_check_device_error, gdn_chunk_fwd
from gated_delta_rule_kk_gb300 import synth
from oracle import recurrence as R

from _util import TOL_BF16, TOL_F32, assert_close, to_dev

pytestmark = pytest.mark.gpu


def run_gpu(inp):
    d = to_dev(inp)
    o, ht = gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], scale=d["scale"],
                          initial_state=d["h0"], cu_seqlens=d["cu_seqlens"],
                          g_is_cumsum=d["g_is_cumsum"])
    assert gdn_check_device_error() == Status.OK
    return o, ht


def run_oracle(inp, heads=None, seqs=None):
    return R.gdn_recurrent(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                           scale=inp["scale"], h0=inp["h0"], cu_seqlens=inp["cu_seqlens"],
                           g_is_cumsum=inp["g_is_cumsum"], heads=heads, seqs=seqs)


def test_tiny_fp32_workload():
    inp = synth.tiny()
    o, ht = run_gpu(inp)
    o_ref, ht_ref = run_oracle(inp)
    assert_close(o, o_ref, TOL_F32, "o")
    assert_close(ht, ht_ref, TOL_F32, "ht")


@pytest.mark.parametrize("T,K,V,H,Hg,dtype,h0", [
    (200, 32, 48, 2, 1, torch.float32, True),     # ragged tail, V not a tile multiple
    (64, 64, 64, 1, 1, torch.float32, False),     # exactly one chunk
    (1, 128, 128, 2, 2, torch.bfloat16, True),    # a single token
    (333, 128, 128, 4, 2, torch.bfloat16, True),  # several chunks + tail, GQA
    (130, 100, 72, 3, 3, torch.float32, True),    # K not a multiple of 32
])
def test_small_shapes(T, K, V, H, Hg, dtype, h0):
    inp = synth.prefill_inputs(100 + T, 2, T, H, Hg, K, V, dtype=dtype,
                               h0_std=0.1 if h0 else None)
    o, ht = run_gpu(inp)
    o_ref, ht_ref = run_oracle(inp)
    tol = TOL_F32 if dtype == torch.float32 else TOL_BF16
    assert_close(o, o_ref, tol, "o")
    assert_close(ht, ht_ref, tol, "ht")


def test_cumsum_gate_input_matches_raw():
    inp = synth.prefill_inputs(7, 1, 150, 2, 2, 64, 64, dtype=torch.float32, h0_std=0.1)
    o1, ht1 = run_gpu(inp)
    g = inp["g"].clone()
    for c in range(0, 150, 64):
        g[:, c:c + 64] = torch.cumsum(inp["g"][:, c:c + 64].double(), dim=1).float()
    inp2 = dict(inp, g=g, g_is_cumsum=True)
    o2, ht2 = run_gpu(inp2)
    o_ref, ht_ref = run_oracle(inp2)
    assert_close(o2, o_ref, TOL_F32, "o (cumsum input)")
    assert_close(ht2, ht_ref, TOL_F32, "ht (cumsum input)")
    assert_close(o1, o2.cpu().double().numpy(), 1e-5, "raw vs cumsum gate input")


def test_varlen_with_empty_and_short_sequences():
    lengths = [0, 1, 63, 64, 65, 0, 130]
    T = sum(lengths)
    inp = synth.prefill_inputs(9, 1, T, 4, 2, 64, 32, dtype=torch.float32, h0_std=None,
                               lengths=lengths)
    # give every sequence its own initial state
    inp["h0"] = torch.randn(len(lengths), 4, 64, 32, generator=torch.Generator().manual_seed(3))
    o, ht = run_gpu(inp)
    o_ref, ht_ref = run_oracle(inp)
    assert_close(o, o_ref, TOL_F32, "o")
    assert_close(ht, ht_ref, TOL_F32, "ht")
    # empty sequences hand their initial state straight back
    assert torch.equal(ht[0].cpu(), inp["h0"][0])
    assert torch.equal(ht[5].cpu(), inp["h0"][5])


@pytest.mark.parametrize("lengths", [
    [70, 0, 300, 1, 129, 64, 65, 250],   # the chain takes them longest first
    [int(x) for x in np.random.default_rng(17).integers(0, 5, 1100)],  # past the ordering limit
], ids=["mixed", "1100_short"])
def test_varlen_tensor_core_path(lengths):
    T = sum(lengths)
    H, Hg, V = (4, 2, 64) if len(lengths) < 100 else (1, 1, 32)
    inp = synth.prefill_inputs(10, 1, T, H, Hg, 128, V, dtype=torch.bfloat16, h0_std=None,
                               lengths=lengths)
    inp["h0"] = 0.1 * torch.randn(len(lengths), H, 128, V, generator=torch.Generator().manual_seed(4))
    o, ht = run_gpu(inp)
    o_ref, ht_ref = run_oracle(inp)
    assert_close(o, o_ref, TOL_BF16, "o")
    assert_close(ht, ht_ref, TOL_BF16, "ht")
    for n in (i for i, x in enumerate(lengths) if x == 0):
        assert torch.equal(ht[n].cpu(), inp["h0"][n])


def test_no_final_state_and_deterministic():
    inp = synth.prefill_inputs(21, 1, 300, 2, 1, 128, 128, dtype=torch.bfloat16)
    d = to_dev(inp)
    o1, ht1 = gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], output_final_state=False)
    o2, _ = gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], output_final_state=False)
    assert ht1 is None
    assert torch.equal(o1, o2)


def test_bad_cu_seqlens_reported_on_device():
    inp = synth.prefill_inputs(5, 1, 100, 1, 1, 32, 32, dtype=torch.float32, lengths=[40, 60])
    d = to_dev(inp)
    bad = torch.tensor([0, 70, 50], dtype=torch.int32, device="cuda")  # decreasing
    gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], cu_seqlens=bad)
    assert gdn_check_device_error() == Status.BAD_SEQLENS
    assert gdn_check_device_error() == Status.OK  # reading clears it


# ---- the named workloads at full size, oracle on sampled chains -------------

def test_gdn_prefill_workload_sampled():
    inp = synth.gdn_prefill()
    o, ht = run_gpu(inp)
    for n, h in ((0, 0), (1, 9), (1, 15)):
        o_ref, ht_ref = run_oracle(inp, heads=[h], seqs=[n])
        assert_close(o[n, :, h], o_ref[n, :, h], TOL_BF16, f"o seq {n} head {h}")
        assert_close(ht[n, h], ht_ref[n, h], TOL_BF16, f"ht seq {n} head {h}")


def test_varlen_gqa_workload_sampled():
    inp = synth.varlen_gqa()
    o, ht = run_gpu(inp)
    cu = inp["cu_seqlens"].numpy()
    longest = int(np.argmax(np.diff(cu)))
    for n, h in ((longest, 5), (0, 0), (7, 15)):
        o_ref, ht_ref = run_oracle(inp, heads=[h], seqs=[n])
        s, e = cu[n], cu[n + 1]
        assert_close(o[0, s:e, h], o_ref[0, s:e, h], TOL_BF16, f"o seq {n} head {h}")
        assert_close(ht[n, h], ht_ref[n, h], TOL_BF16, f"ht seq {n} head {h}")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_zero_length_batch_returns_the_initial_state(dtype):
    # T = 0: no token is read or written (the empty tensors' pointers are NULL);
    # the final state is the initial state, or zeros without one
    import gated_delta_rule_kk_gb300 as gdn
    B, H, Hg, K, V = 3, 4, 2, 128, 128
    q = torch.empty((B, 0, Hg, K), dtype=dtype, device="cuda")
    v = torch.empty((B, 0, H, V), dtype=dtype, device="cuda")
    g = torch.empty((B, 0, H), dtype=torch.float32, device="cuda")
    h0 = torch.randn((B, H, K, V), generator=torch.Generator().manual_seed(5)).cuda()
    o, ht = gdn_chunk_fwd(q, q, v, g, g, initial_state=h0)
    torch.cuda.synchronize()
    assert gdn_check_device_error() == Status.OK
    assert tuple(o.shape) == (B, 0, H, V)
    assert torch.equal(ht, h0)
    _, ht0 = gdn_chunk_fwd(q, q, v, g, g)
    torch.cuda.synchronize()
    assert torch.equal(ht0, torch.zeros_like(h0))
    o_h, ht_h = gdn.gdn_chunk_fwd_host(q.cpu(), q.cpu(), v.cpu(), g.cpu(), g.cpu(),
                                       initial_state=h0.cpu())
    torch.cuda.synchronize()
    assert tuple(o_h.shape) == (B, 0, H, V)
    assert torch.equal(ht_h, h0.cpu())
