"""KDA (per-channel gate) chunked forward on the GPU against the fp64 oracle."""
import pytest
import torch

from gated_delta_rule_kk_gb300 import Status, gdn_check_device_error, gdn_chunk_fwd, kda_chunk_fwd
from gated_delta_rule_kk_gb300 import synth
from oracle import recurrence as R

from _fullsize import prefill_all_chains
from _util import TOL_BF16, TOL_F32, assert_close, to_dev

pytestmark = pytest.mark.gpu


def run_gpu(inp):
    """o in fp32 (the value the bound applies to) and ht; for bf16 inputs the
    default bf16 o must be that value rounded to nearest even, bit for bit."""
    d = to_dev(inp)
    kw = dict(scale=d["scale"], initial_state=d["h0"], cu_seqlens=d["cu_seqlens"],
              g_is_cumsum=d["g_is_cumsum"])
    o, ht = kda_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], out_dtype=torch.float32, **kw)
    if d["q"].dtype == torch.bfloat16:
        o16, ht16 = kda_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], **kw)
        assert torch.equal(o16, o.to(torch.bfloat16)), "bf16 o is not the RNE of the fp32 o"
        assert torch.equal(ht16, ht)
    assert gdn_check_device_error() == Status.OK
    return o, ht


def run_oracle(inp, heads=None, seqs=None):
    return R.kda_recurrent(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                           scale=inp["scale"], h0=inp["h0"], cu_seqlens=inp["cu_seqlens"],
                           g_is_cumsum=inp["g_is_cumsum"], heads=heads, seqs=seqs)


@pytest.mark.parametrize("T,K,V,H,HV,dtype,h0", [
    (150, 32, 32, 1, 2, torch.float32, True),     # tail, grouped value heads
    (64, 128, 64, 2, 2, torch.float32, False),
    (257, 128, 128, 2, 4, torch.bfloat16, True),
    (5, 48, 40, 1, 1, torch.float32, True),       # shorter than a sub-chunk
    (200, 128, 32, 1, 2, torch.bfloat16, True),   # tensor cores, one 32-column value tile
    (130, 128, 96, 2, 2, torch.bfloat16, False),  # tensor cores, three value tiles
])
def test_small_shapes(T, K, V, H, HV, dtype, h0):
    inp = synth.prefill_inputs(200 + T, 1, T, HV, H, K, V, dtype=dtype,
                               h0_std=0.1 if h0 else None, per_channel=True)
    o, ht = run_gpu(inp)
    o_ref, ht_ref = run_oracle(inp)
    tol = TOL_F32 if dtype == torch.float32 else TOL_BF16
    assert_close(o, o_ref, tol, "o")
    assert_close(ht, ht_ref, tol, "ht")


def test_raw_gate_input_and_varlen():
    lengths = [70, 0, 9, 128]
    T = sum(lengths)
    inp = synth.prefill_inputs(31, 1, T, 2, 2, 64, 64, dtype=torch.float32, h0_std=0.1,
                               lengths=lengths, per_channel=True)
    o, ht = run_gpu(inp)
    o_ref, ht_ref = run_oracle(inp)
    assert_close(o, o_ref, TOL_F32, "o")
    assert_close(ht, ht_ref, TOL_F32, "ht")
    # the same gates handed over raw (difference the chunk-local cumsum back)
    cu = inp["cu_seqlens"].tolist()
    g = inp["g"].double().clone()
    raw = g.clone()
    for n in range(len(lengths)):
        for t in range(cu[n], cu[n + 1]):
            if (t - cu[n]) % 64:
                raw[:, t] = g[:, t] - g[:, t - 1]
    inp2 = dict(inp, g=raw.float(), g_is_cumsum=False)
    o2, ht2 = run_gpu(inp2)
    o_ref2, ht_ref2 = run_oracle(inp2)
    assert_close(o2, o_ref2, TOL_F32, "o (raw gate)")
    assert_close(ht2, ht_ref2, TOL_F32, "ht (raw gate)")


def test_channel_constant_gate_equals_gdn():
    inp = synth.prefill_inputs(41, 1, 200, 2, 2, 64, 64, dtype=torch.float32, h0_std=0.1)
    d = to_dev(inp)
    o1, ht1 = gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], initial_state=d["h0"])
    gk = d["g"][..., None].expand(-1, -1, -1, 64).contiguous()
    o2, ht2 = kda_chunk_fwd(d["q"], d["k"], d["v"], gk, d["beta"], initial_state=d["h0"],
                            g_is_cumsum=False)
    assert_close(o2, o1.cpu().double().numpy(), 1e-5, "o")
    assert_close(ht2, ht1.cpu().double().numpy(), 1e-5, "ht")


def test_kda_prefill_workload_all_heads():
    """B=1, T=8192, H=HV=32, K=V=128, bf16, chunk-local cumsum gate: all 32 heads."""
    inp = synth.kda_prefill()
    o, ht = run_gpu(inp)
    o_ref, ht_ref = prefill_all_chains(inp, kda=True)
    assert_close(o, o_ref, TOL_BF16, "o")
    assert_close(ht, ht_ref, TOL_BF16, "ht")


# ---- per-channel gates the synthetic workload never reaches (tensor cores) --

def _raw_problem(seed, T=200):
    inp = synth.prefill_inputs(seed, 1, T, 2, 1, 128, 128, dtype=torch.bfloat16, h0_std=0.1,
                               per_channel=True)
    # hand the gates over raw so the edits below are per-token rates
    r = torch.Generator().manual_seed(seed)
    g = -torch.rand(inp["g"].shape, generator=r) * 0.05
    return dict(inp, g=g, g_is_cumsum=False)


def _check(inp):
    o, ht = run_gpu(inp)
    o_ref, ht_ref = run_oracle(inp)
    assert_close(o, o_ref, TOL_BF16, "o")
    assert_close(ht, ht_ref, TOL_BF16, "ht")


@pytest.mark.parametrize("gate_input", ["cumsum", "raw"])
def test_tensor_core_packed_sequences_many_chains(gate_input):
    """bf16, K = V = 128 (the tensor-core path) on packed sequences with an
    empty and a one-token one, 4 query/key heads for 16 value heads, an
    initial state, and more chain CTAs than SMs; the gate given as chunk-local
    cumsums (counted from each sequence start) or raw."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    lengths = [130, 0, 1, 64, 65, 200, 3, 90]
    H, HV, N = 4, 16, len(lengths)
    inp = synth.prefill_inputs(71, 1, sum(lengths), HV, H, 128, 128, dtype=torch.bfloat16,
                               lengths=lengths, per_channel=True)
    inp["h0"] = 0.1 * torch.randn(N, HV, 128, 128, generator=torch.Generator().manual_seed(72))
    if gate_input == "raw":
        r = torch.Generator().manual_seed(73)
        inp = dict(inp, g=-torch.rand(inp["g"].shape, generator=r) * 0.05, g_is_cumsum=False)
    assert 4 * HV * N > sms
    o, ht = run_gpu(inp)
    o_ref, ht_ref = run_oracle(inp)
    assert_close(o, o_ref, TOL_BF16, "o")
    assert_close(ht, ht_ref, TOL_BF16, "ht")
    # the empty sequence hands its initial state back unchanged
    assert torch.equal(ht[1].cpu(), inp["h0"][1])


def test_strong_channel_gates_take_the_exact_exponentials():
    """Channels 0..15 of head 0 fall below -80 inside chunk 1 (-2.5 per token):
    that chunk is gated with exact per-element exponentials."""
    inp = _raw_problem(61)
    g = inp["g"].clone()
    g[:, 64:128, 0, :16] = -2.5
    g[:, 128:, 1, 100:] = -4.0
    _check(dict(inp, g=g))


def test_positive_channel_gates():
    """Mildly positive per-channel log-gates (0.005 +- 0.02 a token: the
    state grows by about e^0.3 a chunk), mixed with negative ones.  (The gated
    query of the inter-chunk output is one bf16 operand; under strong growth,
    0.02 +- 0.05 a token, its rounding reaches 2.2e-2 of RMS(o).)"""
    inp = _raw_problem(62)
    r = torch.Generator().manual_seed(8)
    g = 0.005 + 0.02 * torch.randn(inp["g"].shape, generator=r)
    _check(dict(inp, g=g.float()))


def test_channel_gate_reset():
    """A -1000 rate zeroes the decay: every channel of head 0 at token 90, and
    half the channels of head 1 at a chunk's first token (128)."""
    inp = _raw_problem(63)
    g = inp["g"].clone()
    g[:, 90, 0, :] = -1000.0
    g[:, 128, 1, :64] = -1000.0
    _check(dict(inp, g=g))


def test_zero_length_batch_returns_the_initial_state():
    B, H, K, V = 2, 4, 128, 64
    q = torch.empty((B, 0, H, K), dtype=torch.bfloat16, device="cuda")
    v = torch.empty((B, 0, H, V), dtype=torch.bfloat16, device="cuda")
    g = torch.empty((B, 0, H, K), dtype=torch.float32, device="cuda")
    beta = torch.empty((B, 0, H), dtype=torch.float32, device="cuda")
    h0 = torch.randn((B, H, K, V), generator=torch.Generator().manual_seed(6)).cuda()
    o, ht = kda_chunk_fwd(q, q, v, g, beta, initial_state=h0)
    torch.cuda.synchronize()
    assert gdn_check_device_error() == Status.OK
    assert tuple(o.shape) == (B, 0, H, V)
    assert torch.equal(ht, h0)


@pytest.mark.parametrize("dtype,K", [(torch.bfloat16, 128), (torch.float32, 64)])
def test_state_v_first_layout(dtype, K):
    inp = synth.prefill_inputs(83, 1, 140, 4, 2, K, 64, dtype=dtype, h0_std=0.1,
                               per_channel=True)
    d = to_dev(inp)
    o1, ht1 = kda_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], initial_state=d["h0"],
                            out_dtype=torch.float32)
    h0t = d["h0"].transpose(-1, -2).contiguous()
    o2, ht2 = kda_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], initial_state=h0t,
                            state_v_first=True, out_dtype=torch.float32)
    assert gdn_check_device_error() == Status.OK
    assert torch.equal(o1, o2)
    assert torch.equal(ht2, ht1.transpose(-1, -2))
    o_ref, ht_ref = run_oracle(inp)
    tol = TOL_F32 if dtype == torch.float32 else TOL_BF16
    assert_close(o2, o_ref, tol, "o")
    assert_close(ht2.transpose(-1, -2), ht_ref, tol, "ht")
