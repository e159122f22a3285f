"""GDN chunked forward on the GPU against the fp64 oracle (through the C ABI)."""
import numpy as np
import pytest
import torch

from gated_delta_rule_kk_gb300 import Status, gdn_check_device_error, gdn_chunk_fwd
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
    o, ht = gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], out_dtype=torch.float32, **kw)
    if d["q"].dtype == torch.bfloat16:
        o16, ht16 = gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], **kw)
        assert o16.dtype == torch.bfloat16
        assert torch.equal(o16, o.to(torch.bfloat16)), "bf16 o is not the RNE of the fp32 o"
        assert torch.equal(ht16, ht)
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
    (200, 128, 32, 2, 1, torch.bfloat16, True),   # tensor cores, one 32-column value tile
    (150, 128, 96, 2, 2, torch.bfloat16, False),  # tensor cores, three value tiles
    (200, 128, 128, 8, 1, torch.bfloat16, True),  # tensor cores, 8 value heads on 1 key head
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


# ---- the named workloads at full size, every chain against the oracle ------

def test_gdn_prefill_workload_all_chains():
    """B=2, T=4096, H=Hg=16, K=V=128, bf16: all 32 (sequence, head) chains."""
    inp = synth.gdn_prefill()
    o, ht = run_gpu(inp)
    o_ref, ht_ref = prefill_all_chains(inp)
    assert_close(o, o_ref, TOL_BF16, "o")
    assert_close(ht, ht_ref, TOL_BF16, "ht")


def test_varlen_gqa_workload_all_chains():
    """8 packed sequences (32,068 tokens), Hg=4 key heads for H=16 value heads:
    all 128 (sequence, head) chains."""
    inp = synth.varlen_gqa()
    o, ht = run_gpu(inp)
    o_ref, ht_ref = prefill_all_chains(inp)
    assert_close(o, o_ref, TOL_BF16, "o")
    assert_close(ht, ht_ref, TOL_BF16, "ht")


# ---- more chains than SMs: the chain grid runs in several waves ----------

@pytest.mark.parametrize("case", ["packed", "batch", "v64"])
def test_chains_outnumbering_the_sms(case):
    """(V / 32) H N chain CTAs above the SM count, so that CTAs start as
    others finish: packed sequences with empty and one-token ones (taken
    longest first), GQA and an initial state; an equal-length batch; and
    V = 64 (two value tiles a head)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    if case == "packed":
        lengths = [150, 0, 1, 64, 65, 200, 3, 129, 90, 17, 256, 40]
        H, Hg, V = 16, 4, 128
        inp = synth.prefill_inputs(61, 1, sum(lengths), H, Hg, 128, V, dtype=torch.bfloat16,
                                   lengths=lengths)
        inp["h0"] = 0.1 * torch.randn(len(lengths), H, 128, V,
                                      generator=torch.Generator().manual_seed(62))
        N = len(lengths)
    elif case == "batch":
        N, H, Hg, V = 5, 16, 16, 128
        inp = synth.prefill_inputs(63, N, 130, H, Hg, 128, V, dtype=torch.bfloat16, h0_std=0.1)
    else:
        N, H, Hg, V = 10, 16, 8, 64
        inp = synth.prefill_inputs(64, N, 100, H, Hg, 128, V, dtype=torch.bfloat16, h0_std=0.1)
    assert (V // 32) * H * N > sms
    _check(inp)


# ---- gates the synthetic workloads never reach, on the tensor-core path ----

def _tc_problem(seed, T=256, H=2, Hg=1):
    return synth.prefill_inputs(seed, 1, T, H, Hg, 128, 128, dtype=torch.bfloat16, h0_std=0.1)


def _check(inp):
    o, ht = run_gpu(inp)
    o_ref, ht_ref = run_oracle(inp)
    assert_close(o, o_ref, TOL_BF16, "o")
    assert_close(ht, ht_ref, TOL_BF16, "ht")


def test_strong_gates_inside_a_chunk_take_the_exact_exponentials():
    """A chunk whose cumulative gate falls below -80 (tokens 64..127 at -2.5
    each) is gated with exact per-element exponentials; its neighbours keep
    the split form.  Head 1 is strong in the tail chunk instead."""
    inp = _tc_problem(51, T=230)
    g = inp["g"].clone()
    g[:, 64:128, 0] = -2.5
    g[:, 192:, 1] = -3.0
    _check(dict(inp, g=g))


def test_positive_log_gates():
    """Log-gates above zero (a growing state), mixed with negative ones."""
    inp = _tc_problem(52, T=200)
    r = torch.Generator().manual_seed(7)
    g = 0.02 + 0.05 * torch.randn(inp["g"].shape, generator=r)
    _check(dict(inp, g=g.float()))


def test_gate_reset_mid_chunk_and_at_a_chunk_start():
    """g = -1000 (exp underflows to exactly zero in fp32) wipes the state: at a
    token inside a chunk for head 0 and at a chunk's first token for head 1."""
    inp = _tc_problem(53, T=200)
    g = inp["g"].clone()
    g[:, 90, 0] = -1000.0
    g[:, 128, 1] = -1000.0
    _check(dict(inp, g=g))


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


# ---- state_v_first: h0 / ht as [V, K] (the chunk_h page's layout flag) -----

@pytest.mark.parametrize("dtype,K,V,lengths", [
    (torch.bfloat16, 128, 128, None),       # tensor cores
    (torch.bfloat16, 128, 64, [70, 0, 130]),  # tensor cores, packed, an empty sequence
    (torch.float32, 64, 48, [1, 0, 99]),     # exact fp32 kernel
])
def test_state_v_first_layout(dtype, K, V, lengths):
    T = 150 if lengths is None else sum(lengths)
    B = 2 if lengths is None else 1
    inp = synth.prefill_inputs(81, B, T, 4, 2, K, V, dtype=dtype, h0_std=0.1, lengths=lengths)
    d = to_dev(inp)
    kw = dict(scale=d["scale"], cu_seqlens=d["cu_seqlens"], out_dtype=torch.float32)
    o1, ht1 = gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], initial_state=d["h0"], **kw)
    h0t = d["h0"].transpose(-1, -2).contiguous()
    o2, ht2 = gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], initial_state=h0t,
                            state_v_first=True, **kw)
    assert gdn_check_device_error() == Status.OK
    assert tuple(ht2.shape) == tuple(h0t.shape)
    # the layout changes where states live, not the arithmetic
    assert torch.equal(o1, o2)
    assert torch.equal(ht2, ht1.transpose(-1, -2))
    o_ref, ht_ref = run_oracle(inp)
    tol = TOL_F32 if dtype == torch.float32 else TOL_BF16
    assert_close(o2, o_ref, tol, "o")
    assert_close(ht2.transpose(-1, -2), ht_ref, tol, "ht")
    if lengths is not None:
        for n in (i for i, x in enumerate(lengths) if x == 0):
            assert torch.equal(ht2[n], h0t[n])


def test_state_v_first_host_entry_point():
    import gated_delta_rule_kk_gb300 as gdn
    inp = synth.prefill_inputs(82, 1, 1000, 2, 1, 128, 128, h0_std=0.1)
    d = to_dev(inp)
    h0t = inp["h0"].transpose(-1, -2).contiguous()
    o1, ht1 = gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], scale=d["scale"],
                            initial_state=h0t.cuda(), state_v_first=True, segments=1)
    o2, ht2 = gdn.gdn_chunk_fwd_host(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                                     scale=inp["scale"], initial_state=h0t.pin_memory(),
                                     state_v_first=True)
    torch.cuda.synchronize()
    assert gdn_check_device_error() == Status.OK
    assert torch.equal(o2, o1.cpu())
    assert torch.equal(ht2, ht1.cpu())
