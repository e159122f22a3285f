"""Pins of the fp64 oracle against facts that do not come from the oracle itself.

Each test fixes the oracle to something independent: a hand-worked example, the
closed-form product of transition matrices, an algebraically different
(chunked) statement of the method, closed forms and invariants.  A dropped
term, a wrong sign, a swapped index or a transposed operand in the oracle makes
at least one of them fail (K != V is used throughout so transposes show up).
"""
import json
import math
import os

import numpy as np
import pytest

from oracle import recurrence as R
from oracle import brute, chunked

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand_problem(rng, B, T, Hg, H, K, V, per_channel=False, with_h0=True, gate_scale=0.3):
    q = rng.standard_normal((B, T, Hg, K))
    k = rng.standard_normal((B, T, Hg, K))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, T, H, V))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((B, T, H))))
    gshape = (B, T, H, K) if per_channel else (B, T, H)
    g = -gate_scale * np.abs(rng.standard_normal(gshape))
    N = B
    h0 = rng.standard_normal((N, H, K, V)) if with_h0 else None
    return q, k, v, g, beta, h0


# ---------------------------------------------------------------- hand example

def test_hand_worked_example():
    with open(os.path.join(GOLDEN, "hand_k2.json")) as f:
        ex = json.load(f)
    q = np.array(ex["q"])[None, :, None, :]
    k = np.array(ex["k"])[None, :, None, :]
    v = np.array(ex["v"])[None, :, None, :]
    beta = np.array(ex["beta"])[None, :, None]
    g = np.log(np.array(ex["decay"]))[None, :, None]
    h0 = np.array(ex["h0"])[None, None]
    o, ht = R.gdn_recurrent(q, k, v, g, beta, scale=ex["scale"], h0=h0)
    np.testing.assert_allclose(o[0, :, 0], np.array(ex["o"]), atol=1e-12)
    np.testing.assert_allclose(ht[0, 0], np.array(ex["ht"]), atol=1e-12)
    for BT in (1, 2, 3):
        oc, htc = chunked.chunked_forward(q, k, v, g, beta, BT, scale=ex["scale"], h0=h0)
        np.testing.assert_allclose(oc[0, :, 0], np.array(ex["o"]), atol=1e-12)
        np.testing.assert_allclose(htc[0, 0], np.array(ex["ht"]), atol=1e-12)


# ---------------------------------------------------------------- brute force

@pytest.mark.parametrize("per_channel", [False, True])
def test_recurrence_matches_transition_product(per_channel):
    rng = np.random.default_rng(11)
    B, T, Hg, H, K, V = 2, 7, 1, 2, 3, 5
    q, k, v, g, beta, h0 = _rand_problem(rng, B, T, Hg, H, K, V, per_channel)
    # unnormalised keys too: the product formula does not care
    k = k * rng.uniform(0.5, 1.5, size=k.shape[:-1] + (1,))
    scale = 0.7
    fn = R.kda_recurrent if per_channel else R.gdn_recurrent
    kw = {"g_is_cumsum": False} if per_channel else {}
    o, ht = fn(q, k, v, g, beta, scale=scale, h0=h0, **kw)
    for b in range(B):
        for h in range(H):
            hk = h // (H // Hg)
            gg = g[b, :, h, :] if per_channel else g[b, :, h]
            ob, Sb = brute.chain_outputs(h0[b, h].T, gg, beta[b, :, h], q[b, :, hk],
                                         k[b, :, hk], v[b, :, h], scale)
            np.testing.assert_allclose(o[b, :, h], ob, rtol=1e-11, atol=1e-11)
            np.testing.assert_allclose(ht[b, h], Sb.T, rtol=1e-11, atol=1e-11)


# ---------------------------------------------------------------- chunked == recurrent

@pytest.mark.parametrize("per_channel", [False, True])
def test_chunked_equals_recurrent_for_every_chunk_length(per_channel):
    rng = np.random.default_rng(5)
    lengths = [5, 8]
    T = sum(lengths)
    cu = np.array([0, 5, 13])
    Hg, H, K, V = 1, 2, 4, 3
    q, k, v, g, beta, _ = _rand_problem(rng, 1, T, Hg, H, K, V, per_channel, with_h0=False)
    h0 = rng.standard_normal((2, H, K, V))
    fn = R.kda_recurrent if per_channel else R.gdn_recurrent
    kw = {"g_is_cumsum": False} if per_channel else {}
    o_ref, ht_ref = fn(q, k, v, g, beta, scale=0.5, h0=h0, cu_seqlens=cu, **kw)
    for BT in range(1, T + 1):
        o, ht = chunked.chunked_forward(q, k, v, g, beta, BT, scale=0.5, h0=h0,
                                        cu_seqlens=cu, per_channel=per_channel)
        np.testing.assert_allclose(o, o_ref, rtol=1e-10, atol=1e-10, err_msg=f"BT={BT}")
        np.testing.assert_allclose(ht, ht_ref, rtol=1e-10, atol=1e-10, err_msg=f"BT={BT}")


def test_unit_lower_inverse_is_inverse():
    rng = np.random.default_rng(3)
    A = np.tril(rng.standard_normal((9, 9)), -1)
    Ti = chunked.unit_lower_inverse(A)
    np.testing.assert_allclose(Ti @ (np.eye(9) + A), np.eye(9), atol=1e-9)


# ---------------------------------------------------------------- closed forms

@pytest.mark.parametrize("per_channel", [False, True])
def test_beta_zero_gate_zero_keeps_state(per_channel):
    rng = np.random.default_rng(7)
    B, T, Hg, H, K, V = 1, 9, 1, 1, 4, 6
    q, k, v, g, beta, h0 = _rand_problem(rng, B, T, Hg, H, K, V, per_channel)
    g[:] = 0.0
    beta[:] = 0.0
    fn = R.kda_recurrent if per_channel else R.gdn_recurrent
    kw = {"g_is_cumsum": False} if per_channel else {}
    o, ht = fn(q, k, v, g, beta, scale=0.3, h0=h0, **kw)
    np.testing.assert_array_equal(ht, h0)
    np.testing.assert_allclose(o[0, :, 0], 0.3 * q[0, :, 0] @ h0[0, 0], atol=1e-13)


def test_delta_rule_writes_value_exactly():
    rng = np.random.default_rng(8)
    B, T, Hg, H, K, V = 1, 6, 1, 1, 5, 3
    q, k, v, g, beta, h0 = _rand_problem(rng, B, T, Hg, H, K, V)
    beta[:] = 1.0
    for t in range(1, T + 1):
        _, ht = R.gdn_recurrent(q[:, :t], k[:, :t], v[:, :t], g[:, :t], beta[:, :t],
                                scale=1.0, h0=h0)
        S = ht[0, 0].T
        np.testing.assert_allclose(S @ k[0, t - 1, 0], v[0, t - 1, 0], atol=1e-12)


def test_gate_to_minus_infinity_resets_state():
    rng = np.random.default_rng(9)
    q, k, v, g, beta, h0 = _rand_problem(rng, 1, 4, 1, 1, 3, 2)
    g[0, 3, 0] = -1e4  # exp underflows to exactly 0
    _, ht = R.gdn_recurrent(q, k, v, g, beta, scale=1.0, h0=h0)
    np.testing.assert_allclose(ht[0, 0].T, beta[0, 3, 0] * np.outer(v[0, 3, 0], k[0, 3, 0]),
                               atol=1e-14)


# ---------------------------------------------------------------- reductions

def test_kda_with_channel_constant_gate_equals_gdn():
    rng = np.random.default_rng(12)
    B, T, H, K, V = 1, 10, 2, 4, 3
    q, k, v, g, beta, h0 = _rand_problem(rng, B, T, H, H, K, V)
    gk = np.repeat(g[..., None], K, axis=-1)
    o1, ht1 = R.gdn_recurrent(q, k, v, g, beta, scale=0.4, h0=h0)
    o2, ht2 = R.kda_recurrent(q, k, v, gk, beta, scale=0.4, h0=h0, g_is_cumsum=False)
    np.testing.assert_allclose(o1, o2, atol=1e-13)
    np.testing.assert_allclose(ht1, ht2, atol=1e-13)


def test_grouped_heads_equal_repeated_heads():
    rng = np.random.default_rng(13)
    B, T, Hg, H, K, V = 2, 6, 2, 6, 3, 4
    q, k, v, g, beta, h0 = _rand_problem(rng, B, T, Hg, H, K, V)
    o1, ht1 = R.gdn_recurrent(q, k, v, g, beta, scale=0.5, h0=h0)
    rep = H // Hg
    o2, ht2 = R.gdn_recurrent(np.repeat(q, rep, axis=2), np.repeat(k, rep, axis=2), v, g, beta,
                              scale=0.5, h0=h0)
    np.testing.assert_allclose(o1, o2, atol=1e-13)
    np.testing.assert_allclose(ht1, ht2, atol=1e-13)


def test_varlen_equals_separate_runs_and_cumsum_gate_input():
    rng = np.random.default_rng(14)
    lengths = [3, 70, 1, 66]
    T = sum(lengths)
    cu = np.concatenate([[0], np.cumsum(lengths)])
    q, k, v, g, beta, _ = _rand_problem(rng, 1, T, 1, 2, 3, 2)
    h0 = rng.standard_normal((4, 2, 3, 2))
    o, ht = R.gdn_recurrent(q, k, v, g, beta, scale=0.5, h0=h0, cu_seqlens=cu)
    # the same gate handed over as the chunk-local cumulative sum (64-token chunks)
    gc = g.copy()
    for n in range(4):
        for c in range(cu[n], cu[n + 1], 64):
            e = min(c + 64, cu[n + 1])
            gc[:, c:e] = np.cumsum(g[:, c:e], axis=1)
    oc, htc = R.gdn_recurrent(q, k, v, gc, beta, scale=0.5, h0=h0, cu_seqlens=cu,
                              g_is_cumsum=True)
    np.testing.assert_allclose(oc, o, atol=1e-12)
    np.testing.assert_allclose(htc, ht, atol=1e-12)
    for n in range(4):
        s, e = cu[n], cu[n + 1]
        o1, ht1 = R.gdn_recurrent(q[:, s:e], k[:, s:e], v[:, s:e], g[:, s:e], beta[:, s:e],
                                  scale=0.5, h0=h0[n:n + 1])
        np.testing.assert_allclose(o[:, s:e], o1, atol=1e-13)
        np.testing.assert_allclose(ht[n], ht1[0], atol=1e-13)


def test_prefix_then_resume_equals_full_run():
    rng = np.random.default_rng(15)
    q, k, v, g, beta, h0 = _rand_problem(rng, 1, 20, 1, 1, 4, 3, per_channel=True)
    o, ht = R.kda_recurrent(q, k, v, g, beta, scale=1.0, h0=h0, g_is_cumsum=False)
    oa, hta = R.kda_recurrent(q[:, :8], k[:, :8], v[:, :8], g[:, :8], beta[:, :8], scale=1.0,
                              h0=h0, g_is_cumsum=False)
    ob, htb = R.kda_recurrent(q[:, 8:], k[:, 8:], v[:, 8:], g[:, 8:], beta[:, 8:], scale=1.0,
                              h0=hta, g_is_cumsum=False)
    np.testing.assert_allclose(np.concatenate([oa, ob], axis=1), o, atol=1e-13)
    np.testing.assert_allclose(htb, ht, atol=1e-13)


# ---------------------------------------------------------------- decode

def test_softplus_against_log1p_and_threshold_edge():
    for x in (-30.0, -1.0, 0.0, 0.5, 19.999, 20.0):
        assert abs(float(R.softplus(np.array(x))) - math.log1p(math.exp(x))) < 1e-15 * max(1, x)
    # above the threshold the value is x itself (not log1p(exp(x)))
    assert float(R.softplus(np.array(20.001))) == 20.001
    assert float(R.softplus(np.array(30.0))) == 30.0
    assert abs(float(R.softplus(np.array(0.0))) - math.log(2.0)) < 1e-16
    # softplus_beta scales the argument and divides the result
    assert abs(float(R.softplus(np.array(1.5), beta=2.0)) - math.log1p(math.exp(3.0)) / 2) < 1e-15
    assert float(R.softplus(np.array(11.0), beta=2.0)) == 11.0


def test_decode_gates_closed_form():
    a = np.array([[[0.3, -2.0]]])
    b = np.array([[[0.0, 1.0]]])
    A_log = np.array([0.0, math.log(2.0)])
    dt = np.array([0.7, 0.5])
    g, beta = R.decode_gates(a, b, A_log, dt)
    assert abs(g[0, 0, 0] + math.log1p(math.exp(1.0))) < 1e-15
    assert abs(g[0, 0, 1] + 2.0 * math.log1p(math.exp(-1.5))) < 1e-15
    assert beta[0, 0, 0] == 0.5
    assert abs(beta[0, 0, 1] - 1.0 / (1.0 + math.exp(-1.0))) < 1e-16


def test_decode_matches_prefill_recurrence_and_chains_over_calls():
    rng = np.random.default_rng(16)
    B, T, H, HV, K, V = 2, 4, 1, 2, 6, 5
    q = rng.standard_normal((B, T, H, K))
    k = rng.standard_normal((B, T, H, K))
    v = rng.standard_normal((B, T, HV, V))
    a = rng.standard_normal((B, T, HV))
    b = rng.standard_normal((B, T, HV))
    A_log = rng.standard_normal(HV)
    dt = rng.standard_normal(HV)
    state = rng.standard_normal((3, HV, V, K))
    slots = np.array([2, 0])
    o, ns = R.gdn_decode(q, k, v, a, b, A_log, dt, state, slots, scale=0.25)
    # the same tokens through the prefill definition with normalised q/k and the gates
    g, beta = R.decode_gates(a, b, A_log, dt)
    qn, kn = R.l2_normalize(q), R.l2_normalize(k)
    h0 = np.transpose(state[slots], (0, 1, 3, 2))
    op, htp = R.gdn_recurrent(qn, kn, v, g, beta, scale=0.25, h0=h0)
    np.testing.assert_allclose(o, op, atol=1e-12)
    np.testing.assert_allclose(ns, np.transpose(htp, (0, 1, 3, 2)), atol=1e-12)
    # four one-token calls chained through the pool equal one four-token call
    st = state.copy()
    outs = []
    for t in range(T):
        ot, nst = R.gdn_decode(q[:, t:t + 1], k[:, t:t + 1], v[:, t:t + 1], a[:, t:t + 1],
                               b[:, t:t + 1], A_log, dt, st, slots, scale=0.25)
        st[slots] = nst
        outs.append(ot)
    np.testing.assert_allclose(np.concatenate(outs, axis=1), o, atol=1e-12)
    np.testing.assert_allclose(st[slots], ns, atol=1e-12)


def test_l2_normalize_eps_inside_root():
    x = np.array([3.0, 4.0])
    np.testing.assert_allclose(R.l2_normalize(x, eps=0.0), [0.6, 0.8], atol=1e-16)
    np.testing.assert_allclose(R.l2_normalize(x, eps=11.0), [0.5, 2.0 / 3.0], atol=1e-16)


# ---------------------------------------------------------------- gate given as a chunk-local cumsum

def _chunk_cumsum_by_hand(g_raw, cu, chunk):
    """Inclusive running sums of the raw gates, restarted at every chunk of
    `chunk` tokens counted from each sequence's first token (token axis 1)."""
    out = np.zeros_like(g_raw)
    for n in range(len(cu) - 1):
        acc = None
        for t in range(cu[n], cu[n + 1]):
            if (t - cu[n]) % chunk == 0:
                acc = np.zeros_like(g_raw[:, t])
            acc = acc + g_raw[:, t]
            out[:, t] = acc
    return out


@pytest.mark.parametrize("chunk", [64, 4])
def test_kda_cumsum_gate_input_equals_raw_and_transition_product(chunk):
    """kda_recurrent's default input form: per-channel gates as chunk-local
    cumulative sums.  Packed sequences whose starts are not chunk-aligned
    (70, 71) and that span several chunks; grouped value heads; K != V."""
    rng = np.random.default_rng(21)
    lengths = [70, 1, 130]
    T = sum(lengths)
    cu = np.concatenate([[0], np.cumsum(lengths)])
    H, HV, K, V = 1, 2, 3, 2
    q, k, v, g_raw, beta, _ = _rand_problem(rng, 1, T, H, HV, K, V, per_channel=True,
                                            with_h0=False, gate_scale=0.2)
    h0 = rng.standard_normal((3, HV, K, V))
    g_cum = _chunk_cumsum_by_hand(g_raw, cu, chunk)
    o1, ht1 = R.kda_recurrent(q, k, v, g_cum, beta, scale=0.6, h0=h0, cu_seqlens=cu,
                              g_is_cumsum=True, chunk_size=chunk)
    o2, ht2 = R.kda_recurrent(q, k, v, g_raw, beta, scale=0.6, h0=h0, cu_seqlens=cu,
                              g_is_cumsum=False)
    np.testing.assert_allclose(o1, o2, atol=1e-12)
    np.testing.assert_allclose(ht1, ht2, atol=1e-12)
    for n in range(3):
        s, e = cu[n], cu[n + 1]
        for hv in range(HV):
            hk = hv // (HV // H)
            ob, Sb = brute.chain_outputs(h0[n, hv].T, g_raw[0, s:e, hv, :], beta[0, s:e, hv],
                                         q[0, s:e, hk], k[0, s:e, hk], v[0, s:e, hv], 0.6)
            np.testing.assert_allclose(o1[0, s:e, hv], ob, rtol=1e-10, atol=1e-10)
            np.testing.assert_allclose(ht1[n, hv], Sb.T, rtol=1e-10, atol=1e-10)


def test_kda_cumsum_gate_reset_counts_chunks_from_each_sequence_start():
    """Counting chunks from the packed row's first token instead (a plausible
    slip) changes the result whenever a sequence starts off a chunk boundary."""
    rng = np.random.default_rng(22)
    lengths = [5, 9]
    cu = np.concatenate([[0], np.cumsum(lengths)])
    q, k, v, g_raw, beta, _ = _rand_problem(rng, 1, 14, 1, 1, 2, 2, per_channel=True,
                                            with_h0=False)
    right = _chunk_cumsum_by_hand(g_raw, cu, 4)
    wrong = _chunk_cumsum_by_hand(g_raw, np.array([0, 14]), 4)
    o_r, _ = R.kda_recurrent(q, k, v, right, beta, scale=1.0, cu_seqlens=cu, chunk_size=4)
    o_w, _ = R.kda_recurrent(q, k, v, wrong, beta, scale=1.0, cu_seqlens=cu, chunk_size=4)
    o_raw, _ = R.kda_recurrent(q, k, v, g_raw, beta, scale=1.0, cu_seqlens=cu, g_is_cumsum=False)
    np.testing.assert_allclose(o_r, o_raw, atol=1e-12)
    assert np.max(np.abs(o_w - o_raw)) > 1e-3


# ---------------------------------------------------------------- decode without the L2 norm

def test_decode_without_l2norm_matches_transition_product():
    """use_qk_l2norm = 0: q and k enter as given (q times scale), so the state
    and outputs are the product of the transitions with the raw keys."""
    rng = np.random.default_rng(23)
    B, T, H, HV, K, V = 2, 3, 1, 2, 4, 3
    q = rng.standard_normal((B, T, H, K)) * 0.4
    k = rng.standard_normal((B, T, H, K)) * 0.4     # not unit length
    v = rng.standard_normal((B, T, HV, V))
    a = rng.standard_normal((B, T, HV))
    b = rng.standard_normal((B, T, HV))
    A_log = rng.standard_normal(HV)
    dt = rng.standard_normal(HV)
    state = rng.standard_normal((3, HV, V, K))
    slots = np.array([1, 2])
    o, ns = R.gdn_decode(q, k, v, a, b, A_log, dt, state, slots, scale=0.3, use_qk_l2norm=False)
    g, beta = R.decode_gates(a, b, A_log, dt)
    for bi in range(B):
        for hv in range(HV):
            hk = hv // (HV // H)
            ob, Sb = brute.chain_outputs(state[slots[bi], hv], g[bi, :, hv], beta[bi, :, hv],
                                         q[bi, :, hk], k[bi, :, hk], v[bi, :, hv], 0.3)
            np.testing.assert_allclose(o[bi, :, hv], ob, rtol=1e-11, atol=1e-11)
            np.testing.assert_allclose(ns[bi, hv], Sb, rtol=1e-11, atol=1e-11)
    # and with the norm on, the same product on the normalised keys and queries
    o_n, ns_n = R.gdn_decode(q, k, v, a, b, A_log, dt, state, slots, scale=0.3)
    assert np.max(np.abs(o_n - o)) > 1e-3
    kn = k / np.sqrt(np.sum(k * k, axis=-1, keepdims=True) + 1e-6)
    qn = q / np.sqrt(np.sum(q * q, axis=-1, keepdims=True) + 1e-6)
    ob, Sb = brute.chain_outputs(state[slots[0], 0], g[0, :, 0], beta[0, :, 0], qn[0, :, 0],
                                 kn[0, :, 0], v[0, :, 0], 0.3)
    np.testing.assert_allclose(o_n[0, :, 0], ob, rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(ns_n[0, 0], Sb, rtol=1e-11, atol=1e-11)
