"""Pins of the chunk-state-pass oracle (gated linear attention, chunk_h page).

The oracle steps the recurrence token by token; these tests tie it to things
it does not compute that way: the multiplied-out closed form of the state,
the reductions between gate kinds (a per-head constant rate is a per-token
gate with equal values; a per-channel gate constant across its channels is the
scalar gate), and what the chunk-start states mean (the first is h0, a
sequence resumed from a chunk-start state continues the same run).
"""
import numpy as np
import pytest

from oracle import brute
from oracle import state_pass as SP



def _inputs(seed, B, T, H, K, V):
    rng = np.random.default_rng(seed)
    k = rng.standard_normal((B, T, H, K))
    v = rng.standard_normal((B, T, H, V))
    raw_g = -np.abs(rng.standard_normal((B, T, H))) * 0.3
    raw_gk = -np.abs(rng.standard_normal((B, T, H, K))) * 0.3
    raw_gv = -np.abs(rng.standard_normal((B, T, H, V))) * 0.3
    h0 = rng.standard_normal((B, H, K, V))
    return k, v, raw_g, raw_gk, raw_gv, h0


def _chunk_cumsum(raw, chunk):
    out = np.empty_like(raw)
    T = raw.shape[1]
    for c in range(0, T, chunk):
        out[:, c:c + chunk] = np.cumsum(raw[:, c:c + chunk], axis=1)
    return out


@pytest.mark.parametrize("gate", SP.GATES)
def test_final_state_matches_closed_form(gate):
    B, T, H, K, V, chunk = 1, 7, 2, 3, 4, 3
    k, v, rg, rgk, rgv, h0 = _inputs(1, B, T, H, K, V)
    gamma = np.array([-0.2, -0.05])
    vals = {None: None, "g": _chunk_cumsum(rg, chunk), "g_gamma": gamma,
            "gk": _chunk_cumsum(rgk, chunk), "gv": _chunk_cumsum(rgv, chunk)}[gate]
    hs, ht = SP.chunk_state_pass(k, v, gate, vals, h0=h0, chunk_size=chunk)
    for h in range(H):
        dk = np.ones((T, K))
        dv = np.ones((T, V))
        if gate == "g":
            dk = np.repeat(np.exp(rg[0, :, h])[:, None], K, axis=1)
        elif gate == "g_gamma":
            dk = np.full((T, K), np.exp(gamma[h]))
        elif gate == "gk":
            dk = np.exp(rgk[0, :, h])
        elif gate == "gv":
            dv = np.exp(rgv[0, :, h])
        ref_t = brute.linear_state_after(h0[0, h], dk, dv, k[0, :, h], v[0, :, h], T)
        np.testing.assert_allclose(ht[0, h], ref_t, rtol=1e-12, atol=1e-12)
        for c in range(hs.shape[0]):  # chunk starts at tokens 0, 3, 6
            ref_c = brute.linear_state_after(h0[0, h], dk, dv, k[0, :, h], v[0, :, h], c * chunk)
            np.testing.assert_allclose(hs[c, h], ref_c, rtol=1e-12, atol=1e-12)


def test_gate_kinds_reduce_to_each_other():
    B, T, H, K, V, chunk = 2, 13, 3, 4, 5, 4
    k, v, rg, _, _, h0 = _inputs(2, B, T, H, K, V)
    g = _chunk_cumsum(rg, chunk)
    ref = SP.chunk_state_pass(k, v, "g", g, h0=h0, chunk_size=chunk)
    gk = np.repeat(g[..., None], K, axis=3)
    gv = np.repeat(g[..., None], V, axis=3)
    for gate, vals in (("gk", gk), ("gv", gv)):
        got = SP.chunk_state_pass(k, v, gate, vals, h0=h0, chunk_size=chunk)
        np.testing.assert_allclose(got[0], ref[0], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(got[1], ref[1], rtol=1e-12, atol=1e-12)
    # a per-head constant rate is the per-token gate with that value everywhere
    gamma = np.array([-0.3, -0.01, 0.0])
    const = _chunk_cumsum(np.broadcast_to(gamma, (B, T, H)).copy(), chunk)
    a = SP.chunk_state_pass(k, v, "g_gamma", gamma, h0=h0, chunk_size=chunk)
    b = SP.chunk_state_pass(k, v, "g", const, h0=h0, chunk_size=chunk)
    np.testing.assert_allclose(a[0], b[0], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(a[1], b[1], rtol=1e-12, atol=1e-12)
    # no gate is a zero gate
    a = SP.chunk_state_pass(k, v, None, None, h0=h0, chunk_size=chunk)
    b = SP.chunk_state_pass(k, v, "g", np.zeros_like(g), h0=h0, chunk_size=chunk)
    np.testing.assert_allclose(a[1], b[1], rtol=1e-12, atol=1e-12)


def test_chunk_starts_resume_the_run_and_packed_sequences_are_separate_runs():
    B, T, H, K, V, chunk = 1, 20, 2, 3, 3, 4
    k, v, _, rgk, _, h0 = _inputs(3, B, T, H, K, V)
    gk = _chunk_cumsum(rgk, chunk)
    hs, ht = SP.chunk_state_pass(k, v, "gk", gk, h0=h0, chunk_size=chunk)
    assert hs.shape == (5, H, K, V)
    np.testing.assert_array_equal(hs[0], h0[0])
    # resuming at chunk 3 (token 12) from its chunk-start state gives the same end
    rs, rt = SP.chunk_state_pass(k[:, 12:], v[:, 12:], "gk", gk[:, 12:], h0=hs[3][None],
                                 chunk_size=chunk)
    np.testing.assert_allclose(rt, ht, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(rs, hs[3:], rtol=1e-12, atol=1e-12)
    # packed sequences (one empty) = separate runs, chunk states one after another
    lens = [6, 0, 9, 5]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    rng = np.random.default_rng(4)
    kk = rng.standard_normal((1, cu[-1], H, K))
    vv = rng.standard_normal((1, cu[-1], H, V))
    raw = -np.abs(rng.standard_normal((1, cu[-1], H)))
    gg = np.empty_like(raw)
    for n in range(len(lens)):
        for c in range(cu[n], cu[n + 1], chunk):
            e = min(c + chunk, cu[n + 1])
            gg[:, c:e] = np.cumsum(raw[:, c:e], axis=1)
    hh0 = rng.standard_normal((len(lens), H, K, V))
    hs_p, ht_p = SP.chunk_state_pass(kk, vv, "g", gg, h0=hh0, cu_seqlens=cu, chunk_size=chunk)
    assert hs_p.shape[0] == sum(-(-n // chunk) for n in lens)
    first = 0
    for n in range(len(lens)):
        a, b = cu[n], cu[n + 1]
        s_n, t_n = SP.chunk_state_pass(kk[:, a:b], vv[:, a:b], "g", gg[:, a:b], h0=hh0[n][None],
                                       chunk_size=chunk)
        np.testing.assert_allclose(ht_p[n], t_n[0], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(hs_p[first:first + s_n.shape[0]], s_n, rtol=1e-12, atol=1e-12)
        first += s_n.shape[0]
    np.testing.assert_array_equal(ht_p[1], hh0[1])  # the empty sequence keeps its state


def _outputs(k, v, q, gate, raw, gamma, h0, scale):
    """o_t = scale S_t^T q_t of one (sequence, head) chain, by stepping the
    forward recurrence (the loss below is linear in h0 and dht)."""
    S = h0.copy()
    outs = []
    for t in range(k.shape[0]):
        if gate == "g":
            S = np.exp(raw[t]) * S
        elif gate == "g_gamma":
            S = np.exp(gamma) * S
        elif gate == "gk":
            S = np.exp(raw[t])[:, None] * S
        elif gate == "gv":
            S = S * np.exp(raw[t])[None, :]
        S = S + np.outer(k[t], v[t])
        outs.append(scale * S.T @ q[t])
    return np.array(outs), S


@pytest.mark.parametrize("gate", SP.GATES)
def test_state_gradient_is_the_adjoint_of_the_forward_pass(gate):
    # L(h0) = sum_t <do_t, o_t> + <dht, S_T> is affine in h0, so for any
    # direction E: L(h0 + E) - L(h0) = <dh0, E>; and dh[c] is the gradient with
    # respect to the state at the end of chunk c (resume the forward run there).
    T, K, V, chunk, scale = 11, 3, 4, 4, 0.7
    rng = np.random.default_rng(7)
    k, v, q, do = (rng.standard_normal((T, K)), rng.standard_normal((T, V)),
                   rng.standard_normal((T, K)), rng.standard_normal((T, V)))
    raw = {None: None, "g": -np.abs(rng.standard_normal(T)) * 0.4, "g_gamma": None,
           "gk": -np.abs(rng.standard_normal((T, K))) * 0.4,
           "gv": -np.abs(rng.standard_normal((T, V))) * 0.4}[gate]
    gamma = -0.3
    h0, dht = rng.standard_normal((K, V)), rng.standard_normal((K, V))
    vals = None
    if gate == "g_gamma":
        vals = np.array([gamma])
    elif gate is not None:
        vals = _chunk_cumsum(raw[None, :, None], chunk)[0, :, 0]
        vals = vals[None, :, None] if raw.ndim == 1 else vals[None, :, None, :]
    dh, dh0 = SP.chunk_state_grad(q[None, :, None], do[None, :, None], gate, vals,
                                  dht=dht[None, None], scale=scale, chunk_size=chunk)

    def loss(start_state, t0):
        o, S = _outputs(k[t0:], v[t0:], q[t0:], gate, None if raw is None else raw[t0:],
                        gamma, start_state, scale)
        return float(np.sum(o * do[t0:]) + np.sum(S * dht))

    E = rng.standard_normal((K, V))
    np.testing.assert_allclose(loss(h0 + E, 0) - loss(h0, 0), np.sum(dh0[0, 0] * E),
                               rtol=1e-10, atol=1e-10)
    for c in range(dh.shape[0]):
        t_end = min((c + 1) * chunk, T)  # the state after token t_end - 1
        if t_end == T:
            np.testing.assert_allclose(dh[c, 0], dht, rtol=1e-12, atol=1e-12)
            continue
        _, S_end = _outputs(k[:t_end], v[:t_end], q[:t_end], gate,
                            None if raw is None else raw[:t_end], gamma, h0, scale)
        np.testing.assert_allclose(loss(S_end + E, t_end) - loss(S_end, t_end),
                                   np.sum(dh[c, 0] * E), rtol=1e-10, atol=1e-10)


def test_state_gradient_grouped_query_heads_share_the_gate():
    B, T, HQ, H, K, V, chunk = 1, 9, 4, 2, 3, 2, 4
    rng = np.random.default_rng(8)
    q, do = rng.standard_normal((B, T, HQ, K)), rng.standard_normal((B, T, HQ, V))
    raw = -np.abs(rng.standard_normal((B, T, H, K))) * 0.3
    gk = _chunk_cumsum(raw, chunk)
    dht = rng.standard_normal((B, HQ, K, V))
    a = SP.chunk_state_grad(q, do, "gk", gk, dht=dht, scale=0.5, chunk_size=chunk)
    b = SP.chunk_state_grad(q, do, "gk", np.repeat(gk, HQ // H, axis=2), dht=dht, scale=0.5,
                            chunk_size=chunk)
    np.testing.assert_allclose(a[0], b[0], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(a[1], b[1], rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("split", [128, 192])
def test_split_size_keeps_every_split_chunk(split):
    # the chunk_h page's split_size: the stored states are those of the chunks
    # whose index is a multiple of split / 64, in order, per sequence
    lengths = [300, 0, 64, 129, 200]
    T, H, K, V = sum(lengths), 2, 8, 4
    rng = np.random.default_rng(21)
    k = rng.standard_normal((1, T, H, K))
    v = rng.standard_normal((1, T, H, V))
    raw = -0.05 * np.abs(rng.standard_normal((1, T, H, K)))
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    gk = np.empty_like(raw)
    for s0, e0 in zip(cu[:-1], cu[1:]):
        for c in range(s0, e0, 64):
            gk[:, c:min(c + 64, e0)] = np.cumsum(raw[:, c:min(c + 64, e0)], axis=1)
    h0 = rng.standard_normal((len(lengths), H, K, V))
    hs1, ht1 = SP.chunk_state_pass(k, v, "gk", gk, h0=h0, cu_seqlens=cu)
    hsS, htS = SP.chunk_state_pass(k, v, "gk", gk, h0=h0, cu_seqlens=cu, split_size=split)
    S = split // 64
    keep, first = [], 0
    for n_chunks in SP.chunk_counts(1, T, cu):
        keep += [first + c for c in range(0, n_chunks, S)]
        first += n_chunks
    assert SP.chunk_counts(1, T, cu, split_size=split) == [-(-x // split) for x in lengths]
    np.testing.assert_array_equal(hsS, hs1[keep])
    np.testing.assert_array_equal(htS, ht1)
    dh1, dh01 = SP.chunk_state_grad(k, v, "gk", gk, dht=h0, cu_seqlens=cu)
    dhS, dh0S = SP.chunk_state_grad(k, v, "gk", gk, dht=h0, cu_seqlens=cu, split_size=split)
    np.testing.assert_array_equal(dhS, dh1[keep])
    np.testing.assert_array_equal(dh0S, dh01)


def test_state_v_first_transposes_every_state():
    # the page's state_v_first: h0 in and every state out are [V, K]; the
    # recurrence is unchanged
    rng = np.random.default_rng(22)
    B, T, H, K, V = 2, 150, 2, 8, 4
    k, v = rng.standard_normal((B, T, H, K)), rng.standard_normal((B, T, H, V))
    raw = -0.05 * np.abs(rng.standard_normal((B, T, H)))
    g = np.concatenate([np.cumsum(raw[:, c:c + 64], axis=1) for c in range(0, T, 64)], axis=1)
    h0 = rng.standard_normal((B, H, K, V))
    hs, ht = SP.chunk_state_pass(k, v, "g", g, h0=h0)
    hsT, htT = SP.chunk_state_pass(k, v, "g", g, h0=h0.swapaxes(-1, -2), state_v_first=True)
    np.testing.assert_array_equal(hsT, hs.swapaxes(-1, -2))
    np.testing.assert_array_equal(htT, ht.swapaxes(-1, -2))
    dh, dh0 = SP.chunk_state_grad(k, v, "g", g, dht=h0)
    dhT, dh0T = SP.chunk_state_grad(k, v, "g", g, dht=h0.swapaxes(-1, -2), state_v_first=True)
    np.testing.assert_array_equal(dhT, dh.swapaxes(-1, -2))
    np.testing.assert_array_equal(dh0T, dh0.swapaxes(-1, -2))
