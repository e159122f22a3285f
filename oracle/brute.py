"""Closed-form product of per-token transition matrices (test infrastructure).

Part of the oracle (test infrastructure only).  This is the pin for the token
recurrence: it does not step a state, it multiplies out

    S_t = S_0 M_1 ... M_t + sum_{j<=t} beta_j v_j k_j^T M_{j+1} ... M_t,
    M_s = D_s (I - beta_s k_s k_s^T),

with ``D_s = exp(g_s) I`` (scalar gate) or ``diag(exp(g_s[:]))`` (per-channel
gate), and ``o_t = scale S_t q_t``.  Meant for tiny sizes (T <= 8, K, V <= 8):
every ``S_t`` is rebuilt from scratch.
"""
from __future__ import annotations

import numpy as np


def _transition(g_s, beta_s, k_s):
    K = k_s.shape[0]
    g_s = np.asarray(g_s, dtype=np.float64)
    D = np.diag(np.exp(g_s)) if g_s.ndim == 1 else np.exp(float(g_s)) * np.eye(K)
    return D @ (np.eye(K) - beta_s * np.outer(k_s, k_s))


def state_after(S0, g, beta, k, v, t):
    """``S_t`` of one chain from the product formula (tokens ``0..t-1``)."""
    K = k.shape[1]
    Ms = [_transition(g[s], beta[s], k[s]) for s in range(t)]

    def prod(a, b):
        P = np.eye(K)
        for s in range(a, b):
            P = P @ Ms[s]
        return P

    S = S0 @ prod(0, t)
    for j in range(t):
        S = S + beta[j] * np.outer(v[j], k[j]) @ prod(j + 1, t)
    return S


def chain_outputs(S0, g, beta, q, k, v, scale):
    """``o_t`` for every token of one chain and the final state ``S_T``.

    S0 [V, K]; g [T] or [T, K]; beta [T]; q, k [T, K]; v [T, V].
    """
    T = q.shape[0]
    o = np.zeros((T, v.shape[1]))
    for t in range(1, T + 1):
        o[t - 1] = scale * state_after(S0, g, beta, k, v, t) @ q[t - 1]
    return o, state_after(S0, g, beta, k, v, T)


def linear_state_after(h0, decay_k, decay_v, k, v, t):
    """State of the gated linear-attention recurrence h <- Dk_s h Dv_s + k_s v_s^T
    after tokens ``0..t-1``, multiplied out (no stepping):

        h_t = (Dk_t ... Dk_1) h0 (Dv_1 ... Dv_t)
              + sum_{j<t} (Dk_t ... Dk_{j+1}) k_j v_j^T (Dv_{j+1} ... Dv_t)

    ``decay_k[s]`` (K) and ``decay_v[s]`` (V) are the diagonals of token s's
    key-side and value-side decay (the scalar and per-head gates put the same
    factor on every key channel and ones on the value side).
    """
    K, V = h0.shape

    def left(a, b):  # Dk_{b-1} ... Dk_a
        P = np.eye(K)
        for s in range(a, b):
            P = np.diag(decay_k[s]) @ P
        return P

    def right(a, b):  # Dv_a ... Dv_{b-1}
        P = np.eye(V)
        for s in range(a, b):
            P = P @ np.diag(decay_v[s])
        return P

    h = left(0, t) @ h0 @ right(0, t)
    for j in range(t):
        h = h + left(j + 1, t) @ np.outer(k[j], v[j]) @ right(j + 1, t)
    return h
