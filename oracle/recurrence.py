"""Token-by-token fp64 definition of the gated delta rule (test infrastructure).

This module is part of the oracle, which is test infrastructure: only tests,
the smoke check and the CPU-baseline leg of the benchmark use it.  It shares no
code with the CUDA library.

The method, as the pages state it per token (FlashInfer
``gdn_decode_bf16_state.py``, helpers ``decay_h_from_smem_and_compute_pred``,
``update_h_with_delta`` and ``compute_output``): with the state ``S`` stored as
a ``[V, K]`` matrix,

    S    <- exp(g_t) * S                   (decay first)
    pred  = S k_t
    delta = beta_t * (v_t - pred)
    S    <- S + delta k_t^T
    o_t   = scale * S q_t

which is ``S_t = S_{t-1} exp(g_t) (I - beta_t k_t k_t^T) + beta_t v_t k_t^T``.
KDA replaces the scalar ``exp(g_t)`` by ``diag(exp(g_t[:]))`` acting on the K
columns of ``S`` (vLLM kimi_k3 ``kda/chunk_intra`` page, kernel docstring and
the per-channel ``exp2(g)`` factors of ``chunk_kda_fwd_kernel_inter_solve_fused``).

Everything is float64.  Inputs are the exact values the GPU receives (bf16 or
fp32, widened).  The prefill state layout at the interface is ``h = S^T``
``[K, V]`` (KDA ``chunk_h.py`` page, ``chunk_fwd_h``: ``h``/``ht`` are
``[N, H, K, V]``, ``ht`` in fp32).
"""
from __future__ import annotations

import math

import numpy as np


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor -> numpy float64
        x = x.detach().cpu().double().numpy()
    return np.asarray(x, dtype=np.float64)


def sequence_bounds(B: int, T: int, cu_seqlens=None):
    """Sequences as ``(batch_row, bos, eos)`` triples.

    Without ``cu_seqlens`` there are ``B`` sequences of length ``T`` (one per
    batch row).  With it, ``B`` must be 1 and sequence ``n`` covers tokens
    ``cu_seqlens[n] .. cu_seqlens[n+1]`` of that row (sglang
    ``fla/chunk_fwd.py``, kernel prologue: ``bos, eos`` from ``cu_seqlens``).
    """
    if cu_seqlens is None:
        return [(b, 0, T) for b in range(B)]
    cu = [int(x) for x in np.asarray(cu_seqlens).reshape(-1)]
    if B != 1:
        raise ValueError("variable-length input needs B == 1")
    if cu[0] != 0 or cu[-1] != T or any(cu[i + 1] < cu[i] for i in range(len(cu) - 1)):
        raise ValueError("cu_seqlens must rise from 0 to T")
    return [(0, cu[n], cu[n + 1]) for n in range(len(cu) - 1)]


def raw_gate_from_chunk_cumsum(gamma, bos: int, eos: int, chunk_size: int = 64):
    """Per-token log-gates from a chunk-local inclusive cumulative sum.

    ``gamma[t]`` holds the sum of the raw gates from the first token of t's
    chunk up to t, chunks being ``chunk_size`` tokens counted from the start of
    the sequence (sglang ``fla/chunk_fwd.py``, ``chunk_gated_delta_rule_fwd_intra``
    docstring: ``g`` is the cumulative sum inside each chunk).  The raw gate is
    the difference of neighbours inside a chunk and the value itself at a
    chunk's first token.  Works on the token axis 0; extra axes (KDA's K) ride
    along.
    """
    gamma = np.asarray(gamma, dtype=np.float64)
    raw = gamma.copy()
    for t in range(bos, eos):
        if (t - bos) % chunk_size != 0:
            raw[t] = gamma[t] - gamma[t - 1]
    return raw


def gdn_recurrent(q, k, v, g, beta, scale=None, h0=None, cu_seqlens=None,
                  g_is_cumsum=False, chunk_size=64, heads=None, seqs=None):
    """Scalar-gate (GDN) forward, token by token.

    Shapes (sglang ``fla/chunk_fwd.py``, ``chunk_gated_delta_rule_fwd_intra``
    docstring; grouped heads from its kernel prologue where key head
    ``i_h // (H // Hg)`` serves value head ``i_h``):
      q, k  [B, T, Hg, K];  v  [B, T, H, V];  g, beta  [B, T, H]
      h0    [N, H, K, V] or None (zeros)
    ``g`` is the natural-log gate per token, or its chunk-local cumulative sum
    when ``g_is_cumsum``.  ``heads``/``seqs`` restrict the work to a subset of
    value heads / sequences (the other outputs stay zero).

    Returns ``o`` [B, T, H, V] and ``ht`` [N, H, K, V], both float64.
    """
    q, k, v, g, beta, h0 = map(_f64, (q, k, v, g, beta, h0))
    B, T, Hg, K = q.shape
    H, V = v.shape[2], v.shape[3]
    if H % Hg:
        raise ValueError("H must be a multiple of Hg")
    if scale is None:
        scale = 1.0 / math.sqrt(K)
    bounds = sequence_bounds(B, T, cu_seqlens)
    N = len(bounds)
    o = np.zeros((B, T, H, V))
    ht = np.zeros((N, H, K, V))
    head_list = range(H) if heads is None else heads
    seq_list = range(N) if seqs is None else seqs
    for n in seq_list:
        b, bos, eos = bounds[n]
        for h in head_list:
            hk = h // (H // Hg)
            S = np.zeros((V, K)) if h0 is None else h0[n, h].T.copy()
            gg = g[b, :, h]
            if g_is_cumsum:
                gg = raw_gate_from_chunk_cumsum(gg, bos, eos, chunk_size)
            for t in range(bos, eos):
                S = math.exp(gg[t]) * S
                kt = k[b, t, hk]
                pred = S @ kt
                delta = beta[b, t, h] * (v[b, t, h] - pred)
                S = S + np.outer(delta, kt)
                o[b, t, h] = scale * (S @ q[b, t, hk])
            ht[n, h] = S.T
    return o, ht


def kda_recurrent(q, k, v, g, beta, scale=None, h0=None, cu_seqlens=None,
                  g_is_cumsum=True, chunk_size=64, heads=None, seqs=None):
    """Per-channel-gate (KDA) forward, token by token.

    Shapes (vLLM kimi_k3 ``kda/chunk_intra`` page, kernel arguments; value head
    ``i_hv`` reads key head ``i_hv // (HV // H)``):
      q, k  [B, T, H, K];  v  [B, T, HV, V];  g  [B, T, HV, K];  beta  [B, T, HV]
      h0    [N, HV, K, V] or None
    ``g`` is the chunk-local cumulative sum of the per-channel log gates when
    ``g_is_cumsum`` (the default, as in that kernel), else the raw gates.

    Returns ``o`` [B, T, HV, V] and ``ht`` [N, HV, K, V], float64.
    """
    q, k, v, g, beta, h0 = map(_f64, (q, k, v, g, beta, h0))
    B, T, H, K = q.shape
    HV, V = v.shape[2], v.shape[3]
    if HV % H:
        raise ValueError("HV must be a multiple of H")
    if scale is None:
        scale = 1.0 / math.sqrt(K)
    bounds = sequence_bounds(B, T, cu_seqlens)
    N = len(bounds)
    o = np.zeros((B, T, HV, V))
    ht = np.zeros((N, HV, K, V))
    head_list = range(HV) if heads is None else heads
    seq_list = range(N) if seqs is None else seqs
    for n in seq_list:
        b, bos, eos = bounds[n]
        for hv in head_list:
            hk = hv // (HV // H)
            S = np.zeros((V, K)) if h0 is None else h0[n, hv].T.copy()
            gg = g[b, :, hv, :]
            if g_is_cumsum:
                gg = raw_gate_from_chunk_cumsum(gg, bos, eos, chunk_size)
            for t in range(bos, eos):
                S = S * np.exp(gg[t])[None, :]
                kt = k[b, t, hk]
                pred = S @ kt
                delta = beta[b, t, hv] * (v[b, t, hv] - pred)
                S = S + np.outer(delta, kt)
                o[b, t, hv] = scale * (S @ q[b, t, hk])
            ht[n, hv] = S.T
    return o, ht


def softplus(x, beta=1.0, threshold=20.0):
    """``(1/beta) log(1 + exp(beta x))``, or ``x`` once ``beta x > threshold``.

    FlashInfer ``gdn_decode_bf16_state.py``, ``compute_single_gate``.
    """
    bx = beta * x
    return np.where(bx <= threshold, np.log1p(np.exp(np.minimum(bx, threshold))) / beta, x)


def decode_gates(a, b, A_log, dt_bias, softplus_beta=1.0, softplus_threshold=20.0):
    """Decay log-gate ``g`` and write strength ``beta`` of the decode step.

    FlashInfer ``gdn_decode_bf16_state.py``, ``compute_single_gate``:
    ``g = -exp(A_log) * softplus(a + dt_bias)``, ``beta = sigmoid(b)``.
    ``a``, ``b`` are ``[B, T, HV]``; ``A_log``, ``dt_bias`` are ``[HV]``.
    """
    a, b, A_log, dt_bias = map(_f64, (a, b, A_log, dt_bias))
    x = a + dt_bias[None, None, :]
    g = -np.exp(A_log)[None, None, :] * softplus(x, softplus_beta, softplus_threshold)
    beta = 1.0 / (1.0 + np.exp(-b))
    return g, beta


def l2_normalize(x, eps=1e-6):
    """``x / sqrt(sum(x^2) + eps)`` over the last axis.

    FlashInfer ``gdn_decode_bf16_state.py``, ``normalize_and_store_qk_to_smem``
    (eps inside the square root; the public ``gated_delta_rule`` passes 1e-6).
    """
    x = _f64(x)
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps)


def gdn_decode(q, k, v, a, b, A_log, dt_bias, state, slot_indices=None, scale=None,
               softplus_beta=1.0, softplus_threshold=20.0, eps=1e-6, use_qk_l2norm=True):
    """Decode step for T = 1..4 tokens against a pooled state.

    FlashInfer ``gdn_decode_bf16_state.py``, public ``gated_delta_rule``:
      q, k  [B, T, H, K];  v  [B, T, HV, V];  a, b  [B, T, HV]
      A_log, dt_bias  [HV];  state  [pool, HV, V, K] (K fastest)
      slot_indices  [B] (identity when None)
    Value head ``hv`` reads key head ``hv // (HV // H)``.  ``q`` is
    L2-normalised and then multiplied by ``scale``; ``k`` is L2-normalised.

    Returns ``o`` [B, T, HV, V] and ``new_state`` [B, HV, V, K] (the state of
    each batch entry's slot after its T tokens, before any rounding).
    """
    q, k, v, state = map(_f64, (q, k, v, state))
    B, T, H, K = q.shape
    HV, V = v.shape[2], v.shape[3]
    if scale is None:
        scale = 1.0 / math.sqrt(K)
    if slot_indices is None:
        slot_indices = np.arange(B)
    slot_indices = [int(s) for s in np.asarray(slot_indices).reshape(-1)]
    g, beta = decode_gates(a, b, A_log, dt_bias, softplus_beta, softplus_threshold)
    if use_qk_l2norm:
        qn = l2_normalize(q, eps) * scale
        kn = l2_normalize(k, eps)
    else:
        qn = q * scale
        kn = k
    o = np.zeros((B, T, HV, V))
    new_state = np.zeros((B, HV, V, K))
    for bi in range(B):
        for hv in range(HV):
            hk = hv // (HV // H)
            S = state[slot_indices[bi], hv].copy()
            for t in range(T):
                S = math.exp(g[bi, t, hv]) * S
                pred = S @ kn[bi, t, hk]
                delta = beta[bi, t, hv] * (v[bi, t, hv] - pred)
                S = S + np.outer(delta, kn[bi, t, hk])
                o[bi, t, hv] = S @ qn[bi, t, hk]
            new_state[bi, hv] = S
    return o, new_state
