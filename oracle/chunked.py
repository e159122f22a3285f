"""Independent fp64 chunked (WY) rewrite of the recurrence (test infrastructure).

Part of the oracle (test infrastructure only).  It is a second, algebraically
equivalent statement of the method that works one chunk of ``BT`` tokens at a
time, for any ``BT >= 1``.  Agreement with the token recurrence for every
``BT`` pins both, and it spells out the chunk algebra a chunked kernel follows.

Per chunk with chunk-local inclusive cumulative gate ``gamma`` (sglang
``fla/chunk_fwd.py``, fused KK^T + solve kernel, Steps 1-4; KDA ``chunk_h.py``,
``chunk_fwd_kernel_h``; vLLM kimi_k3 ``kda/chunk_intra``,
``chunk_kda_fwd_kernel_inter_solve_fused``), with the state ``h = S^T``
``[K, V]`` at the start of the chunk:

    A[i, j]   = beta_i sum_c k_i[c] k_j[c] exp(gamma_i[c] - gamma_j[c])   (i > j)
    Aqk[i, j] =        sum_c q_i[c] k_j[c] exp(gamma_i[c] - gamma_j[c])   (i >= j)
    T_inv     = (I + A)^{-1}                       (forward substitution)
    w         = T_inv diag(beta) (k * exp(gamma))  (WY recompute)
    u         = T_inv diag(beta) v
    v_new     = u - w h
    o         = scale ((q * exp(gamma)) h + Aqk v_new)
    h        <- diag(exp(gamma_L)) h + (k * exp(gamma_L - gamma))^T v_new

For the scalar gate the per-channel factors collapse to one value per token.
Entries outside the triangles are never formed, so no ``inf * 0`` arises.
"""
from __future__ import annotations

import math

import numpy as np

from .recurrence import _f64, raw_gate_from_chunk_cumsum, sequence_bounds


def unit_lower_inverse(A):
    """``(I + A)^{-1}`` for strictly lower-triangular ``A`` by forward substitution.

    Row ``i`` of the inverse is ``e_i - sum_{j<i} A[i, j] * row_j``: the scalar
    row recurrence of sglang ``fla/chunk_fwd.py`` Step 3, here over the whole
    chunk at once.
    """
    L = A.shape[0]
    Ti = np.zeros((L, L))
    for i in range(L):
        row = np.zeros(L)
        row[i] = 1.0
        for j in range(i):
            row -= A[i, j] * Ti[j]
        Ti[i] = row
    return Ti


def _chunk_step(h, qc, kc, vc, gc, bc, scale):
    """One chunk.  gc is the raw log-gate per token, [L] or [L, K]."""
    L, K = kc.shape
    gamma = np.cumsum(gc, axis=0)
    if gamma.ndim == 1:
        gamma = np.repeat(gamma[:, None], K, axis=1)
    A = np.zeros((L, L))
    Aqk = np.zeros((L, L))
    for i in range(L):
        for j in range(i + 1):
            f = np.exp(gamma[i] - gamma[j])
            Aqk[i, j] = np.sum(qc[i] * kc[j] * f)
            if j < i:
                A[i, j] = bc[i] * np.sum(kc[i] * kc[j] * f)
    Ti = unit_lower_inverse(A)
    w = Ti @ (bc[:, None] * kc * np.exp(gamma))
    u = Ti @ (bc[:, None] * vc)
    v_new = u - w @ h
    o = scale * ((qc * np.exp(gamma)) @ h + Aqk @ v_new)
    gL = gamma[L - 1]
    h_next = np.exp(gL)[:, None] * h + (kc * np.exp(gL[None, :] - gamma)).T @ v_new
    return o, h_next


def chunked_forward(q, k, v, g, beta, BT, scale=None, h0=None, cu_seqlens=None,
                    g_is_cumsum=False, cumsum_chunk=64, per_channel=False):
    """Chunked forward for either gate kind.

    Same shapes and conventions as ``recurrence.gdn_recurrent`` (scalar gate,
    ``per_channel=False``: g [B, T, H]) or ``recurrence.kda_recurrent``
    (``per_channel=True``: g [B, T, HV, K]).  ``BT`` is this rewrite's chunk
    length; ``cumsum_chunk`` is the chunking that a cumulative ``g`` refers to.
    """
    q, k, v, g, beta, h0 = map(_f64, (q, k, v, g, beta, h0))
    B, T, Hk, K = q.shape
    H, V = v.shape[2], v.shape[3]
    if scale is None:
        scale = 1.0 / math.sqrt(K)
    bounds = sequence_bounds(B, T, cu_seqlens)
    N = len(bounds)
    o = np.zeros((B, T, H, V))
    ht = np.zeros((N, H, K, V))
    for n, (b, bos, eos) in enumerate(bounds):
        for h in range(H):
            hk = h // (H // Hk)
            gg = g[b, :, h, :] if per_channel else g[b, :, h]
            if g_is_cumsum:
                gg = raw_gate_from_chunk_cumsum(gg, bos, eos, cumsum_chunk)
            st = np.zeros((K, V)) if h0 is None else h0[n, h].copy()
            for s in range(bos, eos, BT):
                e = min(s + BT, eos)
                oc, st = _chunk_step(st, q[b, s:e, hk], k[b, s:e, hk], v[b, s:e, h],
                                     gg[s:e], beta[b, s:e, h], scale)
                o[b, s:e, h] = oc
            ht[n, h] = st
    return o, ht
