"""Chunk state pass of gated linear attention, token by token, fp64.

This module is part of the oracle, which is test infrastructure: only tests,
the smoke check and the CPU legs of the benchmark use it.  It shares no code
with the CUDA library.

The KDA ``_fla/ops/common/chunk_h.py`` page (``chunk_fwd_kernel_h`` and its
host wrapper ``chunk_fwd_h``) computes, for every sequence and head, the state
``h`` (``[K, V]``) at the start of every chunk of ``chunk_size`` tokens and,
optionally, the final state, for the gated linear-attention recurrence

    h <- decay_t(h) + k_t v_t^T          (token t, after the decay)

with one of these decays (the page's kernel works in base 2; the gates here
are natural logarithms, as everywhere in this library):

    "g"        e^{r_t} h            r_t per token and head
    "g_gamma"  e^{gamma_h} h        one rate per head, the same for every token
    "gk"       diag(e^{r_t}) h      r_t per token, head and key channel
    "gv"       h diag(e^{r_t})      r_t per token, head and value channel
    None       h                    no decay

The per-token gates ``g``, ``gk``, ``gv`` are taken the way the page's kernel
takes them: as inclusive cumulative sums inside each chunk (chunks counted
from each sequence's first token); the raw per-token rate ``r_t`` is recovered
by differencing inside a chunk.  ``g_gamma`` is the raw rate itself (the
page's kernel forms the in-chunk cumulative sum ``gamma * (i + 1)``).

Output layout: the chunk states of all sequences one after another, sequence
n contributing ceil(len_n / chunk_size) entries -- for B equal sequences of T
tokens that is ``[B, NT, H, K, V]`` flattened over (B, NT).  With the page's
``split_size`` (a multiple of the chunk size) only the chunks whose index is
a multiple of split_size / chunk_size are stored, at index chunk // (split_size
/ chunk_size): ceil(len_n / split_size) entries per sequence.
"""
from __future__ import annotations

import numpy as np

from .recurrence import _f64, raw_gate_from_chunk_cumsum, sequence_bounds

GATES = (None, "g", "g_gamma", "gk", "gv")


def chunk_counts(B: int, T: int, cu_seqlens=None, chunk_size: int = 64, split_size=None):
    """Number of stored states of every sequence (0 for an empty one): one per
    chunk, or one per split of ``split_size`` tokens."""
    span = chunk_size if split_size is None else split_size
    return [-(-(eos - bos) // span) for _, bos, eos in sequence_bounds(B, T, cu_seqlens)]


def _split(chunk_size, split_size):
    if split_size is None:
        return 1
    if split_size <= 0 or split_size % chunk_size:
        raise ValueError("split_size must be a positive multiple of chunk_size")
    return split_size // chunk_size


def chunk_state_pass(k, v, gate=None, gate_values=None, h0=None, cu_seqlens=None,
                     chunk_size: int = 64, split_size=None, state_v_first: bool = False):
    """Chunk-start states ``hs`` ``[sum NT_n, H, K, V]`` and final states
    ``ht`` ``[N, H, K, V]`` of the gated linear-attention recurrence.

    k ``[B, T, H, K]``, v ``[B, T, H, V]``; gate_values: ``g`` ``[B, T, H]``,
    ``g_gamma`` ``[H]``, ``gk`` ``[B, T, H, K]``, ``gv`` ``[B, T, H, V]``
    (chunk-local cumulative sums except ``g_gamma``); h0 ``[N, H, K, V]`` or
    None (zeros); split_size stores every (split_size / chunk_size)-th chunk.
    With state_v_first every state (h0 in, hs and ht out) is [.., V, K]: the
    page's layout flag, which transposes the stored states and nothing else.
    """
    NTS = _split(chunk_size, split_size)
    if gate not in GATES:
        raise ValueError(f"unknown gate {gate!r}")
    k, v = _f64(k), _f64(v)
    B, T, H, K = k.shape
    V = v.shape[3]
    gv_ = _f64(gate_values)
    seqs = sequence_bounds(B, T, cu_seqlens)
    N = len(seqs)
    h0 = np.zeros((N, H, K, V)) if h0 is None else _f64(h0)
    if state_v_first:
        h0 = h0.swapaxes(-1, -2)
    counts = chunk_counts(B, T, cu_seqlens, chunk_size, split_size)
    hs = np.zeros((sum(counts), H, K, V))
    ht = np.zeros((N, H, K, V))
    first = 0
    for n, (b, bos, eos) in enumerate(seqs):
        raw = None
        if gate in ("g", "gk", "gv"):
            raw = raw_gate_from_chunk_cumsum(gv_[b], bos, eos, chunk_size)
        for h in range(H):
            S = h0[n, h].copy()
            for t in range(bos, eos):
                i = t - bos
                if i % chunk_size == 0 and (i // chunk_size) % NTS == 0:
                    hs[first + i // chunk_size // NTS, h] = S
                if gate == "g":
                    S = np.exp(raw[t, h]) * S
                elif gate == "g_gamma":
                    S = np.exp(gv_[h]) * S
                elif gate == "gk":
                    S = np.exp(raw[t, h])[:, None] * S
                elif gate == "gv":
                    S = S * np.exp(raw[t, h])[None, :]
                S = S + np.outer(k[b, t, h], v[b, t, h])
            ht[n, h] = S
        first += counts[n]
    if state_v_first:
        return hs.swapaxes(-1, -2), ht.swapaxes(-1, -2)
    return hs, ht


def chunk_state_grad(q, do, gate=None, gate_values=None, dht=None, cu_seqlens=None,
                     scale=None, chunk_size: int = 64, split_size=None,
                     state_v_first: bool = False):
    """Backward state pass (the chunk_h page's ``chunk_bwd_kernel_dh``).

    For the gated linear attention above with outputs o_t = scale S_t^T q_t
    (S_t the state after token t), the gradient G_t = dL/dS_t of a loss with
    dL/do_t = do_t obeys, going backwards,

        G <- G + scale q_t do_t^T      (token t's output)
        G <- decay_t^T(G)              (to the state before token t)

    starting from G = dht after the last token.  Returns ``dh``
    ``[sum NT_n, HQ, K, V]``, the gradient with respect to the state at the
    end of every chunk (taken before that chunk's tokens are folded in), and
    ``dh0`` ``[N, HQ, K, V]``.  q ``[B, T, HQ, K]``, do ``[B, T, HQ, V]``;
    the gate has H heads (HQ a multiple of H, query head hq uses gate head
    hq // (HQ / H)), given as in :func:`chunk_state_pass`.  With split_size
    only chunks whose index is a multiple of split_size / chunk_size are
    stored, at index chunk // (split_size / chunk_size).  state_v_first: dht,
    dh and dh0 are [.., V, K], as in :func:`chunk_state_pass`.
    """
    NTS = _split(chunk_size, split_size)
    if gate not in GATES:
        raise ValueError(f"unknown gate {gate!r}")
    q, do = _f64(q), _f64(do)
    B, T, HQ, K = q.shape
    V = do.shape[3]
    scale = 1.0 / np.sqrt(K) if scale is None else float(scale)
    gv_ = _f64(gate_values)
    if gate is None:
        H = HQ
    elif gate == "g_gamma":
        H = gv_.shape[0]
    else:
        H = gv_.shape[2]
    group = HQ // H
    seqs = sequence_bounds(B, T, cu_seqlens)
    N = len(seqs)
    dht = np.zeros((N, HQ, K, V)) if dht is None else _f64(dht)
    if state_v_first:
        dht = dht.swapaxes(-1, -2)
    counts = chunk_counts(B, T, cu_seqlens, chunk_size, split_size)
    dh = np.zeros((sum(counts), HQ, K, V))
    dh0 = np.zeros((N, HQ, K, V))
    first = 0
    for n, (b, bos, eos) in enumerate(seqs):
        raw = None
        if gate in ("g", "gk", "gv"):
            raw = raw_gate_from_chunk_cumsum(gv_[b], bos, eos, chunk_size)
        for hq in range(HQ):
            h = hq // group
            G = dht[n, hq].copy()
            for t in range(eos - 1, bos - 1, -1):
                i = t - bos
                if ((i % chunk_size == chunk_size - 1 or t == eos - 1)
                        and (i // chunk_size) % NTS == 0):
                    dh[first + i // chunk_size // NTS, hq] = G
                G = G + scale * np.outer(q[b, t, hq], do[b, t, hq])
                if gate == "g":
                    G = np.exp(raw[t, h]) * G
                elif gate == "g_gamma":
                    G = np.exp(gv_[h]) * G
                elif gate == "gk":
                    G = np.exp(raw[t, h])[:, None] * G
                elif gate == "gv":
                    G = G * np.exp(raw[t, h])[None, :]
            dh0[n, hq] = G
        first += counts[n]
    if state_v_first:
        return dh.swapaxes(-1, -2), dh0.swapaxes(-1, -2)
    return dh, dh0
