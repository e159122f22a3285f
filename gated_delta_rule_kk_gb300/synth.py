"""Seeded synthetic inputs for the chunked forward and the decode step.

This module only draws numbers: it holds none of the method's arithmetic and is
shared by the tests, the benchmark and the smoke check, which feed the same
tensors to the CUDA library and to the CPU oracle.  Every draw comes from
``numpy.random.default_rng(seed)`` in a fixed order and is cast to the storage
dtype after drawing.  Results are CPU torch tensors.

Workloads (named by what they are):

* ``tiny``    B=1, T=128, H=Hg=1, K=V=32, fp32, scalar gate, h0 = 0
* ``gdn``     B=2, T=4096, H=Hg=16, K=V=128, bf16 q/k/v, h0 ~ N(0, 0.1)
* ``varlen``  8 sequences, lengths ~ U[64, 8192] with total in [30000, 36000],
              Hg=4 key heads for H=16 value heads, K=V=128, bf16, h0 = 0
* ``kda``     B=1, T=8192, H=HV=32, K=V=128, bf16, per-channel gate given as
              the chunk-local cumulative sum (64-token chunks), h0 = 0
* ``decode``  B=pool=256, T in {1,2,4}, H=16, HV=32, K=V=128, bf16 state
              ~ N(0, 0.05)

Recipe shared by the prefill workloads: q, k ~ N(0, 1) then L2-normalised per
token (over K); v ~ N(0, 1); beta = sigmoid(N(0, 1)); per-token log-gate
g = logsigmoid(N(0, 1) + shift) with shift 3 (scalar gate) or 4 (per-channel).
"""
from __future__ import annotations

import numpy as np
import torch

GATE_SHIFT_SCALAR = 3.0
GATE_SHIFT_CHANNEL = 4.0


def _logsigmoid(x):
    return -np.logaddexp(0.0, -x)


def _sigmoid(x):
    return 1.0 / (1.0 + np.exp(-x))


def _unit_rows(x):
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True))


def _t(x, dtype):
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(dtype) if dtype != torch.float32 else t


def draw_lengths(rng, n=8, lo=64, hi=8192, total_lo=30000, total_hi=36000):
    """Sequence lengths ~ U[lo, hi], redrawn until their sum lies in range."""
    while True:
        lens = rng.integers(lo, hi + 1, size=n)
        if total_lo <= int(lens.sum()) <= total_hi:
            return [int(x) for x in lens]


def prefill_inputs(seed, B, T, H, Hg, K, V, dtype=torch.bfloat16, h0_std=None,
                   lengths=None, per_channel=False, g_shift=None, normalize=True,
                   chunk=64):
    """Inputs of one chunked-forward problem.

    ``lengths`` (list) makes a variable-length batch: B must be 1 and T their
    sum; ``cu_seqlens`` is returned.  ``per_channel`` draws a [B,T,H,K] gate
    and returns its chunk-local cumulative sum (chunks of ``chunk`` tokens
    counted from each sequence start); otherwise g is [B,T,H] and raw.
    Draw order: q, k, v, beta, g, h0.
    """
    rng = np.random.default_rng(seed)
    if lengths is not None:
        assert B == 1 and sum(lengths) == T
    q = rng.standard_normal((B, T, Hg, K))
    k = rng.standard_normal((B, T, Hg, K))
    if normalize:
        q, k = _unit_rows(q), _unit_rows(k)
    v = rng.standard_normal((B, T, H, V))
    beta = _sigmoid(rng.standard_normal((B, T, H)))
    if g_shift is None:
        g_shift = GATE_SHIFT_CHANNEL if per_channel else GATE_SHIFT_SCALAR
    gshape = (B, T, H, K) if per_channel else (B, T, H)
    g = _logsigmoid(rng.standard_normal(gshape) + g_shift)
    N = len(lengths) if lengths is not None else B
    h0 = None
    if h0_std is not None:
        h0 = rng.standard_normal((N, H, K, V)) * h0_std
    cu = None
    if lengths is not None:
        cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    if per_channel:
        # chunk-local inclusive cumulative sum along T, restarting every
        # `chunk` tokens from each sequence start (float32 like the interface)
        g = g.astype(np.float32)
        starts = cu[:-1] if cu is not None else [0]
        ends = cu[1:] if cu is not None else [T]
        out = np.empty_like(g)
        for s0, e0 in zip(starts, ends):
            for c in range(int(s0), int(e0), chunk):
                ce = min(c + chunk, int(e0))
                out[:, c:ce] = np.cumsum(g[:, c:ce], axis=1, dtype=np.float32)
        g = out
    res = {
        "q": _t(q, dtype), "k": _t(k, dtype), "v": _t(v, dtype),
        "g": _t(g, torch.float32), "beta": _t(beta, torch.float32),
        "h0": None if h0 is None else _t(h0, torch.float32),
        "cu_seqlens": None if cu is None else torch.from_numpy(cu),
        "scale": 1.0 / float(np.sqrt(K)),
        "g_is_cumsum": bool(per_channel),
        "dims": dict(B=B, T=T, H=H, Hg=Hg, K=K, V=V,
                     N=(len(lengths) if lengths is not None else B)),
    }
    return res


def decode_inputs(seed, B, T, H, HV, K, V, pool=None, state_std=0.05,
                  slots=None):
    """Inputs of one decode step.  Draw order: state, q, k, v, a, b, A_log, dt_bias."""
    rng = np.random.default_rng(seed)
    pool = B if pool is None else pool
    state = rng.standard_normal((pool, HV, V, K)) * state_std
    q = rng.standard_normal((B, T, H, K))
    k = rng.standard_normal((B, T, H, K))
    v = rng.standard_normal((B, T, HV, V))
    a = rng.standard_normal((B, T, HV))
    b = rng.standard_normal((B, T, HV))
    A_log = rng.standard_normal(HV)
    dt_bias = rng.standard_normal(HV)
    bf = torch.bfloat16
    return {
        "state": _t(state, bf), "q": _t(q, bf), "k": _t(k, bf), "v": _t(v, bf),
        "a": _t(a, bf), "b": _t(b, bf),
        "A_log": _t(A_log, torch.float32), "dt_bias": _t(dt_bias, torch.float32),
        "slot_indices": None if slots is None else torch.tensor(slots, dtype=torch.int32),
        "scale": 1.0 / float(np.sqrt(K)),
        "dims": dict(B=B, T=T, H=H, HV=HV, K=K, V=V, pool=pool),
    }


def _chunk_cumsum_gate(rng, gate, B, T, H, K, V, lengths, chunk):
    """Gate values of the state passes: logsigmoid(N(0, 1) + 3) rates, as
    chunk-local inclusive cumulative sums (fp32) except g_gamma."""
    if gate is None:
        return None
    shape = {"g": (B, T, H), "gk": (B, T, H, K), "gv": (B, T, H, V), "g_gamma": (H,)}
    raw = _logsigmoid(rng.standard_normal(shape[gate]) + GATE_SHIFT_SCALAR)
    if gate == "g_gamma":
        return raw
    cu = np.concatenate([[0], np.cumsum(lengths)]) if lengths is not None else [0, T]
    raw = raw.astype(np.float32)
    gv = np.empty_like(raw)
    for s0, e0 in zip(cu[:-1], cu[1:]):
        for c in range(int(s0), int(e0), chunk):
            ce = min(c + chunk, int(e0))
            gv[:, c:ce] = np.cumsum(raw[:, c:ce], axis=1, dtype=np.float32)
    return gv


def state_pass_inputs(seed, B, T, H, K, V, gate, dtype=torch.bfloat16, lengths=None,
                      h0_std=None, chunk=64):
    """Inputs of one chunk state pass (gated linear attention).

    k ~ N(0, 1) L2-normalised per token, v ~ N(0, 1); the gate's per-token
    rates are logsigmoid(N(0, 1) + 3) ("g": per token and head, "gk": per key
    channel, "gv": per value channel), given as chunk-local inclusive
    cumulative sums (chunks of ``chunk`` tokens from each sequence start);
    "g_gamma" is one logsigmoid(N(0, 1) + 3) per head; None draws no gate.
    Draw order: k, v, gate, h0.
    """
    rng = np.random.default_rng(seed)
    if lengths is not None:
        assert B == 1 and sum(lengths) == T
    k = _unit_rows(rng.standard_normal((B, T, H, K)))
    v = rng.standard_normal((B, T, H, V))
    gv = _chunk_cumsum_gate(rng, gate, B, T, H, K, V, lengths, chunk)
    N = len(lengths) if lengths is not None else B
    h0 = None if h0_std is None else rng.standard_normal((N, H, K, V)) * h0_std
    return {
        "k": _t(k, dtype), "v": _t(v, dtype), "gate": gate,
        "gate_values": None if gv is None else _t(gv, torch.float32),
        "h0": None if h0 is None else _t(h0, torch.float32),
        "cu_seqlens": None if lengths is None else torch.from_numpy(
            np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)),
        "dims": dict(B=B, T=T, H=H, K=K, V=V, N=N),
    }


# ---- the named workloads -------------------------------------------------

def tiny():
    return prefill_inputs(0, 1, 128, 1, 1, 32, 32, dtype=torch.float32)


def gdn_prefill():
    return prefill_inputs(1, 2, 4096, 16, 16, 128, 128, h0_std=0.1)


def varlen_gqa():
    lens = draw_lengths(np.random.default_rng(2))
    # lengths come from their own stream so the tensor draws below are stable
    return prefill_inputs(2, 1, sum(lens), 16, 4, 128, 128, lengths=lens)


def kda_prefill():
    return prefill_inputs(3, 1, 8192, 32, 32, 128, 128, per_channel=True)


def decode(T=1):
    return decode_inputs(4, 256, T, 16, 32, 128, 128)


WORKLOADS = {
    "tiny": tiny, "gdn": gdn_prefill, "varlen": varlen_gqa, "kda": kda_prefill,
}


def state_grad_inputs(seed, B, T, HQ, H, K, V, gate, dtype=torch.bfloat16, lengths=None,
                      dht_std=None, chunk=64):
    """Inputs of one backward state pass: q ~ N(0, 1) L2-normalised per token
    and do ~ N(0, 1) with HQ heads, the gate (as :func:`state_pass_inputs`)
    with H heads, dht ~ N(0, dht_std) [N, HQ, K, V] or None.
    Draw order: q, do, gate, dht.
    """
    rng = np.random.default_rng(seed)
    if lengths is not None:
        assert B == 1 and sum(lengths) == T
    q = _unit_rows(rng.standard_normal((B, T, HQ, K)))
    do = rng.standard_normal((B, T, HQ, V))
    gv = _chunk_cumsum_gate(rng, gate, B, T, H, K, V, lengths, chunk)
    N = len(lengths) if lengths is not None else B
    dht = None if dht_std is None else rng.standard_normal((N, HQ, K, V)) * dht_std
    return {
        "q": _t(q, dtype), "do": _t(do, dtype), "gate": gate,
        "gate_values": None if gv is None else _t(gv, torch.float32),
        "dht": None if dht is None else _t(dht, torch.float32),
        "cu_seqlens": None if lengths is None else torch.from_numpy(
            np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)),
        "scale": K ** -0.5,
        "dims": dict(B=B, T=T, HQ=HQ, H=H, K=K, V=V, N=N),
    }
