"""The oracle on every chain of a full-size workload, spread over the host cores.

Each (sequence, value head) chain of a prefill problem, and each slice of a
decode batch, is an independent call of the token-by-token definition; this
module slices the synthetic inputs per chain, runs the calls through
``oracle.parallel`` (spawn-started worker processes) and reassembles the
outputs in the layout the library writes.
"""
import numpy as np

from oracle import parallel


def _f32(x):
    return None if x is None else x.detach().cpu().float().numpy()


def prefill_all_chains(inp, kda=False, workers=None):
    """Oracle ``o`` [B,T,H,V] and ``ht`` [N,H,K,V] of a synth prefill problem."""
    q, k, v, g, beta, h0 = (_f32(inp[n]) for n in ("q", "k", "v", "g", "beta", "h0"))
    dm = inp["dims"]
    B, T, H, Hk, K, V, N = dm["B"], dm["T"], dm["H"], dm["Hg"], dm["K"], dm["V"], dm["N"]
    cu = inp["cu_seqlens"]
    if cu is None:
        bounds = [(b, 0, T) for b in range(B)]
    else:
        c = [int(x) for x in cu]
        bounds = [(0, c[n], c[n + 1]) for n in range(N)]
    specs, where = [], []
    for n, (b, s, e) in enumerate(bounds):
        for h in range(H):
            hk = h // (H // Hk)
            args = (q[b:b + 1, s:e, hk:hk + 1], k[b:b + 1, s:e, hk:hk + 1],
                    v[b:b + 1, s:e, h:h + 1], g[b:b + 1, s:e, h:h + 1],
                    beta[b:b + 1, s:e, h:h + 1])
            kw = dict(scale=inp["scale"], g_is_cumsum=inp["g_is_cumsum"],
                      h0=None if h0 is None else h0[n:n + 1, h:h + 1])
            specs.append(("kda_recurrent" if kda else "gdn_recurrent", args, kw))
            where.append((n, b, s, e, h))
    res = parallel.map_calls(specs, workers)
    o = np.zeros((B, T, H, V))
    ht = np.zeros((N, H, K, V))
    for (n, b, s, e, h), (oc, hc) in zip(where, res):
        o[b, s:e, h] = oc[0, :, 0]
        ht[n, h] = hc[0, 0]
    return o, ht


def decode_all_entries(inp, slice_len=16, workers=None, **kw):
    """Oracle ``o`` [B,T,HV,V] and new slot states [B,HV,V,K] of a synth decode
    problem, batch entries taken ``slice_len`` at a time."""
    q, k, v, a, b = (_f32(inp[n]) for n in ("q", "k", "v", "a", "b"))
    A_log, dt_bias, state = _f32(inp["A_log"]), _f32(inp["dt_bias"]), _f32(inp["state"])
    B = q.shape[0]
    slots = np.arange(B) if inp["slot_indices"] is None else inp["slot_indices"].numpy()
    specs = []
    for s in range(0, B, slice_len):
        e = min(B, s + slice_len)
        specs.append(("gdn_decode", (q[s:e], k[s:e], v[s:e], a[s:e], b[s:e], A_log, dt_bias,
                                     state[slots[s:e]], None), dict(scale=inp["scale"], **kw)))
    res = parallel.map_calls(specs, workers)
    return (np.concatenate([r[0] for r in res], axis=0),
            np.concatenate([r[1] for r in res], axis=0))
