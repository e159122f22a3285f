"""Python entry points with the C names: torch tensors in, library call, tensors out.

Only argument marshalling happens here (shape reading, dtype/contiguity
checks, output allocation through PyTorch's caching allocator, the current
stream).  All arithmetic runs in the CUDA library.
"""
from __future__ import annotations

import ctypes

import torch

from . import _lib
from ._lib import (DType, GateKind, GdnChunkArgs, GdnDecodeArgs, GdnStateArgs, GdnStateBwdArgs,
                   KdaChunkArgs)

CHUNK = 64


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _need(t, name, dtypes, device):
    if t is None:
        raise ValueError(f"{name} is required")
    if not t.is_cuda or t.device != device:
        raise ValueError(f"{name} must be a CUDA tensor on {device}")
    if t.dtype not in dtypes:
        raise ValueError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _io_dtype(q):
    if q.dtype == torch.bfloat16:
        return DType.BF16, (torch.bfloat16,)
    if q.dtype == torch.float32:
        return DType.F32, (torch.float32,)
    raise ValueError(f"q/k/v must be float32 or bfloat16, got {q.dtype}")


def _out_fp32(q, out_dtype):
    """Whether o is written as float32: out_dtype None means q's dtype."""
    if out_dtype is None or out_dtype == q.dtype:
        return q.dtype == torch.float32
    if out_dtype == torch.float32:
        return True
    raise ValueError(f"out_dtype must be None, {q.dtype} or torch.float32")


def _chunk_common(q, k, v, g, beta, initial_state, cu_seqlens, output_final_state, out,
                  final_state, value_heads_name, state_v_first=False, out_dtype=None):
    dev = q.device
    dt, dts = _io_dtype(q)
    _need(q, "q", dts, dev)
    _need(k, "k", dts, dev)
    _need(v, "v", dts, dev)
    _need(g, "g", (torch.float32,), dev)
    _need(beta, "beta", (torch.float32,), dev)
    B, T, Hk, K = q.shape
    Hv, V = v.shape[2], v.shape[3]
    if k.shape != q.shape or v.shape[:2] != (B, T):
        raise ValueError("q, k must be [B,T,Hk,K] and v [B,T,Hv,V]")
    if cu_seqlens is not None:
        _need(cu_seqlens, "cu_seqlens", (torch.int32,), dev)
        N = cu_seqlens.numel() - 1
    else:
        N = B
    SK, SV = (V, K) if state_v_first else (K, V)
    if initial_state is not None:
        _need(initial_state, "initial_state", (torch.float32,), dev)
        if tuple(initial_state.shape) != (N, Hv, SK, SV):
            raise ValueError(f"initial_state must be [{N},{Hv},{SK},{SV}]")
    odt = torch.float32 if _out_fp32(q, out_dtype) else q.dtype
    if out is None:
        out = torch.empty((B, T, Hv, V), dtype=odt, device=dev)
    else:
        _need(out, "out", (odt,), dev)
    if output_final_state and final_state is None:
        final_state = torch.empty((N, Hv, SK, SV), dtype=torch.float32, device=dev)
    elif final_state is not None:
        _need(final_state, "final_state", (torch.float32,), dev)
    return dt, (B, T, Hk, Hv, K, V, N), out, final_state


def _attach_workspace(args, size_fn, workspace, device):
    """Ask the library how much scratch the call needs and hand it a buffer
    (from PyTorch's caching allocator unless the caller passes one)."""
    lib = _lib.load()
    n = ctypes.c_size_t(0)
    _lib.check(size_fn(lib)(ctypes.byref(args), ctypes.byref(n)), "workspace_size")
    if n.value == 0:
        return None
    if workspace is None:
        workspace = torch.empty(n.value, dtype=torch.uint8, device=device)
    elif workspace.numel() * workspace.element_size() < n.value or not workspace.is_cuda:
        raise ValueError(f"workspace needs {n.value} bytes on the GPU")
    args.workspace = ctypes.c_void_p(workspace.data_ptr())
    args.workspace_bytes = workspace.numel() * workspace.element_size()
    return workspace


def gdn_chunk_fwd(q, k, v, g, beta, scale=None, initial_state=None, cu_seqlens=None,
                  output_final_state=True, g_is_cumsum=False, out=None, final_state=None,
                  workspace=None, stream=None, state_v_first=False, out_dtype=None, segments=0):
    """GDN chunked forward.  Returns ``(o, ht)`` (``ht`` None if not requested).

    q, k [B,T,Hg,K]; v [B,T,H,V]; g, beta [B,T,H] float32; initial_state
    [N,H,K,V] float32 ([N,H,V,K] with ``state_v_first``, as ``ht``);
    cu_seqlens [N+1] int32 (then B == 1).  ``out_dtype=torch.float32`` writes
    o in float32 (the value a bf16 o is the round-to-nearest-even of).
    ``segments``: the state pass's segment count (0 = the library's choice,
    1 = one sequential chain per sequence, >= 2 = segment-parallel).
    """
    dt, (B, T, Hg, H, K, V, N), out, ht = _chunk_common(
        q, k, v, g, beta, initial_state, cu_seqlens, output_final_state, out, final_state, "H",
        state_v_first, out_dtype)
    a = GdnChunkArgs(dtype=int(dt), q=_ptr(q), k=_ptr(k), v=_ptr(v), g=_ptr(g), beta=_ptr(beta),
                     h0=_ptr(initial_state), ht=_ptr(ht), o=_ptr(out), cu_seqlens=_ptr(cu_seqlens),
                     B=B, T=T, H=H, Hg=Hg, K=K, V=V, N=N, chunk_size=CHUNK,
                     g_is_cumsum=int(bool(g_is_cumsum)), state_v_first=int(bool(state_v_first)),
                     o_fp32=int(out.dtype == torch.float32), segments=int(segments),
                     scale=float(scale) if scale is not None else 0.0,
                     workspace=None, workspace_bytes=0)
    ws = _attach_workspace(a, lambda lib: lib.gdn_chunk_workspace_size, workspace, q.device)
    lib = _lib.load()
    _lib.check(lib.gdn_chunk_fwd(ctypes.byref(a), _stream(stream)), "gdn_chunk_fwd")
    del ws  # the caching allocator keeps it valid for work already on `stream`
    return out, ht


def gdn_chunk_segment_count(B, T, H, Hg, K, V, N=None, dtype=torch.bfloat16, varlen=False,
                            segments=0):
    """Segments per sequence the state pass of ``gdn_chunk_fwd`` uses for
    these sizes (1: one sequential chain per sequence)."""
    dt = DType.BF16 if dtype == torch.bfloat16 else DType.F32
    a = GdnChunkArgs(dtype=int(dt), B=B, T=T, H=H, Hg=Hg, K=K, V=V, N=N or B, chunk_size=CHUNK,
                     segments=int(segments),
                     cu_seqlens=ctypes.c_void_p(16) if varlen else None)
    n = ctypes.c_int32(0)
    _lib.check(_lib.load().gdn_chunk_segment_count(ctypes.byref(a), ctypes.byref(n)),
               "gdn_chunk_segment_count")
    return n.value


def _need_host(t, name, dtypes):
    if t is None:
        raise ValueError(f"{name} is required")
    if t.device.type != "cpu":
        raise ValueError(f"{name} must be a CPU tensor")
    if t.dtype not in dtypes:
        raise ValueError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def gdn_chunk_fwd_host(q, k, v, g, beta, scale=None, initial_state=None, cu_seqlens=None,
                       output_final_state=True, g_is_cumsum=False, out=None, final_state=None,
                       workspace=None, stream=None, device=None, state_v_first=False,
                       out_dtype=None):
    """``gdn_chunk_fwd`` from and to host memory, copies included.

    Every tensor is a CPU tensor (pinned ones copy asynchronously and fastest);
    the library copies them to ``workspace`` (a CUDA uint8 tensor, allocated on
    ``device`` if not passed), runs the forward and copies ``o`` and ``ht``
    back, piece by piece so that copies overlap the kernels.  Everything is
    enqueued on ``stream``; the host outputs are complete once it has
    completed.  Returns ``(o, ht)`` as CPU tensors.
    """
    dt, dts = _io_dtype(q)
    for t, name in ((q, "q"), (k, "k"), (v, "v")):
        _need_host(t, name, dts)
    _need_host(g, "g", (torch.float32,))
    _need_host(beta, "beta", (torch.float32,))
    B, T, Hg, K = q.shape
    H, V = v.shape[2], v.shape[3]
    if k.shape != q.shape or v.shape[:2] != (B, T):
        raise ValueError("q, k must be [B,T,Hg,K] and v [B,T,H,V]")
    N = B
    if cu_seqlens is not None:
        _need_host(cu_seqlens, "cu_seqlens", (torch.int32,))
        N = cu_seqlens.numel() - 1
    SK, SV = (V, K) if state_v_first else (K, V)
    if initial_state is not None:
        _need_host(initial_state, "initial_state", (torch.float32,))
        if tuple(initial_state.shape) != (N, H, SK, SV):
            raise ValueError(f"initial_state must be [{N},{H},{SK},{SV}]")
    odt = torch.float32 if _out_fp32(q, out_dtype) else q.dtype
    if out is None:
        out = torch.empty((B, T, H, V), dtype=odt, pin_memory=True)
    else:
        _need_host(out, "out", (odt,))
    if output_final_state and final_state is None:
        final_state = torch.empty((N, H, SK, SV), dtype=torch.float32, pin_memory=True)
    elif final_state is not None:
        _need_host(final_state, "final_state", (torch.float32,))
    a = GdnChunkArgs(dtype=int(dt), q=_ptr(q), k=_ptr(k), v=_ptr(v), g=_ptr(g), beta=_ptr(beta),
                     h0=_ptr(initial_state), ht=_ptr(final_state), o=_ptr(out),
                     cu_seqlens=_ptr(cu_seqlens), B=B, T=T, H=H, Hg=Hg, K=K, V=V, N=N,
                     chunk_size=CHUNK, g_is_cumsum=int(bool(g_is_cumsum)),
                     state_v_first=int(bool(state_v_first)), o_fp32=int(odt == torch.float32),
                     scale=float(scale) if scale is not None else 0.0,
                     workspace=None, workspace_bytes=0)
    lib = _lib.load()
    n = ctypes.c_size_t(0)
    _lib.check(lib.gdn_chunk_host_workspace_size(ctypes.byref(a), ctypes.byref(n)),
               "gdn_chunk_host_workspace_size")
    if device is None:
        device = stream.device if stream is not None else torch.device("cuda", torch.cuda.current_device())
    if workspace is None:
        workspace = torch.empty(n.value, dtype=torch.uint8, device=device)
    elif not workspace.is_cuda or workspace.numel() * workspace.element_size() < n.value:
        raise ValueError(f"workspace needs {n.value} bytes on the GPU")
    a.workspace = ctypes.c_void_p(workspace.data_ptr())
    a.workspace_bytes = workspace.numel() * workspace.element_size()
    with torch.cuda.device(workspace.device):
        _lib.check(lib.gdn_chunk_fwd_host(ctypes.byref(a), _stream(stream)), "gdn_chunk_fwd_host")
    del workspace  # the caching allocator keeps it valid for work already on `stream`
    return out, final_state


def gdn_chunk_host_workspace_bytes(q, v, cu_seqlens=None, Hg=None):
    """Device workspace ``gdn_chunk_fwd_host`` needs for q [B,T,Hg,K] and
    v [B,T,H,V] (CPU tensors; only their shapes and dtype are read) and, with
    packed sequences, the CPU int32 ``cu_seqlens``."""
    dt, _ = _io_dtype(q)
    B, T, hg, K = q.shape
    H, V = v.shape[2], v.shape[3]
    N = cu_seqlens.numel() - 1 if cu_seqlens is not None else B
    a = GdnChunkArgs(dtype=int(dt), q=None, k=None, v=None, g=None, beta=None, h0=None, ht=None,
                     o=None, cu_seqlens=_ptr(cu_seqlens), B=B, T=T, H=H, Hg=Hg or hg, K=K, V=V,
                     N=N, chunk_size=CHUNK, g_is_cumsum=0, scale=0.0, workspace=None,
                     workspace_bytes=0)
    n = ctypes.c_size_t(0)
    _lib.check(_lib.load().gdn_chunk_host_workspace_size(ctypes.byref(a), ctypes.byref(n)),
               "gdn_chunk_host_workspace_size")
    return n.value


def gdn_chunk_fwd_noalloc(q, k, v, g, beta, scale=None, initial_state=None, cu_seqlens=None,
                          output_final_state=True, g_is_cumsum=False, out=None,
                          final_state=None, stream=None, state_v_first=False, out_dtype=None):
    """``gdn_chunk_fwd`` for callers that cannot allocate device memory.

    No workspace is requested or allocated: the library uses a fixed device
    array of ``gdn_noalloc_scratch_bytes()`` bytes instead, shared by every
    call on the device (order calls that could overlap).  Outputs are
    allocated here only when ``out`` / ``final_state`` are not passed.
    """
    dt, (B, T, Hg, H, K, V, N), out, ht = _chunk_common(
        q, k, v, g, beta, initial_state, cu_seqlens, output_final_state, out, final_state, "H",
        state_v_first, out_dtype)
    a = GdnChunkArgs(dtype=int(dt), q=_ptr(q), k=_ptr(k), v=_ptr(v), g=_ptr(g), beta=_ptr(beta),
                     h0=_ptr(initial_state), ht=_ptr(ht), o=_ptr(out), cu_seqlens=_ptr(cu_seqlens),
                     B=B, T=T, H=H, Hg=Hg, K=K, V=V, N=N, chunk_size=CHUNK,
                     g_is_cumsum=int(bool(g_is_cumsum)), state_v_first=int(bool(state_v_first)),
                     o_fp32=int(out.dtype == torch.float32), scale=float(scale) if scale is not None else 0.0,
                     workspace=None, workspace_bytes=0)
    lib = _lib.load()
    _lib.check(lib.gdn_chunk_fwd_noalloc(ctypes.byref(a), _stream(stream)),
               "gdn_chunk_fwd_noalloc")
    return out, ht


def gdn_noalloc_scratch_bytes():
    """Size of the fixed scratch array behind ``gdn_chunk_fwd_noalloc``."""
    return int(_lib.load().gdn_noalloc_scratch_bytes())


def kda_chunk_fwd(q, k, v, g, beta, scale=None, initial_state=None, cu_seqlens=None,
                  output_final_state=True, g_is_cumsum=True, out=None, final_state=None,
                  workspace=None, stream=None, state_v_first=False, out_dtype=None, segments=0):
    """KDA chunked forward.  Returns ``(o, ht)``.

    q, k [B,T,H,K]; v [B,T,HV,V]; g [B,T,HV,K] float32 (chunk-local cumsum
    when g_is_cumsum); beta [B,T,HV]; initial_state [N,HV,K,V] float32
    ([N,HV,V,K] with ``state_v_first``, as ``ht``).
    """
    dt, (B, T, H, HV, K, V, N), out, ht = _chunk_common(
        q, k, v, g, beta, initial_state, cu_seqlens, output_final_state, out, final_state, "HV",
        state_v_first, out_dtype)
    a = KdaChunkArgs(dtype=int(dt), q=_ptr(q), k=_ptr(k), v=_ptr(v), g=_ptr(g), beta=_ptr(beta),
                     h0=_ptr(initial_state), ht=_ptr(ht), o=_ptr(out), cu_seqlens=_ptr(cu_seqlens),
                     B=B, T=T, H=H, HV=HV, K=K, V=V, N=N, chunk_size=CHUNK,
                     g_is_cumsum=int(bool(g_is_cumsum)), state_v_first=int(bool(state_v_first)),
                     o_fp32=int(out.dtype == torch.float32), segments=int(segments),
                     scale=float(scale) if scale is not None else 0.0,
                     workspace=None, workspace_bytes=0)
    ws = _attach_workspace(a, lambda lib: lib.kda_chunk_workspace_size, workspace, q.device)
    lib = _lib.load()
    _lib.check(lib.kda_chunk_fwd(ctypes.byref(a), _stream(stream)), "kda_chunk_fwd")
    del ws
    return out, ht


def gdn_decode(q, k, v, a, b, A_log, dt_bias, state, slot_indices=None, scale=None,
               softplus_beta=1.0, softplus_threshold=20.0, eps=1e-6, use_qk_l2norm=True,
               out=None, stream=None, out_dtype=None, new_state_f32=None):
    """Decode T = 1..4 tokens; ``state`` [pool,HV,V,K] bf16 is updated in place.  Returns o.

    ``out_dtype=torch.float32`` writes o in float32; ``new_state_f32`` (a
    [B,HV,V,K] float32 tensor) receives each entry's updated state before its
    rounding into the bf16 pool.
    """
    dev = q.device
    bf = (torch.bfloat16,)
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (a, "a"), (b, "b"), (state, "state")):
        _need(t, n, bf, dev)
    _need(A_log, "A_log", (torch.float32,), dev)
    _need(dt_bias, "dt_bias", (torch.float32,), dev)
    if slot_indices is not None:
        _need(slot_indices, "slot_indices", (torch.int32,), dev)
    B, T, H, K = q.shape
    HV, V = v.shape[2], v.shape[3]
    pool = state.shape[0]
    odt = torch.float32 if _out_fp32(q, out_dtype) else torch.bfloat16
    if out is None:
        out = torch.empty((B, T, HV, V), dtype=odt, device=dev)
    else:
        _need(out, "out", (odt,), dev)
    if new_state_f32 is not None:
        _need(new_state_f32, "new_state_f32", (torch.float32,), dev)
        if tuple(new_state_f32.shape) != (B, HV, V, K):
            raise ValueError(f"new_state_f32 must be [{B},{HV},{V},{K}]")
    args = GdnDecodeArgs(q=_ptr(q), k=_ptr(k), v=_ptr(v), a=_ptr(a), b=_ptr(b),
                         A_log=_ptr(A_log), dt_bias=_ptr(dt_bias), state=_ptr(state),
                         slot_indices=_ptr(slot_indices), o=_ptr(out),
                         new_state_f32=_ptr(new_state_f32),
                         B=B, T=T, H=H, HV=HV, K=K, V=V, pool=pool,
                         use_qk_l2norm=int(bool(use_qk_l2norm)),
                         o_fp32=int(odt == torch.float32),
                         scale=float(scale) if scale is not None else 0.0,
                         softplus_beta=float(softplus_beta),
                         softplus_threshold=float(softplus_threshold), eps=float(eps))
    lib = _lib.load()
    _lib.check(lib.gdn_decode(ctypes.byref(args), _stream(stream)), "gdn_decode")
    return out


def gdn_check_device_error(stream=None):
    """Synchronise ``stream`` and return (and clear) the device error word as a Status."""
    code = ctypes.c_int32(0)
    lib = _lib.load()
    _lib.check(lib.gdn_check_device_error(_stream(stream), ctypes.byref(code)),
               "gdn_check_device_error")
    return _lib.Status(code.value)


_GATES = {None: GateKind.NONE, "g": GateKind.G, "g_gamma": GateKind.G_GAMMA, "gk": GateKind.GK,
          "gv": GateKind.GV}


def _stored_states(B, T, cu_seqlens, split):
    """Number of stored states: ceil(len / split) per sequence (a device sync
    with cu_seqlens)."""
    if cu_seqlens is None:
        return B * ((T + split - 1) // split)
    lens = (cu_seqlens[1:] - cu_seqlens[:-1]).clamp(min=0).to(torch.int64)
    return int(((lens + split - 1) // split).sum().item())


def _split_tokens(split_size):
    split = CHUNK if not split_size else int(split_size)
    if split <= 0 or split % CHUNK:
        raise ValueError(f"split_size must be a positive multiple of {CHUNK}")
    return split


def gdn_chunk_state_fwd(k, v, gate=None, gate_values=None, initial_state=None, cu_seqlens=None,
                        output_final_state=True, output_states=True,
                        states_dtype=torch.float32, out_states=None, final_state=None,
                        num_chunks=None, split_size=None, state_v_first=False, stream=None):
    """Chunk state pass of gated linear attention.  Returns ``(hs, ht)``.

    k [B,T,H,K], v [B,T,H,V] (float32 or bfloat16); gate one of None, "g"
    ([B,T,H]), "g_gamma" ([H]), "gk" ([B,T,H,K]), "gv" ([B,T,H,V]) with
    ``gate_values`` float32 (chunk-local cumulative sums except g_gamma);
    initial_state [N,H,K,V] float32.  hs holds the state at the start of every
    split of ``split_size`` tokens (a multiple of 64; default 64: every
    chunk), sequence after sequence ([C,H,K,V]); with ``cu_seqlens`` and no
    ``num_chunks``, C is read from the lengths (a device sync).  With
    ``state_v_first`` every state (initial_state, hs, ht) is [.., V, K].
    """
    split = _split_tokens(split_size)
    dev = k.device
    dt, dts = _io_dtype(k)
    _need(k, "k", dts, dev)
    _need(v, "v", dts, dev)
    if gate not in _GATES:
        raise ValueError(f"gate must be one of {list(_GATES)}")
    if gate is not None:
        _need(gate_values, "gate_values", (torch.float32,), dev)
    B, T, H, K = k.shape
    V = v.shape[3]
    if v.shape[:3] != (B, T, H):
        raise ValueError("k must be [B,T,H,K] and v [B,T,H,V]")
    if cu_seqlens is not None:
        _need(cu_seqlens, "cu_seqlens", (torch.int32,), dev)
        N = cu_seqlens.numel() - 1
    else:
        N = B
    if num_chunks is None and (output_states or out_states is not None or cu_seqlens is None):
        num_chunks = _stored_states(B, T, cu_seqlens, split)
    SK, SV = (V, K) if state_v_first else (K, V)
    if initial_state is not None:
        _need(initial_state, "initial_state", (torch.float32,), dev)
        if tuple(initial_state.shape) != (N, H, SK, SV):
            raise ValueError(f"initial_state must be [{N},{H},{SK},{SV}]")
    hs = out_states
    if hs is None and output_states:
        hs = torch.empty((num_chunks, H, SK, SV), dtype=states_dtype, device=dev)
    if hs is not None:
        _need(hs, "out_states", (torch.float32, torch.bfloat16), dev)
    ht = final_state
    if ht is None and output_final_state:
        ht = torch.empty((N, H, SK, SV), dtype=torch.float32, device=dev)
    elif ht is not None:
        _need(ht, "final_state", (torch.float32,), dev)
    a = GdnStateArgs(dtype=int(dt), k=_ptr(k), v=_ptr(v), gate=int(_GATES[gate]),
                     gate_values=_ptr(gate_values) if gate is not None else None,
                     h0=_ptr(initial_state), ht=_ptr(ht), hs=_ptr(hs),
                     hs_dtype=int(DType.BF16 if hs is not None and hs.dtype == torch.bfloat16
                                  else DType.F32),
                     cu_seqlens=_ptr(cu_seqlens), B=B, T=T, H=H, K=K, V=V, N=N,
                     chunk_size=CHUNK, num_chunks=int(num_chunks or 0), split_size=split,
                     state_v_first=int(bool(state_v_first)))
    lib = _lib.load()
    _lib.check(lib.gdn_chunk_state_fwd(ctypes.byref(a), _stream(stream)), "gdn_chunk_state_fwd")
    return hs, ht


def gdn_chunk_state_bwd(q, do, gate=None, gate_values=None, dht=None, cu_seqlens=None,
                        scale=None, output_dh0=True, output_states=True,
                        states_dtype=torch.float32, out_states=None, dh0=None,
                        num_chunks=None, split_size=None, state_v_first=False, stream=None):
    """Backward state pass (dh recurrence).  Returns ``(dh, dh0)``.

    q [B,T,HQ,K], do [B,T,HQ,V] (float32 or bfloat16); gate and gate_values
    as :func:`gdn_chunk_state_fwd` with H gate heads (HQ % H == 0); dht
    [N,HQ,K,V] float32.  dh [C,HQ,K,V] is the gradient at the end of the
    first 64-token chunk of every split of ``split_size`` tokens (default 64:
    every chunk), sequence after sequence.  With ``state_v_first`` every
    state gradient (dht, dh, dh0) is [.., V, K].
    """
    split = _split_tokens(split_size)
    dev = q.device
    dt, dts = _io_dtype(q)
    _need(q, "q", dts, dev)
    _need(do, "do", dts, dev)
    if gate not in _GATES:
        raise ValueError(f"gate must be one of {list(_GATES)}")
    B, T, HQ, K = q.shape
    V = do.shape[3]
    if do.shape[:3] != (B, T, HQ):
        raise ValueError("q must be [B,T,HQ,K] and do [B,T,HQ,V]")
    H = HQ
    if gate is not None:
        _need(gate_values, "gate_values", (torch.float32,), dev)
        H = gate_values.shape[0] if gate == "g_gamma" else gate_values.shape[2]
    if cu_seqlens is not None:
        _need(cu_seqlens, "cu_seqlens", (torch.int32,), dev)
        N = cu_seqlens.numel() - 1
    else:
        N = B
    if num_chunks is None and (output_states or out_states is not None or cu_seqlens is None):
        num_chunks = _stored_states(B, T, cu_seqlens, split)
    SK, SV = (V, K) if state_v_first else (K, V)
    if dht is not None:
        _need(dht, "dht", (torch.float32,), dev)
        if tuple(dht.shape) != (N, HQ, SK, SV):
            raise ValueError(f"dht must be [{N},{HQ},{SK},{SV}]")
    dh = out_states
    if dh is None and output_states:
        dh = torch.empty((num_chunks, HQ, SK, SV), dtype=states_dtype, device=dev)
    if dh is not None:
        _need(dh, "out_states", (torch.float32, torch.bfloat16), dev)
    if dh0 is None and output_dh0:
        dh0 = torch.empty((N, HQ, SK, SV), dtype=torch.float32, device=dev)
    elif dh0 is not None:
        _need(dh0, "dh0", (torch.float32,), dev)
    a = GdnStateBwdArgs(dtype=int(dt), q=_ptr(q), do_=_ptr(do), gate=int(_GATES[gate]),
                        gate_values=_ptr(gate_values) if gate is not None else None,
                        dht=_ptr(dht), dh0=_ptr(dh0), dh=_ptr(dh),
                        dh_dtype=int(DType.BF16 if dh is not None and dh.dtype == torch.bfloat16
                                     else DType.F32),
                        cu_seqlens=_ptr(cu_seqlens), B=B, T=T, HQ=HQ, H=H, K=K, V=V, N=N,
                        chunk_size=CHUNK, num_chunks=int(num_chunks or 0),
                        scale=float(scale) if scale is not None else 0.0, split_size=split,
                        state_v_first=int(bool(state_v_first)))
    lib = _lib.load()
    _lib.check(lib.gdn_chunk_state_bwd(ctypes.byref(a), _stream(stream)), "gdn_chunk_state_bwd")
    return dh, dh0
