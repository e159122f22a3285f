"""Host-side checks of gdn_chunk_fwd_host / gdn_chunk_host_workspace_size.

The workspace layout and the argument errors are decided on the host before
any CUDA call, so they are checked here without a GPU.  The copies and the
pipelined forward are checked on the GPU in test_host_io_gpu.py.
"""
import ctypes

import pytest

from gated_delta_rule_kk_gb300 import _lib, build_lib
from gated_delta_rule_kk_gb300._lib import GdnChunkArgs, Status

BLK128 = 82944 + 256 * 128  # tensor-core operand block per (chunk, head), V = 128


def a256(x):
    return (x + 255) // 256 * 256


@pytest.fixture(scope="module")
def lib():
    build_lib.build()
    return _lib.load()


def args(**kw):
    a = dict(dtype=1, q=None, k=None, v=None, g=None, beta=None, h0=None, ht=None, o=None,
             cu_seqlens=None, B=2, T=4096, H=16, Hg=16, K=128, V=128, N=2, chunk_size=64,
             g_is_cumsum=0, scale=0.0, workspace=None, workspace_bytes=0)
    a.update(kw)
    return GdnChunkArgs(**a)


def ws_size(lib, a):
    n = ctypes.c_size_t(7)
    st = lib.gdn_chunk_host_workspace_size(ctypes.byref(a), ctypes.byref(n))
    return st, n.value


def test_time_cut_layout(lib):
    # B=2, T=4096 (64 chunks): four time pieces halving towards a last piece
    # of 4 chunks -> 34, 17, 9, 4 chunks.  Each piece has its own q, k, v, o,
    # g, beta slices; two whole fp32 states; and the tensor-core scratch of the
    # largest piece (B=2, 34 chunks x 16 heads).
    st, n = ws_size(lib, args())
    assert st == Status.OK
    chunks = (34, 17, 9, 4)
    rows = [2 * 64 * c for c in chunks]
    qk = sum(a256(r * 16 * 128 * 2) for r in rows)
    vo = sum(a256(r * 16 * 128 * 2) for r in rows)
    gb = sum(a256(r * 16 * 4) for r in rows)
    state = a256(2 * 16 * 128 * 128 * 4)
    scratch = 256 + 2 * 34 * 16 * BLK128
    assert n == 2 * qk + 2 * vo + 2 * gb + 2 * state + scratch


@pytest.mark.parametrize("T,chunks", [
    (705, (8, 4)),             # 12 chunks: the shortest sequence that is cut in time
    (2100, (19, 9, 5)),        # ragged tail inside the last piece
    (64 * 1000, None),         # at most 8 pieces
])
def test_time_cut_piece_counts(lib, T, chunks):
    st, n = ws_size(lib, args(B=1, N=1, T=T, dtype=0, H=1, Hg=1, K=16, V=16))
    assert st == Status.OK
    if chunks is not None:
        tok = [64 * c for c in chunks]
        tok[-1] -= 64 * sum(chunks) - T
        per = sum(2 * a256(t * 16 * 4) * 2 + 2 * a256(t * 4) for t in tok)
        assert n == per + 2 * a256(16 * 16 * 4)
    else:
        # eight pieces: 8 slices of each of the six per-row regions, each
        # padded to 256 bytes, so the total sits within 6*8*256 of the tight sum
        tight = 2 * (T * 64) * 2 + 2 * T * 4 + 2 * a256(16 * 16 * 4)
        assert tight <= n <= tight + 6 * 8 * 256


def test_704_tokens_are_cut_by_sequence(lib):
    st, n = ws_size(lib, args(B=1, N=1, T=704, dtype=0, H=1, Hg=1, K=16, V=16))
    assert st == Status.OK
    assert n == 2 * a256(704 * 64) * 2 + 2 * a256(704 * 4) + 2 * a256(16 * 16 * 4)


def test_short_sequences_cut_by_batch(lib):
    # T=512 (8 chunks) is too short to cut in time: cut the 16 sequences into
    # 16*512/2048 = 4 pieces of 4 whole sequences.
    st, n = ws_size(lib, args(B=16, N=16, T=512))
    assert st == Status.OK
    rows = 4 * 512
    slices = 4 * (2 * a256(rows * 4096) + 2 * a256(rows * 4096) + 2 * a256(rows * 64)
                  + 2 * a256(4 * 16 * 128 * 128 * 4))
    assert n == slices + 256 + 4 * 8 * 16 * BLK128


def test_fp32_needs_no_scratch(lib):
    st, n = ws_size(lib, args(dtype=0, B=1, N=1, T=100, H=2, Hg=1, K=64, V=48))
    assert st == Status.OK
    elt = 4
    assert n == (2 * a256(100 * 64 * elt) + 2 * a256(100 * 2 * 48 * elt) + 2 * a256(100 * 2 * 4)
                 + 2 * a256(2 * 64 * 48 * 4))


def test_varlen_pieces_follow_sequence_ends(lib):
    cu = (ctypes.c_int32 * 5)(0, 3000, 3000, 7000, 8192)
    st, n = ws_size(lib, args(B=1, N=4, T=8192, cu_seqlens=ctypes.cast(cu, ctypes.c_void_p)))
    assert st == Status.OK
    # pieces: sequences {0} (3000 rows), {1, 2} (4000 rows), {3} (1192 rows)
    rows = (3000, 4000, 1192)
    nseq = (1, 2, 1)
    per = sum(2 * a256(r * 4096) * 2 + 2 * a256(r * 64) for r in rows)
    states = 2 * sum(a256(s * 16 * 128 * 128 * 4) for s in nseq)
    offsets = a256((4 + 4 + 4) * 4)  # 2, 3, 2 offsets, each padded to 4 ints
    # scratch of the largest piece: ceil(4000/64) + 2 chunks per head
    scratch = 256 + (63 + 2) * 16 * BLK128
    assert n == per + states + offsets + scratch


@pytest.mark.parametrize("cu", [(1, 10, 20), (0, 10, 19), (0, 12, 10), (0, 25, 20)])
def test_bad_seqlens_found_on_host(lib, cu):
    arr = (ctypes.c_int32 * 3)(*cu)
    a = args(B=1, N=2, T=20, cu_seqlens=ctypes.cast(arr, ctypes.c_void_p))
    st, _ = ws_size(lib, a)
    assert st == Status.BAD_SEQLENS, lib.gdn_last_error_message()


@pytest.mark.parametrize("change,expect", [
    (dict(K=256), Status.UNSUPPORTED),
    (dict(H=5), Status.UNSUPPORTED),
    (dict(N=3), Status.INVALID_ARG),
    (dict(chunk_size=32), Status.UNSUPPORTED),
    (dict(dtype=9), Status.INVALID_ARG),
])
def test_size_errors(lib, change, expect):
    st, _ = ws_size(lib, args(**change))
    assert st == expect


def test_call_errors_before_any_cuda_call(lib):
    buf = ctypes.create_string_buffer(64)
    p = ctypes.cast(buf, ctypes.c_void_p)
    assert lib.gdn_chunk_fwd_host(None, None) == Status.INVALID_ARG
    full = dict(q=p, k=p, v=p, g=p, beta=p, o=p)
    for missing in ("q", "v", "beta", "o"):
        a = args(**{**full, missing: None})
        assert lib.gdn_chunk_fwd_host(ctypes.byref(a), None) == Status.INVALID_ARG
        assert missing in lib.gdn_last_error_message().decode()
    a = args(**full, K=256)
    assert lib.gdn_chunk_fwd_host(ctypes.byref(a), None) == Status.UNSUPPORTED
    a = args(**full)
    assert lib.gdn_chunk_fwd_host(ctypes.byref(a), None) == Status.WORKSPACE
    a = args(**full, workspace=0x10010, workspace_bytes=1 << 40)
    assert lib.gdn_chunk_fwd_host(ctypes.byref(a), None) == Status.MISALIGNED
    a = args(**full, workspace=0x10000, workspace_bytes=1000)
    assert lib.gdn_chunk_fwd_host(ctypes.byref(a), None) == Status.WORKSPACE
    assert "needed" in lib.gdn_last_error_message().decode()
