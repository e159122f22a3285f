"""Host-side checks of the C interface that need no GPU.

The library is loaded (built first if needed), every function the header
declares must be exported, the ctypes structures must match the C layout
(checked by compiling a probe against include/gdn.h with gcc), and argument
errors must come back as status codes before any CUDA call is made.
"""
import ctypes
import os
import re
import shutil
import subprocess
import tempfile

import pytest
import torch

from gated_delta_rule_kk_gb300 import _lib, build_lib
from gated_delta_rule_kk_gb300._lib import (GdnChunkArgs, GdnDecodeArgs, GdnStateArgs,
                                            GdnStateBwdArgs, KdaChunkArgs, Status)

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gdn.h")


@pytest.fixture(scope="module")
def lib():
    build_lib.build()
    return _lib.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+char\s*\*|gdn_status_t|size_t)\s*(\w+)\s*\(", text, re.M)))


def test_header_declares_expected_entry_points():
    names = declared_functions()
    for n in ("gdn_chunk_fwd", "kda_chunk_fwd", "gdn_decode", "gdn_check_device_error",
              "gdn_chunk_workspace_size", "kda_chunk_workspace_size", "gdn_status_string",
              "gdn_last_error_message"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert set(names) == set(_lib.SIGNATURES), "binding and header disagree"
    for n in names:
        assert hasattr(lib, n), f"{n} not exported"


def test_status_strings(lib):
    for s in Status:
        assert lib.gdn_status_string(int(s)).decode() == "GDN_" + ("OK" if s == 0 else "ERR_" + s.name)
    assert lib.gdn_status_string(99).decode() == "GDN_ERR_UNKNOWN"


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_ctypes_structs_match_c_layout():
    probe = r"""
#include <stdio.h>
#include <stddef.h>
#include "gdn.h"
#define F(S, f) printf(#S " " #f " %zu\n", offsetof(S, f));
int main(void) {
  printf("gdn_chunk_args size %zu\n", sizeof(gdn_chunk_args));
  printf("kda_chunk_args size %zu\n", sizeof(kda_chunk_args));
  printf("gdn_decode_args size %zu\n", sizeof(gdn_decode_args));
  printf("gdn_state_args size %zu\n", sizeof(gdn_state_args));
  printf("gdn_state_bwd_args size %zu\n", sizeof(gdn_state_bwd_args));
  %FIELDS%
  return 0;
}
"""
    lines = []
    for cname, cls in (("gdn_chunk_args", GdnChunkArgs), ("kda_chunk_args", KdaChunkArgs),
                       ("gdn_decode_args", GdnDecodeArgs), ("gdn_state_args", GdnStateArgs),
                       ("gdn_state_bwd_args", GdnStateBwdArgs)):
        for fname, _ in cls._fields_:
            lines.append(f"F({cname}, {fname})")
    src = probe.replace("%FIELDS%", "\n  ".join(lines))
    with tempfile.TemporaryDirectory() as d:
        c = os.path.join(d, "probe.c")
        exe = os.path.join(d, "probe")
        open(c, "w").write(src)
        subprocess.check_call(["gcc", "-std=c99", "-I", os.path.join(ROOT, "include"), c, "-o", exe])
        out = subprocess.check_output([exe], text=True).split("\n")
    got = {}
    for ln in out:
        if ln.strip():
            s, f, v = ln.split()
            got[(s, f)] = int(v)
    for cname, cls in (("gdn_chunk_args", GdnChunkArgs), ("kda_chunk_args", KdaChunkArgs),
                       ("gdn_decode_args", GdnDecodeArgs), ("gdn_state_args", GdnStateArgs),
                       ("gdn_state_bwd_args", GdnStateBwdArgs)):
        assert got[(cname, "size")] == ctypes.sizeof(cls), cname
        for fname, _ in cls._fields_:
            assert got[(cname, fname)] == getattr(cls, fname).offset, (cname, fname)


# ---- argument checks: all of these return before any CUDA call -------------

FAKE = 0x10000  # 16-byte aligned, never dereferenced: validation fails first


def good_chunk(**kw):
    a = dict(dtype=1, q=FAKE, k=FAKE, v=FAKE, g=FAKE, beta=FAKE, h0=None, ht=None, o=FAKE,
             cu_seqlens=None, B=2, T=128, H=4, Hg=2, K=128, V=128, N=2, chunk_size=64,
             g_is_cumsum=0, scale=0.0, workspace=None, workspace_bytes=0)
    a.update(kw)
    return GdnChunkArgs(**a)


@pytest.mark.parametrize("change,expect", [
    (dict(q=None), Status.INVALID_ARG),
    (dict(o=None), Status.INVALID_ARG),
    (dict(beta=None), Status.INVALID_ARG),
    (dict(k=FAKE + 2), Status.MISALIGNED),
    (dict(h0=FAKE + 8), Status.MISALIGNED),
    (dict(dtype=7), Status.INVALID_ARG),
    (dict(chunk_size=32), Status.UNSUPPORTED),
    (dict(K=256), Status.UNSUPPORTED),
    (dict(H=5), Status.UNSUPPORTED),
    (dict(B=0), Status.INVALID_ARG),
    (dict(N=3), Status.INVALID_ARG),
    (dict(cu_seqlens=FAKE), Status.INVALID_ARG),  # B=2 with cu_seqlens
    (dict(g_is_cumsum=2), Status.INVALID_ARG),
    (dict(scale=float("nan")), Status.INVALID_ARG),
])
def test_gdn_chunk_argument_errors(lib, change, expect):
    a = good_chunk(**change)
    st = lib.gdn_chunk_fwd(ctypes.byref(a), None)
    assert st == expect, (change, Status(st), lib.gdn_last_error_message())
    assert lib.gdn_last_error_message().decode() != ""


def test_null_args_pointer(lib):
    assert lib.gdn_chunk_fwd(None, None) == Status.INVALID_ARG
    assert lib.kda_chunk_fwd(None, None) == Status.INVALID_ARG
    assert lib.gdn_decode(None, None) == Status.INVALID_ARG
    assert lib.gdn_check_device_error(None, None) == Status.INVALID_ARG


def test_kda_head_grouping_error(lib):
    a = KdaChunkArgs(dtype=1, q=FAKE, k=FAKE, v=FAKE, g=FAKE, beta=FAKE, o=FAKE, B=1, T=64,
                     H=3, HV=4, K=128, V=128, N=1, chunk_size=64, g_is_cumsum=1)
    assert lib.kda_chunk_fwd(ctypes.byref(a), None) == Status.UNSUPPORTED


def good_decode(**kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, a=FAKE, b=FAKE, A_log=FAKE, dt_bias=FAKE, state=FAKE,
             slot_indices=None, o=FAKE, B=4, T=1, H=2, HV=4, K=128, V=128, pool=4,
             use_qk_l2norm=1, scale=0.0, softplus_beta=1.0, softplus_threshold=20.0, eps=1e-6)
    a.update(kw)
    return GdnDecodeArgs(**a)


@pytest.mark.parametrize("change,expect", [
    (dict(T=0), Status.UNSUPPORTED),
    (dict(T=5), Status.UNSUPPORTED),
    (dict(K=64), Status.UNSUPPORTED),
    (dict(V=96), Status.UNSUPPORTED),
    (dict(HV=3), Status.UNSUPPORTED),
    (dict(pool=2), Status.INVALID_ARG),   # identity slots need pool >= B
    (dict(state=None), Status.INVALID_ARG),
    (dict(A_log=FAKE + 4), Status.MISALIGNED),
    (dict(slot_indices=FAKE + 4), Status.MISALIGNED),
    (dict(use_qk_l2norm=3), Status.INVALID_ARG),
    (dict(eps=float("inf")), Status.INVALID_ARG),
])
def test_decode_argument_errors(lib, change, expect):
    a = good_decode(**change)
    assert lib.gdn_decode(ctypes.byref(a), None) == expect


def test_workspace_size(lib):
    # the tensor-core path (bf16, K = 128, V % 32 == 0, V <= 128) needs per
    # (chunk, head) operand blocks of 82944 + 256 V bytes plus the chunk table
    # (N + 1 offsets and N sequence indices, int32, rounded up to 256 bytes)
    blk = 82944 + 256 * 128
    a = good_chunk()
    n = ctypes.c_size_t(123)
    assert lib.gdn_chunk_workspace_size(ctypes.byref(a), ctypes.byref(n)) == Status.OK
    assert n.value == 256 + 2 * 2 * 4 * blk
    # packed sequences: at most ceil(T/64) + N chunks
    a = good_chunk(B=1, N=3, cu_seqlens=FAKE, T=200)
    assert lib.gdn_chunk_workspace_size(ctypes.byref(a), ctypes.byref(n)) == Status.OK
    assert n.value == 256 + (4 + 3) * 4 * blk
    a = good_chunk(B=1, N=100, cu_seqlens=FAKE, T=6400)
    assert lib.gdn_chunk_workspace_size(ctypes.byref(a), ctypes.byref(n)) == Status.OK
    assert n.value == 1024 + (100 + 100) * 4 * blk
    # V beyond 128 takes the CUDA-core path
    a = good_chunk(V=160)
    assert lib.gdn_chunk_workspace_size(ctypes.byref(a), ctypes.byref(n)) == Status.OK
    assert n.value == 0
    # the exact fp32 path needs none
    a = good_chunk(dtype=0)
    assert lib.gdn_chunk_workspace_size(ctypes.byref(a), ctypes.byref(n)) == Status.OK
    assert n.value == 0
    k = KdaChunkArgs(dtype=1, B=1, T=64, H=2, HV=2, K=128, V=64, N=1, chunk_size=64)
    assert lib.kda_chunk_workspace_size(ctypes.byref(k), ctypes.byref(n)) == Status.OK
    assert n.value == 256 + 1 * 2 * (82944 + 256 * 64)


def test_workspace_errors_found_on_host(lib):
    a = good_chunk(workspace=None, workspace_bytes=0)
    assert lib.gdn_chunk_fwd(ctypes.byref(a), None) == Status.WORKSPACE
    a = good_chunk(workspace=FAKE, workspace_bytes=100)
    assert lib.gdn_chunk_fwd(ctypes.byref(a), None) == Status.WORKSPACE
    a = good_chunk(workspace=FAKE + 16, workspace_bytes=1 << 30)
    assert lib.gdn_chunk_fwd(ctypes.byref(a), None) == Status.MISALIGNED


def good_state(**kw):
    a = dict(dtype=1, k=FAKE, v=FAKE, gate=1, gate_values=FAKE, h0=None, ht=None, hs=FAKE,
             hs_dtype=0, cu_seqlens=None, B=2, T=130, H=4, K=128, V=64, N=2, chunk_size=64,
             num_chunks=6)
    a.update(kw)
    return GdnStateArgs(**a)


@pytest.mark.parametrize("change,expect", [
    (dict(dtype=5), Status.INVALID_ARG),
    (dict(gate=7), Status.INVALID_ARG),
    (dict(gate=0), Status.INVALID_ARG),            # gate values without a gate
    (dict(gate_values=None), Status.INVALID_ARG),   # a gate without values
    (dict(k=None), Status.INVALID_ARG),
    (dict(v=FAKE + 4), Status.MISALIGNED),
    (dict(K=256), Status.UNSUPPORTED),
    (dict(V=60), Status.UNSUPPORTED),
    (dict(K=36), Status.UNSUPPORTED),
    (dict(chunk_size=32), Status.UNSUPPORTED),
    (dict(N=3), Status.INVALID_ARG),
    (dict(cu_seqlens=FAKE), Status.INVALID_ARG),    # B=2 with cu_seqlens
    (dict(num_chunks=5), Status.INVALID_ARG),       # 2 sequences x 3 chunks do not fit
    (dict(hs_dtype=3), Status.INVALID_ARG),
    (dict(h0=FAKE + 8), Status.MISALIGNED),
])
def test_state_pass_argument_errors(lib, change, expect):
    a = good_state(**change)
    assert lib.gdn_chunk_state_fwd(ctypes.byref(a), None) == expect
    assert lib.gdn_last_error_message().decode() != ""


@pytest.mark.parametrize("change,expect", [
    (dict(H=3), Status.UNSUPPORTED),               # HQ = 4 not a multiple
    (dict(do_=None), Status.INVALID_ARG),
    (dict(scale=float("inf")), Status.INVALID_ARG),
    (dict(K=20), Status.UNSUPPORTED),
    (dict(num_chunks=1), Status.INVALID_ARG),
    (dict(gate=1, gate_values=None), Status.INVALID_ARG),
])
def test_state_bwd_argument_errors(lib, change, expect):
    a = dict(dtype=1, q=FAKE, do_=FAKE, gate=0, gate_values=None, dht=None, dh0=None, dh=FAKE,
             dh_dtype=0, cu_seqlens=None, B=1, T=100, HQ=4, H=2, K=64, V=64, N=1, chunk_size=64,
             num_chunks=2, scale=0.0)
    a.update(change)
    st = lib.gdn_chunk_state_bwd(ctypes.byref(GdnStateBwdArgs(**a)), None)
    assert st == expect, (change, Status(st))


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_plain_c_caller_compiles(tmp_path):
    # tests/c_abi_program.c, the plain C caller the GPU tests run, builds
    # against include/gdn.h with -Wall -Werror
    from c_program import compile_program
    try:
        compile_program(str(tmp_path), link=False)
    except subprocess.CalledProcessError as e:
        raise AssertionError(e.stderr)


def test_grid_limits_are_rejected_up_front(lib):
    # sequences and heads index grid dimensions y and z (at most 65535)
    a = good_chunk(B=1, N=70000, cu_seqlens=FAKE, T=70000)
    assert lib.gdn_chunk_fwd(ctypes.byref(a), None) == Status.UNSUPPORTED
    assert "65535" in lib.gdn_last_error_message().decode()
    st = GdnStateArgs(dtype=1, k=FAKE, v=FAKE, gate=0, B=1, T=70000, H=2, K=64, V=64, N=70000,
                      chunk_size=64, cu_seqlens=FAKE)
    assert lib.gdn_chunk_state_fwd(ctypes.byref(st), None) == Status.UNSUPPORTED
    bw = GdnStateBwdArgs(dtype=1, q=FAKE, do_=FAKE, gate=0, B=1, T=100, HQ=70000, H=70000, K=64,
                         V=64, N=1, chunk_size=64)
    assert lib.gdn_chunk_state_bwd(ctypes.byref(bw), None) == Status.UNSUPPORTED


@pytest.mark.parametrize("split,expect", [(100, Status.INVALID_ARG), (-64, Status.INVALID_ARG),
                                          (128, Status.OK)])
def test_state_split_size(lib, split, expect):
    # split_size: 0 or a positive multiple of 64; the stored states then number
    # ceil(T / split_size) per sequence (T = 300, split 128: 3 per sequence)
    a = GdnStateArgs(dtype=1, k=FAKE, v=FAKE, gate=0, hs=FAKE, hs_dtype=0, B=2, T=300, H=2,
                     K=64, V=64, N=2, chunk_size=64, num_chunks=6, split_size=split)
    st = lib.gdn_chunk_state_fwd(ctypes.byref(a), None)
    if expect == Status.OK:
        # the sizes pass; the first CUDA call then fails without a GPU
        assert st != Status.INVALID_ARG, lib.gdn_last_error_message()
        a.num_chunks = 5
        assert lib.gdn_chunk_state_fwd(ctypes.byref(a), None) == Status.INVALID_ARG
        assert "needed" in lib.gdn_last_error_message().decode()
    else:
        assert st == expect


def test_state_pass_binding_rejects_bad_split_before_any_call():
    # the binding checks split_size first, so no library call (or GPU) is
    # needed to see the error
    import torch
    import gated_delta_rule_kk_gb300 as gdn
    k = torch.zeros(1, 64, 2, 64)
    v = torch.zeros(1, 64, 2, 64)
    for bad in (100, -64, 32):
        with pytest.raises(ValueError, match="multiple of 64"):
            gdn.gdn_chunk_state_fwd(k, v, split_size=bad)
        with pytest.raises(ValueError, match="multiple of 64"):
            gdn.gdn_chunk_state_bwd(k, v, split_size=bad)


def test_self_test_wait_rejects_bad_arguments(lib):
    for arrive, polls in ((2, 1), (0, 0), (0, -5), (1, (1 << 22) + 1)):
        assert lib.gdn_self_test_wait(arrive, polls, None) == Status.INVALID_ARG


def test_chunk_state_v_first_flag_is_checked(lib):
    for cls, fn in ((GdnChunkArgs, "gdn_chunk_fwd"), (KdaChunkArgs, "kda_chunk_fwd")):
        a = cls(dtype=1, q=0x10000, k=0x10000, v=0x10000, g=0x10000, beta=0x10000, o=0x10000,
                B=1, T=64, K=128, V=128, N=1, chunk_size=64, state_v_first=2)
        if cls is GdnChunkArgs:
            a.H, a.Hg = 1, 1
        else:
            a.H, a.HV = 1, 1
        assert getattr(lib, fn)(ctypes.byref(a), None) == Status.INVALID_ARG
        assert b"state_v_first" in lib.gdn_last_error_message()


def test_segments_range_is_checked(lib):
    base = dict(dtype=1, q=0x10000, k=0x10000, v=0x10000, g=0x10000, beta=0x10000, o=0x10000,
                B=1, T=64, H=1, Hg=1, K=128, V=128, N=1, chunk_size=64)
    a = GdnChunkArgs(segments=-1, **base)
    assert lib.gdn_chunk_fwd(ctypes.byref(a), None) == Status.INVALID_ARG
    a = GdnChunkArgs(segments=65, **base)
    assert lib.gdn_chunk_fwd(ctypes.byref(a), None) == Status.UNSUPPORTED
    a = GdnChunkArgs(segments=4, **base)
    n4, n1 = ctypes.c_size_t(0), ctypes.c_size_t(0)
    assert lib.gdn_chunk_workspace_size(ctypes.byref(a), ctypes.byref(n4)) == Status.OK
    a.segments = 1
    assert lib.gdn_chunk_workspace_size(ctypes.byref(a), ctypes.byref(n1)) == Status.OK
    # the segment scratch: per (sequence, segment, head) a [K, K + V] and a [K, V] fp32 state
    assert n4.value - n1.value == 4 * 128 * (256 + 128) * 4


def test_segment_count_choice(lib):
    """The library's own choice: none for the benchmarked shapes (their chains
    already fill the SMs), the segment-parallel pass for one long sequence
    with few heads; an explicit count is returned as given."""
    import gated_delta_rule_kk_gb300 as gdn
    assert gdn.gdn_chunk_segment_count(2, 4096, 16, 16, 128, 128) == 1
    assert gdn.gdn_chunk_segment_count(1, 8192, 32, 32, 128, 128) == 1
    assert gdn.gdn_chunk_segment_count(1, 8192, 1, 1, 128, 128) > 1
    assert gdn.gdn_chunk_segment_count(1, 8192, 2, 2, 128, 128, segments=3) == 3
    assert gdn.gdn_chunk_segment_count(1, 8192, 1, 1, 64, 64, dtype=torch.float32) == 1
    assert gdn.gdn_chunk_segment_count(1, 300, 1, 1, 128, 128) == 1  # too few chunks
