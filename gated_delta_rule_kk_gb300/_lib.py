"""ctypes binding of ``include/gdn.h``: argument marshalling only.

Every computation runs in the CUDA library ``lib/libgdn_gb300.so``; there is
no CPU or PyTorch fallback.  If the library is missing, every entry point
raises ``RuntimeError``.
"""
from __future__ import annotations

import ctypes
import enum
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
# GDN_CHECKED=1 selects the checked build (bounds checks in every kernel; see
# build_lib), which must have been built first.
CHECKED = os.environ.get("GDN_CHECKED", "0") == "1"
LIB_PATH = os.path.join(HERE, "lib", "libgdn_gb300_checked.so" if CHECKED else "libgdn_gb300.so")

c_int32, c_float, c_void_p, c_size_t = ctypes.c_int32, ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t


class Status(enum.IntEnum):
    OK = 0
    INVALID_ARG = 1
    UNSUPPORTED = 2
    MISALIGNED = 3
    WORKSPACE = 4
    CUDA = 5
    TIMEOUT = 6
    BAD_SEQLENS = 7
    BAD_SLOT = 8
    BOUNDS = 9


class DType(enum.IntEnum):
    F32 = 0
    BF16 = 1


class GdnChunkArgs(ctypes.Structure):
    _fields_ = [
        ("dtype", c_int32),
        ("q", c_void_p), ("k", c_void_p), ("v", c_void_p),
        ("g", c_void_p), ("beta", c_void_p), ("h0", c_void_p), ("ht", c_void_p),
        ("o", c_void_p), ("cu_seqlens", c_void_p),
        ("B", c_int32), ("T", c_int32), ("H", c_int32), ("Hg", c_int32),
        ("K", c_int32), ("V", c_int32), ("N", c_int32),
        ("chunk_size", c_int32), ("g_is_cumsum", c_int32), ("state_v_first", c_int32),
        ("o_fp32", c_int32), ("segments", c_int32), ("scale", c_float),
        ("workspace", c_void_p), ("workspace_bytes", c_size_t),
    ]


class KdaChunkArgs(ctypes.Structure):
    _fields_ = [
        ("dtype", c_int32),
        ("q", c_void_p), ("k", c_void_p), ("v", c_void_p),
        ("g", c_void_p), ("beta", c_void_p), ("h0", c_void_p), ("ht", c_void_p),
        ("o", c_void_p), ("cu_seqlens", c_void_p),
        ("B", c_int32), ("T", c_int32), ("H", c_int32), ("HV", c_int32),
        ("K", c_int32), ("V", c_int32), ("N", c_int32),
        ("chunk_size", c_int32), ("g_is_cumsum", c_int32), ("state_v_first", c_int32),
        ("o_fp32", c_int32), ("segments", c_int32), ("scale", c_float),
        ("workspace", c_void_p), ("workspace_bytes", c_size_t),
    ]


class GdnDecodeArgs(ctypes.Structure):
    _fields_ = [
        ("q", c_void_p), ("k", c_void_p), ("v", c_void_p),
        ("a", c_void_p), ("b", c_void_p),
        ("A_log", c_void_p), ("dt_bias", c_void_p),
        ("state", c_void_p), ("slot_indices", c_void_p), ("o", c_void_p),
        ("new_state_f32", c_void_p),
        ("B", c_int32), ("T", c_int32), ("H", c_int32), ("HV", c_int32),
        ("K", c_int32), ("V", c_int32), ("pool", c_int32),
        ("use_qk_l2norm", c_int32), ("o_fp32", c_int32),
        ("scale", c_float), ("softplus_beta", c_float), ("softplus_threshold", c_float),
        ("eps", c_float),
    ]


class GateKind(enum.IntEnum):
    NONE = 0
    G = 1
    G_GAMMA = 2
    GK = 3
    GV = 4


class GdnStateArgs(ctypes.Structure):
    _fields_ = [
        ("dtype", c_int32),
        ("k", c_void_p), ("v", c_void_p),
        ("gate", c_int32), ("gate_values", c_void_p),
        ("h0", c_void_p), ("ht", c_void_p),
        ("hs", c_void_p), ("hs_dtype", c_int32),
        ("cu_seqlens", c_void_p),
        ("B", c_int32), ("T", c_int32), ("H", c_int32), ("K", c_int32), ("V", c_int32),
        ("N", c_int32), ("chunk_size", c_int32),
        ("num_chunks", ctypes.c_int64),
        ("split_size", c_int32),
        ("state_v_first", c_int32),
    ]


class GdnStateBwdArgs(ctypes.Structure):
    _fields_ = [
        ("dtype", c_int32),
        ("q", c_void_p), ("do_", c_void_p),
        ("gate", c_int32), ("gate_values", c_void_p),
        ("dht", c_void_p), ("dh0", c_void_p),
        ("dh", c_void_p), ("dh_dtype", c_int32),
        ("cu_seqlens", c_void_p),
        ("B", c_int32), ("T", c_int32), ("HQ", c_int32), ("H", c_int32), ("K", c_int32),
        ("V", c_int32), ("N", c_int32), ("chunk_size", c_int32),
        ("num_chunks", ctypes.c_int64),
        ("scale", c_float),
        ("split_size", c_int32),
        ("state_v_first", c_int32),
    ]


# name -> (argtypes, restype); exactly the functions include/gdn.h declares
SIGNATURES = {
    "gdn_chunk_workspace_size": ([ctypes.POINTER(GdnChunkArgs), ctypes.POINTER(c_size_t)], c_int32),
    "gdn_chunk_fwd": ([ctypes.POINTER(GdnChunkArgs), c_void_p], c_int32),
    "gdn_chunk_segment_count": ([ctypes.POINTER(GdnChunkArgs), ctypes.POINTER(c_int32)], c_int32),
    "gdn_chunk_fwd_host": ([ctypes.POINTER(GdnChunkArgs), c_void_p], c_int32),
    "gdn_chunk_host_workspace_size": ([ctypes.POINTER(GdnChunkArgs), ctypes.POINTER(c_size_t)],
                                      c_int32),
    "kda_chunk_workspace_size": ([ctypes.POINTER(KdaChunkArgs), ctypes.POINTER(c_size_t)], c_int32),
    "kda_chunk_fwd": ([ctypes.POINTER(KdaChunkArgs), c_void_p], c_int32),
    "gdn_decode": ([ctypes.POINTER(GdnDecodeArgs), c_void_p], c_int32),
    "gdn_chunk_state_fwd": ([ctypes.POINTER(GdnStateArgs), c_void_p], c_int32),
    "gdn_chunk_state_bwd": ([ctypes.POINTER(GdnStateBwdArgs), c_void_p], c_int32),
    "gdn_chunk_fwd_noalloc": ([ctypes.POINTER(GdnChunkArgs), c_void_p], c_int32),
    "gdn_noalloc_scratch_bytes": ([], c_size_t),
    "gdn_self_test_wait": ([c_int32, c_int32, c_void_p], c_int32),
    "gdn_self_test_bounds": ([c_int32, c_int32, ctypes.POINTER(c_int32), c_void_p], c_int32),
    "gdn_check_device_error": ([c_void_p, ctypes.POINTER(c_int32)], c_int32),
    "gdn_status_string": ([c_int32], ctypes.c_char_p),
    "gdn_last_error_message": ([], ctypes.c_char_p),
}

_lock = threading.Lock()
_lib = None


class GdnError(RuntimeError):
    """A library call returned a status other than GDN_OK."""

    def __init__(self, status, func, message=""):
        self.status = Status(status) if status in Status._value2member_map_ else status
        super().__init__(f"{func}: {self.status!r} {message}".strip())


def load(path: str | None = None):
    """Load the shared library once and declare its signatures."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            how = ("`python -m gated_delta_rule_kk_gb300.build_lib --checked`" if p.endswith("_checked.so")
                   else "`python -c 'import __graft_entry__ as g; g.build()'`")
            raise RuntimeError(f"CUDA library {p} is missing: build it with {how}")
        lib = ctypes.CDLL(p)
        for name, (argtypes, restype) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.argtypes = argtypes
            fn.restype = restype
        if path is None:
            _lib = lib
        return lib


def check(status: int, func: str):
    if status != Status.OK:
        msg = load().gdn_last_error_message()
        raise GdnError(status, func, msg.decode() if msg else "")
