"""The checked build (``-DGDN_CHECKED``) on the GPU.

Every kernel of a checked build compares the index ranges a CTA derives with
the extents of the tensors they index before it touches memory, and records
GDN_ERR_BOUNDS instead when one falls outside.  These tests build that library,
show that the check fires on an out-of-range index (gdn_self_test_bounds) and
never on valid work, and that the checked build computes exactly what the
release build does: the same tiny and ragged problems through both libraries,
results compared bit for bit.  They run in a child process with
GDN_CHECKED=1, which makes the package load the checked library.
"""
import json
import os
import subprocess
import sys

import pytest

from gated_delta_rule_kk_gb300 import build_lib

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import ctypes, json, sys
sys.path.insert(0, sys.argv[1])
import torch
from gated_delta_rule_kk_gb300 import _lib, synth
import gated_delta_rule_kk_gb300 as gdn

checked = _lib.load()                       # GDN_CHECKED=1: the checked library
release = _lib.load(sys.argv[2])           # the release library, loaded beside it
out = {"checked_flag": None, "self_test": {}, "cases": {}}

flag = ctypes.c_int32(-1)
for idx, ext in ((1, 3), (3, 3), (-1, 3)):
    assert checked.gdn_self_test_bounds(idx, ext, ctypes.byref(flag), None) == 0
    out["self_test"][f"{idx}/{ext}"] = int(gdn.gdn_check_device_error())
out["checked_flag"] = flag.value
rel = ctypes.c_int32(-1)
_lib._lib = release                        # each library has its own error word
assert release.gdn_self_test_bounds(3, 3, ctypes.byref(rel), None) == 0
out["release_flag"] = rel.value
out["release_self_test"] = int(gdn.gdn_check_device_error())

def dev(inp):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}

def prefill(inp, kda=False, segments=0):
    d = dev(inp)
    fn = gdn.kda_chunk_fwd if kda else gdn.gdn_chunk_fwd
    kw = dict(scale=d["scale"], initial_state=d["h0"], cu_seqlens=d["cu_seqlens"],
              g_is_cumsum=d["g_is_cumsum"], segments=segments)
    return fn(d["q"], d["k"], d["v"], d["g"], d["beta"], **kw)

def decode(T):
    d = dev(synth.decode_inputs(50 + T, 5, T, 2, 4, 128, 128))
    state = d["state"].clone()
    o = gdn.gdn_decode(d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"], d["dt_bias"], state,
                       slot_indices=d["slot_indices"], scale=d["scale"])
    return o, state

def state_pass():
    d = dev(synth.state_pass_inputs(9, 1, 150, 2, 128, 128, "g", h0_std=0.1))
    return gdn.gdn_chunk_state_fwd(d["k"], d["v"], gate="g", gate_values=d["gate_values"],
                                   initial_state=d["h0"])

cases = {}
for T in (1, 15, 16, 17, 63, 64, 65, 200):
    cases[f"gdn_tc_T{T}"] = lambda T=T: prefill(synth.prefill_inputs(T, 1, T, 2, 2, 128, 128,
                                                                     h0_std=0.1))
lens = [1, 15, 16, 17, 63, 64, 65]
cases["gdn_tc_packed_grouped"] = lambda: prefill(synth.prefill_inputs(
    7, 1, sum(lens), 4, 2, 128, 128, lengths=lens))
cases["gdn_fp32_T65"] = lambda: prefill(synth.prefill_inputs(8, 2, 65, 2, 1, 32, 32,
                                                             dtype=torch.float32, h0_std=0.1))
cases["kda_tc_T65"] = lambda: prefill(synth.prefill_inputs(9, 1, 65, 2, 2, 128, 128,
                                                           per_channel=True, h0_std=0.1), kda=True)
cases["gdn_tc_segments"] = lambda: prefill(synth.prefill_inputs(10, 1, 700, 1, 1, 128, 128,
                                                                h0_std=0.1), segments=3)
for T in (1, 2, 3, 4):
    cases[f"decode_T{T}"] = lambda T=T: decode(T)
cases["state_pass_g"] = state_pass

for name, fn in cases.items():
    _lib._lib = checked
    a = fn()
    err = int(gdn.gdn_check_device_error())
    _lib._lib = release
    b = fn()
    assert int(gdn.gdn_check_device_error()) == 0
    same = all(torch.equal(x, y) for x, y in zip(a, b))
    out["cases"][name] = {"device_error": err, "bit_identical": bool(same)}
print(json.dumps(out))
"""


@pytest.fixture(scope="module")
def child_result():
    checked_lib = build_lib.build(checked=True)
    release_lib = build_lib.build()
    env = dict(os.environ, GDN_CHECKED="1")
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT, release_lib], env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout + r.stderr
    assert checked_lib.endswith("_checked.so")
    return json.loads(r.stdout.strip().splitlines()[-1])


def test_bounds_check_fires_only_in_the_checked_build(child_result):
    res = child_result
    assert res["checked_flag"] == 1 and res["release_flag"] == 0
    bounds = 9  # GDN_ERR_BOUNDS
    assert res["self_test"] == {"1/3": 0, "3/3": bounds, "-1/3": bounds}
    assert res["release_self_test"] == 0


def test_checked_build_matches_the_release_build(child_result):
    cases = child_result["cases"]
    assert len(cases) == 17
    for name, r in cases.items():
        assert r["device_error"] == 0, f"{name}: the checked build recorded {r['device_error']}"
        assert r["bit_identical"], f"{name}: checked and release results differ"
