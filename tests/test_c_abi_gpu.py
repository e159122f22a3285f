"""The C boundary used from plain C: tests/c_abi_program.c allocates its own
device buffers with the CUDA runtime and calls gdn_chunk_fwd (tensor-core
path: bf16, K = V = 128) and gdn_chunk_fwd_host (pageable host buffers); no
Python or PyTorch runs in that process.  Its outputs are checked against the
oracle here, and the two entry points against each other bit for bit."""
import os
import subprocess

import numpy as np
import pytest
import torch

from gated_delta_rule_kk_gb300 import gdn_chunk_fwd, synth
from oracle import recurrence as R

from _util import TOL_BF16, assert_close
from c_program import compile_program

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.contiguous().view(torch.int16).numpy().astype(np.uint16)


def test_plain_c_caller(tmp_path):
    B, T, H, Hg, K, V = 2, 300, 4, 2, 128, 128
    inp = synth.prefill_inputs(90, B, T, H, Hg, K, V, dtype=torch.bfloat16, h0_std=0.1)
    with open(tmp_path / "in.bin", "wb") as f:
        np.array([B, T, H, Hg, K, V], dtype=np.int32).tofile(f)
        np.array([inp["scale"]], dtype=np.float32).tofile(f)
        for key in ("q", "k", "v"):
            _bits(inp[key]).tofile(f)
        for key in ("g", "beta", "h0"):
            inp[key].contiguous().numpy().astype(np.float32).tofile(f)
    exe = compile_program(str(tmp_path))
    run = subprocess.run([exe, str(tmp_path / "in.bin"), str(tmp_path / "dev.bin"),
                          str(tmp_path / "host.bin")], capture_output=True, text=True, timeout=300)
    assert run.returncode == 0, run.stderr
    n_o, n_s = B * T * H * V, B * H * K * V

    def load(name):
        raw = np.fromfile(tmp_path / name, dtype=np.uint8)
        o_bits = raw[:2 * n_o].view(np.uint16).astype(np.uint32) << 16
        o = o_bits.view(np.float32).reshape(B, T, H, V)
        ht = raw[2 * n_o:].view(np.float32).reshape(B, H, K, V)
        return o, ht, raw

    o_d, ht_d, raw_d = load("dev.bin")
    o_h, ht_h, raw_h = load("host.bin")
    assert raw_d.size == 2 * n_o + 4 * n_s
    assert np.array_equal(raw_d, raw_h), "host entry point differs from the device entry point"
    o_ref, ht_ref = R.gdn_recurrent(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                                    scale=inp["scale"], h0=inp["h0"])
    # the same call with o in fp32 (through the binding): the C caller's bf16 o
    # is its round-to-nearest-even bit for bit, and the fp32 o meets the bound
    d = {k2: (v2.cuda() if isinstance(v2, torch.Tensor) else v2) for k2, v2 in inp.items()}
    o32, ht32 = gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], scale=d["scale"],
                              initial_state=d["h0"], out_dtype=torch.float32)
    o16 = torch.from_numpy(o_d.copy()).to(torch.bfloat16)
    assert torch.equal(o16, o32.cpu().to(torch.bfloat16))
    assert np.array_equal(ht_d, ht32.cpu().numpy())
    assert_close(o32, o_ref, TOL_BF16, "o")
    assert_close(ht_d, ht_ref, TOL_BF16, "ht")
