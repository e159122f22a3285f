#!/usr/bin/env python
"""Benchmark of the gated delta-rule hot path on one GB300 (replicas on N GPUs).

Headline: GDN chunked forward, B=2, T=4096, H=Hg=16, K=V=128, bf16 q/k/v, fp32
g/beta, 64-token chunks, fp32 initial state in and final state out.  One step
is one library call over that batch (gate cumsum, intra-chunk solve + WY,
sequential state pass and output, all inside the call).  L2 is flushed
(a 512 MB write) before every step; CUDA events on the launch stream time
each step.  The same JSON line also carries, measured the same way, the
per-channel-gate (KDA) forward (B=1, T=8192, H=HV=32) and the decode step
(B=pool=256, HV=32, H=16, T = 1, 2, 4, bf16 state updated in place).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun every rank runs the same workload on its own GPU (independent
replicas, no collective on the data path); rank 0 prints one JSON line with the
whole-job throughput (tokens of all ranks / slowest rank's time).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "GDN chunk-fwd tokens/s and % roofline at 1 GB300; decode state GB/s vs HBM peak"
UNIT = "tokens/s"
WORKLOAD = ("GDN chunked prefill: B=2, T=4096, H=Hg=16, K=V=128, bf16 q/k/v, fp32 g/beta "
            "(logsigmoid(N(0,1)+3) per token), BT=64, h0 ~ N(0,0.1) fp32, final state returned")
FLUSH_BYTES = 512 << 20
# kernels one chunked-forward call launches on the tensor-core path: the
# parallel intra-chunk kernel and the sequential state/output kernel
LAUNCHES_PER_CALL = 2
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def log(*a):
    print(*a, file=sys.stderr, flush=True)


# ------------------------------------------------------------------ accounting

def gdn_bytes(B, T, H, Hg, K, V, N, h0=True, ht=True, elt=2):
    """Algorithmic HBM bytes of one chunked forward: every input read once, o written
    once, initial/final state read/written once."""
    per_token = Hg * K * elt * 2 + H * V * elt * 2 + H * 4 * 2
    return B * T * per_token + N * H * K * V * 4 * (int(h0) + int(ht))


def kda_bytes(B, T, H, HV, K, V, N, h0=False, ht=True, elt=2):
    per_token = H * K * elt * 2 + HV * V * elt * 2 + HV * K * 4 + HV * 4
    return B * T * per_token + N * HV * K * V * 4 * (int(h0) + int(ht))


def chunk_flops(B, T, H, K, V, BT=64):
    """6KV + 5 BT K per token and value head: w h, k^T v_new, q h (three BT x K x V
    GEMMs per chunk) and KK^T, w, u, qk^T, Aqk v_new counted on the triangle."""
    return B * T * H * (6 * K * V + 5 * BT * K)


def decode_state_bytes(B, HV, K, V):
    return 2 * B * HV * K * V * 2


def decode_total_bytes(B, T, H, HV, K, V):
    return (decode_state_bytes(B, HV, K, V) + B * T * (2 * H * K * 2 + 2 * HV * V * 2 + 2 * HV * 2)
            + 2 * HV * 4)


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


def traffic_record(kernel):
    """DRAM bytes per launch from the committed ncu summary, if it matches the
    current kernel source (sha of its .cu file)."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    for ln in open(path):
        f = ln.split()
        if len(f) < 3 or f[0] != kernel:
            continue
        kv = dict(x.split("=", 1) for x in f[1:] if "=" in x)
        src = os.path.join(ROOT, "gated_delta_rule_kk_gb300", "csrc", kv.get("source", ""))
        if not os.path.exists(src):
            return None
        sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:12]
        if sha != kv.get("sha"):
            return None
        return float(kv["bytes_per_launch"])
    return None


# ------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
        return False

    def summary(self):
        rows = []
        for ln in (self.out or "").splitlines():
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 7:
                continue
            try:
                rows.append((float(f[0]), float(f[1]), f[3:7]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        seen = sorted({names[i] for _, _, r in rows for i, x in enumerate(r) if x.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": seen, "samples": len(rows)}


# ------------------------------------------------------------------ timing

def time_steps(fn, steps, warmup, flush, stream):
    """Warm up, then time `steps` calls with events on `stream`, flushing L2 before
    each.  Returns per-step milliseconds."""
    for _ in range(warmup):
        flush.zero_()
        fn()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    for e0, e1 in evs:
        flush.zero_()
        e0.record(stream)
        fn()
        e1.record(stream)
    torch.cuda.synchronize()
    return [e0.elapsed_time(e1) for e0, e1 in evs]


def max_over_ranks(x, world, device):
    """The largest of every rank's `x` (the whole job takes as long as its
    slowest replica); `x` itself on one rank.  Works with gloo (CPU tensors)
    and NCCL (device tensors)."""
    if world <= 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(units_per_step, steps, world, total_ms):
    """Units all `world` replicas processed per second over the timed region."""
    return units_per_step * steps * world / (total_ms / 1e3)


def to_dev(inp, dev):
    return {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


# ------------------------------------------------------------------ our arm

def run_ours(args, rank, world, dev):
    import gated_delta_rule_kk_gb300 as gdn
    from gated_delta_rule_kk_gb300 import synth

    hbm, tc_burst, tc_sust, peak_src = measured_peaks()
    stream = torch.cuda.current_stream()
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)

    # ---- headline: GDN chunked forward
    inp = synth.gdn_prefill()
    dm = inp["dims"]
    d = to_dev(inp, dev)
    o = torch.empty_like(d["v"])
    ht = torch.empty((dm["N"], dm["H"], dm["K"], dm["V"]), dtype=torch.float32, device=dev)

    def step():
        gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], scale=d["scale"],
                          initial_state=d["h0"], out=o, final_state=ht)

    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(torch.cuda.current_device()) as clk:
        t_wall0 = time.perf_counter()
        ms = time_steps(step, args.steps, args.warmup, flush, stream)
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall0
    if world > 1:
        torch.distributed.barrier()
    status = gdn.gdn_check_device_error()
    if status != gdn.Status.OK:
        raise RuntimeError(f"device error during bench: {status.name}")
    tot_ms = max_over_ranks(sum(ms), world, dev)
    ms_step = tot_ms / args.steps
    tokens = dm["B"] * dm["T"]
    value = replica_throughput(tokens, args.steps, world, tot_ms)
    nbytes = gdn_bytes(dm["B"], dm["T"], dm["H"], dm["Hg"], dm["K"], dm["V"], dm["N"])
    flops = chunk_flops(dm["B"], dm["T"], dm["H"], dm["K"], dm["V"])
    achieved_gbs = nbytes / (ms_step / 1e3) / 1e9
    t_roof = max(nbytes / (hbm * 1e9), flops / (tc_burst * 1e12))
    result = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16 (bf16 inputs; hi/lo bf16 tensor-core products, fp32 accumulation and state)",
        "data": "synthetic (seeded numpy draws, see gated_delta_rule_kk_gb300/synth.py)",
        "config": {"workload": WORKLOAD, "global_batch": dm["B"] * world, "seq_len": dm["T"],
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "flushed (512 MB write) before every timed step"},
        "roofline": {"bound": "hbm", "achieved": achieved_gbs, "peak": hbm, "unit": "GB/s",
                     "frac": achieved_gbs / hbm, "traffic": traffic_record("gdn_chunk"),
                     "peak_source": peak_src, "algorithmic_bytes": nbytes,
                     "algorithmic_flops": flops,
                     "frac_of_roofline_time": t_roof / (ms_step / 1e3)},
        "gpu_launches": args.steps * LAUNCHES_PER_CALL,
        "clocks": clk.summary(),
        "wall_s_timed_region": t_wall,
    }

    # ---- end to end through the C-ABI host entry point: pinned host buffers in
    # and out, every host<->device copy inside the timed region (the library
    # overlaps them with the kernels piece by piece)
    pin = {k: (v.pin_memory() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    o_h = torch.empty(o.shape, dtype=o.dtype).pin_memory()
    ht_h = torch.empty(ht.shape, dtype=ht.dtype).pin_memory()
    keys = ("q", "k", "v", "g", "beta", "h0")
    h2d = sum(pin[k].numel() * pin[k].element_size() for k in keys)
    d2h = o_h.numel() * o_h.element_size() + ht_h.numel() * ht_h.element_size()
    del d, o, ht
    ws = torch.empty(gdn.gdn_chunk_host_workspace_bytes(pin["q"], pin["v"]), dtype=torch.uint8,
                     device=dev)

    def e2e_step():
        gdn.gdn_chunk_fwd_host(pin["q"], pin["k"], pin["v"], pin["g"], pin["beta"],
                               scale=pin["scale"], initial_state=pin["h0"], out=o_h,
                               final_state=ht_h, workspace=ws, stream=stream)

    e2e_ms = time_steps(e2e_step, min(args.steps, 10), 3, flush, stream)
    e2e_tot = max_over_ranks(sum(e2e_ms), world, dev)
    status = gdn.gdn_check_device_error()
    if status != gdn.Status.OK:
        raise RuntimeError(f"device error during the end-to-end run: {status.name}")
    result["e2e"] = {"value": replica_throughput(tokens, len(e2e_ms), world, e2e_tot), "unit": UNIT,
                     "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                     "entry_point": "gdn_chunk_fwd_host (host buffers, pinned)"}
    del pin, ws

    # ---- the other rows of the hot path, same timing rules
    rows = {}
    if not args.no_rows:
        rsteps = max(3, min(args.steps, 10))
        kin = synth.kda_prefill()
        km = kin["dims"]
        kd = to_dev(kin, dev)
        ko = torch.empty_like(kd["v"])
        kht = torch.empty((km["N"], km["H"], km["K"], km["V"]), dtype=torch.float32, device=dev)
        kms = time_steps(lambda: gdn.kda_chunk_fwd(kd["q"], kd["k"], kd["v"], kd["g"], kd["beta"],
                                                   out=ko, final_state=kht),
                         rsteps, max(3, args.warmup // 2), flush, stream)
        kt = statistics.mean(kms)
        kb = kda_bytes(km["B"], km["T"], km["Hg"], km["H"], km["K"], km["V"], km["N"])
        kf = chunk_flops(km["B"], km["T"], km["H"], km["K"], km["V"])
        rows["kda"] = {
            "workload": "KDA chunked prefill: B=1, T=8192, H=HV=32, K=V=128, bf16, per-channel "
                        "gate (chunk-local cumsum of logsigmoid(N(0,1)+4)), h0=0, ht returned",
            "tokens_per_s": km["B"] * km["T"] / (kt / 1e3), "ms_per_call": kt,
            "roofline": {"bound": "hbm", "achieved": kb / (kt / 1e3) / 1e9, "peak": hbm,
                         "unit": "GB/s", "frac": kb / (kt / 1e3) / 1e9 / hbm,
                         "algorithmic_bytes": kb, "algorithmic_flops": kf,
                         "traffic": traffic_record("kda_chunk")}}
        del kd, ko, kht, kin
        # packed sequences with grouped heads: 8 lengths in [64, 8192], Hg=4, H=16
        vin = synth.varlen_gqa()
        vm = vin["dims"]
        vd = to_dev(vin, dev)
        vo = torch.empty_like(vd["v"])
        vht = torch.empty((vm["N"], vm["H"], vm["K"], vm["V"]), dtype=torch.float32, device=dev)
        vms = time_steps(lambda: gdn.gdn_chunk_fwd(vd["q"], vd["k"], vd["v"], vd["g"], vd["beta"],
                                                   scale=vd["scale"], cu_seqlens=vd["cu_seqlens"],
                                                   out=vo, final_state=vht),
                         rsteps, max(3, args.warmup // 2), flush, stream)
        vt = statistics.mean(vms)
        vtok = vm["B"] * vm["T"]
        vb = gdn_bytes(vm["B"], vm["T"], vm["H"], vm["Hg"], vm["K"], vm["V"], vm["N"], h0=False)
        vf = chunk_flops(vm["B"], vm["T"], vm["H"], vm["K"], vm["V"])
        lens = (vd["cu_seqlens"][1:] - vd["cu_seqlens"][:-1]).tolist()
        rows["gdn_varlen"] = {
            "workload": f"GDN varlen GQA prefill: {vm['N']} packed sequences, lengths {lens} "
                        f"(sum {vtok}), Hg=4, H=16, K=V=128, bf16, h0=0, ht returned",
            "tokens_per_s": vtok / (vt / 1e3), "ms_per_call": vt,
            "roofline": {"bound": "hbm", "achieved": vb / (vt / 1e3) / 1e9, "peak": hbm,
                         "unit": "GB/s", "frac": vb / (vt / 1e3) / 1e9 / hbm,
                         "algorithmic_bytes": vb, "algorithmic_flops": vf,
                         "traffic": traffic_record("gdn_varlen")}}
        del vd, vo, vht, vin
        # few long chains: one sequence of 8192 tokens, two heads (8 chains of
        # 32 value columns on 152 SMs): the library's segment-parallel state
        # pass against one sequential chain per sequence
        fin = synth.prefill_inputs(7, 1, 8192, 2, 2, 128, 128, h0_std=0.1)
        fm = fin["dims"]
        fd = to_dev(fin, dev)
        fo = torch.empty_like(fd["v"])
        fht = torch.empty((1, 2, 128, 128), dtype=torch.float32, device=dev)
        nseg = gdn.gdn_chunk_segment_count(1, 8192, 2, 2, 128, 128)
        ftimes = {}
        for segs in (1, 0):
            fms = time_steps(lambda: gdn.gdn_chunk_fwd(fd["q"], fd["k"], fd["v"], fd["g"], fd["beta"],
                                                       scale=fd["scale"], initial_state=fd["h0"],
                                                       out=fo, final_state=fht, segments=segs),
                             rsteps, max(3, args.warmup // 2), flush, stream)
            ftimes[segs] = statistics.mean(fms)
        fb = gdn_bytes(1, 8192, 2, 2, 128, 128, 1)
        rows["gdn_few_chains"] = {
            "workload": "GDN chunked prefill with few long chains: B=1, T=8192, H=Hg=2, "
                        "K=V=128, bf16, h0 ~ N(0,0.1), ht returned",
            "segments_chosen": nseg, "ms_per_call": ftimes[0], "ms_one_chain": ftimes[1],
            "tokens_per_s": 8192 / (ftimes[0] / 1e3),
            "roofline": {"bound": "hbm", "achieved": fb / (ftimes[0] / 1e3) / 1e9, "peak": hbm,
                         "unit": "GB/s", "frac": fb / (ftimes[0] / 1e3) / 1e9 / hbm,
                         "algorithmic_bytes": fb, "traffic": traffic_record("gdn_few_chains")}}
        del fd, fo, fht, fin
        # chunk state pass (gated linear attention), per-token gate and per-key gate
        for sgate in ("g", "gk"):
            sin = synth.state_pass_inputs(5, 2, 4096, 16, 128, 128, sgate, h0_std=0.1)
            sm = sin["dims"]
            sk, sv = sin["k"].to(dev), sin["v"].to(dev)
            sg, sh0 = sin["gate_values"].to(dev), sin["h0"].to(dev)
            nchunk = sm["B"] * ((sm["T"] + 63) // 64)
            shs = torch.empty((nchunk, sm["H"], sm["K"], sm["V"]), dtype=torch.float32, device=dev)
            sht = torch.empty((sm["N"], sm["H"], sm["K"], sm["V"]), dtype=torch.float32, device=dev)
            sms = time_steps(lambda: gdn.gdn_chunk_state_fwd(sk, sv, gate=sgate, gate_values=sg,
                                                             initial_state=sh0, out_states=shs,
                                                             final_state=sht),
                             rsteps, max(3, args.warmup // 2), flush, stream)
            st_ = statistics.mean(sms)
            per_tok = sm["H"] * (sm["K"] + sm["V"]) * 2 + sg.numel() * 4 // (sm["B"] * sm["T"])
            sbytes = (sm["B"] * sm["T"] * per_tok + shs.numel() * 4
                      + 2 * sm["N"] * sm["H"] * sm["K"] * sm["V"] * 4)
            rows[f"state_pass_{sgate}"] = {
                "workload": f"chunk state pass (gated linear attention): B=2, T=4096, H=16, "
                            f"K=V=128, bf16 k/v, gate {sgate}, h0 given, fp32 chunk states "
                            f"[{nchunk},16,128,128] and final state",
                "tokens_per_s": sm["B"] * sm["T"] / (st_ / 1e3), "ms_per_call": st_,
                "roofline": {"bound": "hbm", "achieved": sbytes / (st_ / 1e3) / 1e9, "peak": hbm,
                             "unit": "GB/s", "frac": sbytes / (st_ / 1e3) / 1e9 / hbm,
                             "algorithmic_bytes": sbytes,
                             "traffic": traffic_record(f"state_pass_{sgate}")}}
            del sk, sv, sg, sh0, shs, sht, sin
        # backward state pass (dh recurrence), per-token gate
        gin = synth.state_grad_inputs(6, 2, 4096, 16, 16, 128, 128, "g", dht_std=0.1)
        gm = gin["dims"]
        gq, gdo = gin["q"].to(dev), gin["do"].to(dev)
        gg, gdht = gin["gate_values"].to(dev), gin["dht"].to(dev)
        nchunk = gm["B"] * ((gm["T"] + 63) // 64)
        gdh = torch.empty((nchunk, gm["HQ"], gm["K"], gm["V"]), dtype=torch.float32, device=dev)
        gdh0 = torch.empty((gm["N"], gm["HQ"], gm["K"], gm["V"]), dtype=torch.float32, device=dev)
        gms = time_steps(lambda: gdn.gdn_chunk_state_bwd(gq, gdo, gate="g", gate_values=gg,
                                                         dht=gdht, scale=gin["scale"],
                                                         out_states=gdh, dh0=gdh0),
                         rsteps, max(3, args.warmup // 2), flush, stream)
        gt_ = statistics.mean(gms)
        per_tok = gm["HQ"] * (gm["K"] + gm["V"]) * 2 + gg.numel() * 4 // (gm["B"] * gm["T"])
        gbytes = (gm["B"] * gm["T"] * per_tok + gdh.numel() * 4
                  + 2 * gm["N"] * gm["HQ"] * gm["K"] * gm["V"] * 4)
        rows["state_grad_g"] = {
            "workload": "backward chunk state pass (dh recurrence): B=2, T=4096, HQ=H=16, "
                        f"K=V=128, bf16 q/do, gate g, dht given, fp32 chunk gradients "
                        f"[{nchunk},16,128,128] and dh0",
            "tokens_per_s": gm["B"] * gm["T"] / (gt_ / 1e3), "ms_per_call": gt_,
            "roofline": {"bound": "hbm", "achieved": gbytes / (gt_ / 1e3) / 1e9, "peak": hbm,
                         "unit": "GB/s", "frac": gbytes / (gt_ / 1e3) / 1e9 / hbm,
                         "algorithmic_bytes": gbytes, "traffic": traffic_record("state_grad_g")}}
        del gq, gdo, gg, gdht, gdh, gdh0, gin
        for T in (1, 2, 3, 4):
            din = synth.decode(T)
            dd = to_dev(din, dev)
            m = din["dims"]
            dout = torch.empty_like(dd["v"])
            dms = time_steps(lambda: gdn.gdn_decode(dd["q"], dd["k"], dd["v"], dd["a"], dd["b"],
                                                    dd["A_log"], dd["dt_bias"], dd["state"],
                                                    scale=dd["scale"], out=dout),
                             rsteps, max(3, args.warmup // 2), flush, stream)
            dt = statistics.mean(dms)
            sb = decode_state_bytes(m["B"], m["HV"], m["K"], m["V"])
            tb = decode_total_bytes(m["B"], T, m["H"], m["HV"], m["K"], m["V"])
            rows[f"decode_t{T}"] = {
                "workload": f"GDN decode: B=pool=256, T={T}, H=16, HV=32, K=V=128, bf16 state",
                "us_per_call": dt * 1e3, "state_gb_per_s": sb / (dt / 1e3) / 1e9,
                "total_gb_per_s": tb / (dt / 1e3) / 1e9,
                "roofline": {"bound": "hbm", "achieved": tb / (dt / 1e3) / 1e9, "peak": hbm,
                             "unit": "GB/s", "frac": tb / (dt / 1e3) / 1e9 / hbm,
                             "state_frac": sb / (dt / 1e3) / 1e9 / hbm,
                             "algorithmic_bytes": tb, "traffic": traffic_record(f"decode_t{T}")}}
            del dd, dout, din
        status = gdn.gdn_check_device_error()
        if status != gdn.Status.OK:
            raise RuntimeError(f"device error during bench rows: {status.name}")
    result["rows"] = rows
    return result


# ------------------------------------------------------------------ oracle

def _headline_chain_specs():
    """One oracle call per (sequence, head) chain of the headline workload, its
    inputs sliced to that chain (the chains are independent)."""
    from gated_delta_rule_kk_gb300 import synth
    inp = synth.gdn_prefill()
    dm = inp["dims"]
    f = {k: inp[k].float().numpy() for k in ("q", "k", "v", "g", "beta", "h0")}
    specs = []
    for i in range(dm["B"] * dm["H"]):
        n, h = i % dm["B"], (i // dm["B"]) % dm["H"]
        hk = h // (dm["H"] // dm["Hg"])
        args = (f["q"][n:n + 1, :, hk:hk + 1], f["k"][n:n + 1, :, hk:hk + 1],
                f["v"][n:n + 1, :, h:h + 1], f["g"][n:n + 1, :, h:h + 1],
                f["beta"][n:n + 1, :, h:h + 1])
        specs.append(("gdn_recurrent", args,
                      dict(scale=inp["scale"], h0=f["h0"][n:n + 1, h:h + 1])))
    return specs, dm


def tiny_single_thread_s():
    """Seconds the oracle takes on the tiny fp32 workload (B=1, T=128, K=V=32)
    in this process, one thread."""
    from gated_delta_rule_kk_gb300 import synth
    from oracle import recurrence as R
    inp = synth.tiny()
    t0 = time.perf_counter()
    R.gdn_recurrent(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], scale=inp["scale"])
    return time.perf_counter() - t0


def oracle_sample(target_s):
    """Time the fp64 oracle on whole (sequence, head) chains of the headline
    workload, one chain per host core at a time, until about `target_s`
    seconds have passed.  Returns (token-equivalents per second, seconds,
    chains, cores)."""
    from oracle import parallel
    specs, dm = _headline_chain_specs()
    cores = parallel.default_workers()
    with parallel.ChainPool(cores) as pool:
        pool.map(specs[:cores])  # start the workers (not timed)
        t0 = time.perf_counter()
        chains = 0
        while True:
            batch = [specs[(chains + j) % len(specs)] for j in range(cores)]
            pool.map(batch)
            chains += cores
            el = time.perf_counter() - t0
            if el >= target_s:
                break
    # one chain is T tokens of one of H value heads: T / H token-equivalents
    tok = chains * dm["T"] / dm["H"]
    return tok / el, el, chains, cores


def run_reference(args):
    """The oracle on the host cores, as the reference arm: each step runs one
    whole (sequence, head) chain of the headline workload on every core."""
    from oracle import parallel
    specs, dm = _headline_chain_specs()
    cores = parallel.default_workers()
    times = []
    with parallel.ChainPool(cores) as pool:
        pool.map(specs[:cores])  # start the workers (not timed)
        for i in range(args.warmup + args.steps):
            batch = [specs[(i * cores + j) % len(specs)] for j in range(cores)]
            t0 = time.perf_counter()
            pool.map(batch)
            if i >= args.warmup:
                times.append(time.perf_counter() - t0)
    tok = cores * dm["T"] / dm["H"]
    value = tok / statistics.mean(times)
    sample = (f"per step one whole (sequence, head) chain of the headline workload on each of "
              f"{cores} host cores ({cores} x {dm['T']} tokens x 1 of {dm['H']} heads = "
              f"{tok:.0f} token-equivalents), fp64 numpy token recurrence")
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": statistics.mean(times) * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": WORKLOAD, "global_batch": dm["B"],
                                        "seq_len": dm["T"], "parallelism": "host CPU"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample, "tiny_single_thread_s": tiny_single_thread_s()},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# ------------------------------------------------------------------ main

def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-rows", action="store_true", help="skip the KDA and decode rows")
    ap.add_argument("--cpu-baseline-s", type=float, default=12.0)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return 0
        print(json.dumps(run_reference(args)), flush=True)
        return 0

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=dev)
    import __graft_entry__
    __graft_entry__.build()

    result = run_ours(args, rank, world, dev)
    if rank == 0:
        v, el, chains, cores = oracle_sample(args.cpu_baseline_s)
        result["cpu_baseline"] = {
            "value": v, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{chains} whole (sequence, head) chains of the headline workload, one "
                      f"per core at a time on {cores} cores ({el:.1f} s, fp64 numpy token "
                      f"recurrence)",
            "tiny_single_thread_s": tiny_single_thread_s()}
        print(json.dumps(result), flush=True)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
