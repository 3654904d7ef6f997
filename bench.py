#!/usr/bin/env python
"""Benchmark of the attention hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step = one fused attention forward over the prefill workload
(B=1, H=64, Nq=Nk=8192, d=128, BF16, no mask), the configuration the
headline metric is quoted on. The same run also times, each with its own
warm-up and timed loop, the causal workload (B=2, H=32, 8192^2, causal) and
the backward pass on the prefill shape and the split-KV decode workload
(B=1, H=32, Nk=131072, d=128, 64 splits), and reports them as sub-objects. Rank 0 prints one JSON line.

Inputs are larger than L2 (the prefill inputs are 384 MiB, decode K+V 2 GiB),
so no L2 flush is done between iterations.

For N > 1 (torchrun), every rank runs an independent replica of the
workload on its own GPU (no collective on the data path: the problems are
independent); a barrier and a max over ranks bracket the timed region and
`value` counts the work of all ranks ("scaling": "weak").

--impl reference times the FP64 CPU oracle (the reference implementation
the GPU results are checked against) on a bounded sample of the same
workload, on the host cores.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from online_softmax_02_gb300 import workloads as W  # noqa: E402

METRIC = "attn fwd TFLOP/s & % BF16 tcgen05 peak; split-KV decode HBM GB/s, % of peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# DRAM traffic per launch measured with ncu (dram__bytes_read.sum +
# dram__bytes_write.sum), keyed by the source file of the kernel and its
# SHA-256 at capture time; reported as null when the source has changed.
FWD_SHA = "a90cb2b22764f1bdc2d34a18a6895e271d9c4bb11e6627e2d1a858e49361d061"
DECODE_SHA = "7662e21a7cbf9d910c984e96fe5bbcb4d5fb74d6a0723a8a014cf6588b014b54"
BWD_SHA = "fdbb1b59f065fa898430ea6f21ebe4222e70637f063194ae96c1c755f5445251"
NCU_TRAFFIC = {
    # dram__bytes_read.sum + dram__bytes_write.sum of the dominant kernel, one
    # launch at the full bench workload, 1-pass ncu capture; valid while the
    # kernel source is unchanged.
    "fwd_bf16": {"file": "fwd_sm103.cu", "sha256": FWD_SHA,
                 "bytes_per_launch": 402833152 + 114113792,
                 "workload": "prefill_B1_H64_N8192_d128_bf16"},
    "fwd_bf16_causal": {"file": "fwd_sm103.cu", "sha256": FWD_SHA,
                        "bytes_per_launch": 402730240 + 112965376,
                        "workload": "causal_B2_H32_N8192_d128_bf16"},
    "fwd_bf16_masked": {"file": "fwd_sm103.cu", "sha256": FWD_SHA,
                        "bytes_per_launch": 245462528 + 114034176,
                        "workload": "masked_B8_H16_N4096_d128_bf16_window1024_padded"},
    "fwd_e4m3": {"file": "fwd_sm103.cu", "sha256": FWD_SHA,
                 "bytes_per_launch": 201401088 + 102112256,
                 "workload": "prefill_B1_H64_N8192_d128_e4m3"},
    "decode": {"file": "decode.cu", "sha256": DECODE_SHA,
               "bytes_per_launch": 2147542528 + 3053312 + 1072640,
               "workload": "decode_B1_H32_Nk131072_d128_bf16_splits64 (split and combine kernels)"},
    "backward": {"file": "bwd_sm103.cu", "sha256": BWD_SHA,
                 "bytes_per_launch": (270548736 + 219377920) + (809734144 + 489436928) +
                                     (268457728 + 86584064),
                 "workload": "prefill_B1_H64_N8192_d128_bf16 backward (prep, dK/dV/dQ and "
                             "dQ convert kernels)"},
    "softmax": {"file": "softmax.cu",
                "sha256": "9a40d74a21d385c58919240ac5c54e555e31ccc3e2bd568868bc0f51f562068d",
                "bytes_per_launch": 537604096 + 475967488,
                "workload": "softmax_rows_4096x32768_f32"},
}


# ------------------------------------------------------------------ helpers
def kernel_sha(name):
    path = os.path.join(ROOT, "online_softmax_02_gb300", "csrc", name)
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()


def traffic_for(key, units_scale=1.0):
    rec = NCU_TRAFFIC.get(key)
    if not rec or rec.get("sha256") != kernel_sha(rec["file"]):
        return None
    return rec["bytes_per_launch"] * units_scale


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained")}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def visible_pairs(w: W.Workload, seqlens=None) -> int:
    """Number of (query, key) pairs the mask leaves visible, summed over
    batch and heads (closed form per row)."""
    Nq, Nk = w.Nq, w.Nk
    total = 0
    for b in range(w.B):
        L = Nk if seqlens is None else int(min(max(int(seqlens[b]), 0), Nk))
        i = np.arange(Nq, dtype=np.int64)
        hi = np.full(Nq, L, dtype=np.int64)                 # keys [lo, hi)
        if w.mask_kind & (W.MASK_CAUSAL | W.MASK_WINDOW):
            hi = np.minimum(hi, i + 1)
        lo = np.zeros(Nq, dtype=np.int64)
        if w.mask_kind & W.MASK_WINDOW:
            lo = np.maximum(0, i - w.window + 1)
        total += int(np.maximum(hi - lo, 0).sum())
    return total * w.H


def flops(w, seqlens=None):
    """4 d FLOPs per visible pair: 2 d for q.k and 2 d for p v."""
    return 4.0 * w.d * visible_pairs(w, seqlens)


class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons every 200 ms."""
    FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid):
        self.uuid = uuid
        self.proc = None
        self.lines = []
        self.error = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError as e:
            self.error = str(e)
        time.sleep(0.25)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        time.sleep(0.25)
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.error or not self.lines:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [],
                    "note": self.error or "no nvidia-smi samples"}
        rows = []
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            if self.uuid and self.uuid not in parts[0] and parts[0] not in self.uuid:
                continue
            rows.append(parts)
        if not rows:
            rows = [[p.strip() for p in ln.split(",")] for ln in self.lines if ln.count(",") >= 8]
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for n, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        loaded = [s for s in sm if mx and s > 0.3 * max(mx)] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(rows)}


def gpu_uuid(dev):
    try:
        u = torch.cuda.get_device_properties(dev).uuid
        return "GPU-" + str(u)
    except Exception:   # noqa: BLE001
        return None


# --------------------------------------------------------------- timing
def time_loop(fn, steps, warmup, stream, dist_on):
    """W warm-up calls, then K timed calls bracketed by barrier + sync;
    returns (total ms on this rank via CUDA events, per-launch ms list)."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    if dist_on:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        start.record(stream)
        for a, b in evs:
            a.record(stream)
            fn()
            b.record(stream)
        end.record(stream)
    torch.cuda.synchronize()
    if dist_on:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    total = start.elapsed_time(end)
    per = [a.elapsed_time(b) for a, b in evs]
    return total, per


def max_over_ranks(x, dist_on, device="cuda"):
    """The slowest rank's time: every rank gets the max."""
    if not dist_on:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_step, world, steps, total_ms):
    """Units processed by all ranks per second (replicas: each rank does
    `units_per_step` per step), timed by the slowest rank."""
    return units_per_step * world * steps / (total_ms * 1e-3)


# -------------------------------------------------------------- our arm
def run_ours(args, rank, world, dist_on):
    import online_softmax_02_gb300 as attn
    attn.load()
    # another build for the forward sections (--lib), or the default library
    args.fwd_lib = attn.open_build(os.path.abspath(args.lib)) if args.lib else None
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(dev)
    peaks, peak_src = load_peaks()

    result = {}
    # ---------------- prefill (headline)
    w = W.PREFILL
    if args.heads:
        w = dataclasses.replace(w, H=args.heads, name="%s_H%d" % (w.name, args.heads))
    if args.only not in ("all", "prefill"):
        return run_sections(args, rank, world, dist_on, dev, stream, peaks, result)
    x = W.generate(w)
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)

    def step():
        attn.attn_fwd(q, k, v, o=o, lse=lse, mask_kind=w.mask_kind, stream=stream,
                      lib=args.fwd_lib)

    with ClockSampler(gpu_uuid(dev)) as clk:
        total_ms, per = time_loop(step, args.steps, args.warmup, stream, dist_on)
    attn.attn_check_device_error(stream, lib=args.fwd_lib)
    total_ms = max_over_ranks(total_ms, dist_on)
    fl = flops(w)
    ms_step = total_ms / args.steps
    value = whole_job_rate(fl, world, args.steps, total_ms) / 1e12
    launch_ms = statistics.mean(per)
    achieved = fl / (launch_ms * 1e-3) / 1e12
    roofline = {"bound": "tensor", "achieved": round(achieved, 2),
                "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": round(achieved / peaks["bf16_tflops"], 4),
                "traffic": traffic_for("fwd_bf16", w.H / W.PREFILL.H),
                "peak_source": "%s bf16_tflops (burst) from MEASURED_PEAKS.json" % peak_src
                if peak_src == "measured" else "fallback 1.9 PFLOP/s bf16 burst",
                "kernel": "fwd_sm103_kernel<128>",
                "algorithmic_flops_per_launch": fl}

    # ---------------- e2e: host (pinned) inputs and outputs through the C entry
    # point attn_fwd_host, copies in and out inside the timed region,
    # pipelined with the kernel by groups of heads
    hq, hk, hv = (x[n].pin_memory() for n in ("q", "k", "v"))
    ho = torch.empty(o.shape, dtype=o.dtype).pin_memory()
    hl = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    del q, k, v
    pipe = attn.HostPipeline(w.B, w.H, w.Nq, w.Nk, w.d, device=dev, chunks=args.e2e_chunks,
                             slots=args.e2e_slots)

    def e2e_step():
        attn.attn_fwd_from_host(hq, hk, hv, ho, hl, mask_kind=w.mask_kind, pipeline=pipe,
                                stream=stream)

    e_steps = max(3, args.steps // 4)
    e_total, _ = time_loop(e2e_step, e_steps, args.warmup, stream, dist_on)
    attn.attn_check_device_error(stream)
    e_total = max_over_ranks(e_total, dist_on)
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv))
    d2h = ho.numel() * ho.element_size() + hl.numel() * hl.element_size()
    e2e = {"value": round(fl * world * e_steps / (e_total * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
           "ms_per_step": round(e_total / e_steps, 4),
           "api": "attn_fwd_host (C ABI; host buffers, device workspace, caller's stream)",
           "head_groups": pipe.chunks, "device_slots": pipe.slots,
           "gpu_launches_per_step": attn.attn_fwd_host_groups(w.B, w.H, pipe.chunks),
           "h2d_d2h_GBps": round((h2d + d2h) / (e_total / e_steps * 1e-3) / 1e9, 1)}
    # the e2e result must equal the device-resident result
    e2e["matches_device_result"] = bool(torch.equal(ho.to(dev), o))
    del pipe

    result.update({
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic (seeded N(0,1), rounded to BF16)",
        "config": dict(w.describe(), **{"parallelism": "replicas" if world > 1 else "single",
                                        "l2": "inputs larger than L2 (384 MiB); no flush",
                                        "flop_count": "4*d per visible (query, key) pair"},
                       **({"library": args.lib} if args.lib else {})),
        "gpu_launches": args.steps,
        "e2e": e2e,
        "roofline": roofline,
        "clocks": clk.summary(),
    })
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(w, x, o, lse, args, args.cpu_seconds)
    del o, lse, x
    return run_sections(args, rank, world, dist_on, dev, stream, peaks, result)


def run_sections(args, rank, world, dist_on, dev, stream, peaks, result):
    """The causal and split-KV decode workloads (sub-objects of the line)."""
    import online_softmax_02_gb300 as attn
    if args.only not in ("all", "causal"):
        return run_masked_section(args, rank, world, dist_on, dev, stream, peaks, result)
    # ---------------- causal workload
    wc = W.CAUSAL
    if args.batch:
        wc = dataclasses.replace(wc, B=args.batch, name="%s_B%d" % (wc.name, args.batch))
    xc = W.generate(wc)
    qc, kc, vc = (xc[n].to(dev) for n in ("q", "k", "v"))
    oc = torch.empty_like(qc)
    lc = torch.empty(qc.shape[:3], dtype=torch.float32, device=dev)

    def step_c():
        attn.attn_fwd(qc, kc, vc, o=oc, lse=lc, mask_kind=wc.mask_kind, stream=stream,
                      lib=args.fwd_lib)

    c_total, c_per = time_loop(step_c, args.steps, args.warmup, stream, dist_on)
    attn.attn_check_device_error(stream, lib=args.fwd_lib)
    c_total = max_over_ranks(c_total, dist_on)
    flc = flops(wc)
    causal = {"config": wc.describe(), "ms_per_step": round(c_total / args.steps, 4),
              "value": round(flc * world * args.steps / (c_total * 1e-3) / 1e12, 2),
              "unit": "TFLOP/s", "flop_count": "causal (visible pairs only)",
              "gpu_launches_per_step": 1,
              "dense_equivalent_tflops": round(4.0 * wc.d * wc.B * wc.H * wc.Nq * wc.Nk * world *
                                               args.steps / (c_total * 1e-3) / 1e12, 2),
              "roofline": tensor_roofline(flc, c_per, peaks, "fwd_bf16_causal",
                                          "fwd_sm103_kernel<128> (causal)", wc.B / W.CAUSAL.B)}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        causal["cpu_baseline"] = cpu_baseline(wc, xc, oc, lc, args, args.cpu_seconds / 2)
    del qc, kc, vc, oc, lc, xc
    result["causal"] = causal
    return run_masked_section(args, rank, world, dist_on, dev, stream, peaks, result)


def run_masked_section(args, rank, world, dist_on, dev, stream, peaks, result):
    """Sliding window 1024 plus padding, B8 H16 4096^2 (reported, no target)."""
    import online_softmax_02_gb300 as attn
    if args.only not in ("all", "masked"):
        return run_fp8_section(args, rank, world, dist_on, dev, stream, peaks, result)
    wm = W.MASKED
    if args.batch:
        wm = dataclasses.replace(wm, B=args.batch, name="%s_B%d" % (wm.name, args.batch))
    xm = W.generate(wm)
    qm, km, vm = (xm[n].to(dev) for n in ("q", "k", "v"))
    sl = xm["seqlens_k"].to(dev)
    om = torch.empty_like(qm)
    lm = torch.empty(qm.shape[:3], dtype=torch.float32, device=dev)

    def step_m():
        attn.attn_fwd(qm, km, vm, o=om, lse=lm, mask_kind=wm.mask_kind, window=wm.window,
                      seqlens_k=sl, stream=stream, lib=args.fwd_lib)

    m_total, m_per = time_loop(step_m, args.steps, args.warmup, stream, dist_on)
    attn.attn_check_device_error(stream, lib=args.fwd_lib)
    m_total = max_over_ranks(m_total, dist_on)
    flm = flops(wm, xm["seqlens_k"].numpy())
    result["masked"] = {
        "config": wm.describe(), "ms_per_step": round(m_total / args.steps, 4),
        "value": round(flm * world * args.steps / (m_total * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
        "flop_count": "visible pairs only (window and padding)", "gpu_launches_per_step": 1,
        "roofline": tensor_roofline(flm, m_per, peaks, "fwd_bf16_masked",
                                    "fwd_sm103_kernel<128> (window + padding)",
                                    wm.B / W.MASKED.B)}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["masked"]["cpu_baseline"] = cpu_baseline(wm, xm, om, lm, args,
                                                        args.cpu_seconds / 2)
    del qm, km, vm, om, lm, xm
    return run_fp8_section(args, rank, world, dist_on, dev, stream, peaks, result)


def run_fp8_section(args, rank, world, dist_on, dev, stream, peaks, result):
    """The prefill workload with Q, K, V stored as E4M3 (attn_fwd_fp8)."""
    import online_softmax_02_gb300 as attn
    if args.only not in ("all", "fp8"):
        return run_backward_section(args, rank, world, dist_on, dev, stream, peaks, result)
    w = W.PREFILL
    if args.heads:
        w = dataclasses.replace(w, H=args.heads, name="%s_H%d" % (w.name, args.heads))
    x = W.generate_fp8(w)
    w = dataclasses.replace(w, name=w.name.replace("bf16", "e4m3"))
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    o = torch.empty(q.shape, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)

    def step_f():
        attn.attn_fwd_fp8(q, k, v, x["descale_q"], x["descale_k"], x["descale_v"], o=o, lse=lse,
                          stream=stream, lib=args.fwd_lib)

    f_total, f_per = time_loop(step_f, args.steps, args.warmup, stream, dist_on)
    attn.attn_check_device_error(stream, lib=args.fwd_lib)
    f_total = max_over_ranks(f_total, dist_on)
    fl = flops(w)
    achieved = fl / (statistics.mean(f_per) * 1e-3) / 1e12
    peak8 = 2.0 * peaks["bf16_tflops"]
    result["fp8"] = {
        "config": dict(w.describe(), dtype="e4m3", descale="per tensor, power of two"),
        "ms_per_step": round(f_total / args.steps, 4),
        "value": round(whole_job_rate(fl, world, args.steps, f_total) / 1e12, 2),
        "unit": "TFLOP/s", "gpu_launches_per_step": 1,
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": round(peak8, 1),
                     "unit": "TFLOP/s", "frac": round(achieved / peak8, 4),
                     "traffic": traffic_for("fwd_e4m3", w.H / W.PREFILL.H),
                     "peak_note": "measured bf16 burst x 2 (nominal e4m3 / bf16 dense ratio)"}}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        xr = {n: (x[n].float() * x["descale_" + n]) for n in ("q", "k", "v")}
        result["fp8"]["cpu_baseline"] = cpu_baseline(w, xr, o, lse, args, args.cpu_seconds / 4)
        result["fp8"]["cpu_baseline"]["sample"] += " (E4M3 inputs dequantised exactly to FP32)"
    del q, k, v, o, lse, x
    return run_backward_section(args, rank, world, dist_on, dev, stream, peaks, result)


def run_backward_section(args, rank, world, dist_on, dev, stream, peaks, result):
    """Backward pass on the prefill shape (B1 H64 8192^2 d128, no mask)."""
    import online_softmax_02_gb300 as attn
    if args.only not in ("all", "backward"):
        return run_decode_section(args, rank, world, dist_on, dev, stream, peaks, result)
    w = W.PREFILL
    if args.heads:
        w = dataclasses.replace(w, H=args.heads, name="%s_H%d" % (w.name, args.heads))
    x = W.generate(w)
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    g = torch.Generator("cpu").manual_seed(w.seed + 1)
    do = torch.randn(q.shape, generator=g, dtype=torch.float32).to(torch.bfloat16).to(dev)
    o, lse = attn.attn_fwd(q, k, v, mask_kind=w.mask_kind)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(attn.attn_bwd_workspace_bytes(w.B, w.H, w.Nq, w.d, lib=args.fwd_lib),
                     dtype=torch.uint8, device=dev)

    def step_b():
        attn.attn_bwd(q, k, v, o, do, lse, dq=dq, dk=dk, dv=dv, mask_kind=w.mask_kind,
                      workspace=ws, stream=stream, lib=args.fwd_lib)

    b_steps = max(3, args.steps // 4)
    b_total, b_per = time_loop(step_b, b_steps, args.warmup, stream, dist_on)
    attn.attn_check_device_error(stream, lib=args.fwd_lib)
    b_total = max_over_ranks(b_total, dist_on)
    fl = 2.5 * flops(w)          # five products of 2 d FLOPs per visible pair
    b_ms = statistics.mean(b_per)
    achieved = fl / (b_ms * 1e-3) / 1e12
    result["backward"] = {
        "metric": "attn bwd TFLOP/s", "config": w.describe(),
        "ms_per_step": round(b_total / b_steps, 4),
        "value": round(whole_job_rate(fl, world, b_steps, b_total) / 1e12, 2), "unit": "TFLOP/s",
        "flop_count": "2.5x forward (5 products: S, dP, dV, dK, dQ); at d = 128 the kernels "
                      "execute exactly these (dQ accumulated by the keys-outer kernel)",
        "gpu_launches_per_step": 3,
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2),
                     "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": round(achieved / peaks["bf16_tflops"], 4),
                     "traffic": traffic_for("backward", w.H / W.PREFILL.H),
                     "note": "time and DRAM traffic of the three launches per step"}}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["backward"]["cpu_baseline"] = cpu_baseline_backward(w, x, do, dq, dk, dv)
    del q, k, v, do, o, lse, dq, dk, dv, ws, x
    return run_decode_section(args, rank, world, dist_on, dev, stream, peaks, result)


def run_decode_section(args, rank, world, dist_on, dev, stream, peaks, result):
    import online_softmax_02_gb300 as attn
    if args.only not in ("all", "decode"):
        return run_softmax_section(args, rank, world, dist_on, dev, stream, peaks, result)
    # ---------------- split-KV decode
    wd = W.DECODE
    if args.decode_nk:
        wd = dataclasses.replace(wd, Nk=args.decode_nk, name="%s_Nk%d" % (wd.name, args.decode_nk))
    xd = W.generate(wd)
    qd, kd, vd = (xd[n].to(dev) for n in ("q", "k", "v"))
    od = torch.empty_like(qd)
    ld = torch.empty((wd.B, wd.H, 1), dtype=torch.float32, device=dev)
    ws = torch.empty(attn.attn_decode_workspace_bytes(wd.B, wd.H, wd.d, wd.num_splits),
                     dtype=torch.uint8, device=dev)

    def step_d():
        attn.attn_decode_splitkv(qd, kd, vd, o=od, lse=ld, num_splits=wd.num_splits,
                                 workspace=ws, stream=stream)

    d_total, d_per = time_loop(step_d, args.steps, args.warmup, stream, dist_on)
    attn.attn_check_device_error(stream)
    d_total = max_over_ranks(d_total, dist_on)
    kv_bytes = 2 * wd.B * wd.H * wd.Nk * wd.d * 2
    alg_bytes = kv_bytes + 2 * wd.B * wd.H * wd.d * 2 + wd.B * wd.H * 4
    d_ms = statistics.mean(d_per)
    gbs = alg_bytes / (d_ms * 1e-3) / 1e9
    decode = {"metric": "split-KV decode HBM GB/s", "config": wd.describe(),
              "ms_per_step": round(d_total / args.steps, 4),
              "value": round(alg_bytes * world * args.steps / (d_total * 1e-3) / 1e9, 1),
              "unit": "GB/s", "gpu_launches_per_step": 2,
              "workspace_bytes_per_step": int(2 * ws.numel()),
              "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"],
                           "unit": "GB/s", "frac": round(gbs / peaks["hbm_gbs"], 4),
                           "traffic": traffic_for("decode", wd.Nk / W.DECODE.Nk),
                           "algorithmic_bytes_per_step": alg_bytes,
                           "note": "time is both launches (split + combine) per step"}}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        decode["cpu_baseline"] = cpu_baseline_decode(wd, xd, od, ld, args.cpu_seconds / 2)
    del qd, kd, vd, xd
    result["decode"] = decode
    return run_softmax_section(args, rank, world, dist_on, dev, stream, peaks, result)


def run_softmax_section(args, rank, world, dist_on, dev, stream, peaks, result):
    """Standalone row softmax, [4096, 32768] FP32."""
    import online_softmax_02_gb300 as attn
    if args.only not in ("all", "softmax"):
        return result
    x = W.softmax_inputs(rows=args.softmax_rows or W.SOFTMAX_ROWS).to(dev)
    y = torch.empty_like(x)
    lse = torch.empty(x.shape[0], dtype=torch.float32, device=dev)

    def step_s():
        attn.attn_softmax_rows(x, y=y, lse=lse, stream=stream)

    s_total, s_per = time_loop(step_s, args.steps, args.warmup, stream, dist_on)
    attn.attn_check_device_error(stream)
    s_total = max_over_ranks(s_total, dist_on)
    alg = 2 * x.numel() * x.element_size() + lse.numel() * 4     # read x once, write y and lse
    gbs = alg / (statistics.mean(s_per) * 1e-3) / 1e9
    result["softmax"] = {
        "metric": "row softmax HBM GB/s",
        "config": {"workload": "softmax_rows_%dx%d_f32" % tuple(x.shape),
                   "rows": x.shape[0], "n": x.shape[1]},
        "ms_per_step": round(s_total / args.steps, 4),
        "value": round(whole_job_rate(alg, world, args.steps, s_total) / 1e9, 1), "unit": "GB/s",
        "gpu_launches_per_step": 1,
        "bytes_note": "algorithmic bytes = one HBM read of x, one write of y, the lse; the "
                      "two-pass method's second read of each row is served by L2 (rows of "
                      "128 KiB, 512 threads per row)",
        "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": round(gbs / peaks["hbm_gbs"], 4),
                     "traffic": traffic_for("softmax", x.shape[0] / W.SOFTMAX_ROWS)}}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["softmax"]["cpu_baseline"] = cpu_baseline_softmax(x, y, lse, args.cpu_seconds / 4)
    del x, y, lse
    if not args.no_naive:
        result["softmax"]["naive_attention_context"] = naive_attention_context(args, dev, stream,
                                                                               peaks)
    return result


def naive_attention_context(args, dev, stream, peaks):
    """Context only (not a product path): attention with the score matrix in
    HBM, as costed in P1 "Now the cost" -- S = scale*Q K^T written by a library
    GEMM, read by the row softmax which writes P, P read by a second library
    GEMM -- beside the fused forward on the same inputs (prefill shape)."""
    import online_softmax_02_gb300 as attn
    w = W.PREFILL
    if args.heads:
        w = dataclasses.replace(w, H=args.heads)
    x = W.generate(w)
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    qs = (q.float() * w.scale).to(torch.bfloat16)      # scale folded into Q (context only)
    B, H, N, d = q.shape
    S = torch.empty(B, H, N, N, dtype=torch.bfloat16, device=dev)
    P = torch.empty_like(S)
    o = torch.empty_like(q)
    lse = torch.empty(B * H * N, dtype=torch.float32, device=dev)
    fl = flops(w)

    def naive():
        with torch.cuda.stream(stream):
            torch.matmul(qs, k.transpose(-1, -2), out=S)
            attn.attn_softmax_rows(S.view(-1, N), y=P.view(-1, N), lse=lse, stream=stream)
            torch.matmul(P, v, out=o)

    def softmax_only():
        attn.attn_softmax_rows(S.view(-1, N), y=P.view(-1, N), lse=lse, stream=stream)

    def fused():
        attn.attn_fwd(q, k, v, o=o, mask_kind=w.mask_kind, stream=stream)

    steps, warm = 10, 3
    t_naive = time_loop(naive, steps, warm, stream, False)[0] / steps
    t_sm = time_loop(softmax_only, steps, warm, stream, False)[0] / steps
    t_fused = time_loop(fused, steps, warm, stream, False)[0] / steps
    attn.attn_check_device_error(stream)
    score_bytes = 4 * S.numel() * S.element_size()     # S written + read, P written + read
    out = {"workload": w.name, "score_matrix_bytes_each": S.numel() * S.element_size(),
           "score_traffic_bytes": score_bytes,
           "score_traffic_floor_ms": round(score_bytes / (peaks["hbm_gbs"] * 1e9) * 1e3, 3),
           "naive_ms": round(t_naive, 3), "naive_softmax_ms": round(t_sm, 3),
           "fused_ms": round(t_fused, 3), "naive_over_fused": round(t_naive / t_fused, 2),
           "naive_tflops": round(fl / (t_naive * 1e-3) / 1e12, 1),
           "fused_tflops": round(fl / (t_fused * 1e-3) / 1e12, 1),
           "gemms": "torch.matmul (cuBLAS), BF16 S and P; the softmax is attn_softmax_rows"}
    del S, P
    torch.cuda.empty_cache()
    return out


def tensor_roofline(fl, per_launch_ms, peaks, traffic_key, kernel, units_scale=1.0):
    """Roofline of a forward launch against the measured dense BF16 burst."""
    achieved = fl / (statistics.mean(per_launch_ms) * 1e-3) / 1e12
    return {"bound": "tensor", "achieved": round(achieved, 2), "peak": peaks["bf16_tflops"],
            "unit": "TFLOP/s", "frac": round(achieved / peaks["bf16_tflops"], 4),
            "traffic": traffic_for(traffic_key, units_scale), "kernel": kernel,
            "algorithmic_flops_per_launch": fl}


# ------------------------------------------------------ oracle on the host
def row_visible_keys(w, rows, seqlens=None):
    """Visible keys of each flat row (b*H+h)*Nq+i under the workload's mask."""
    rows = np.asarray(rows, np.int64)
    i = rows % w.Nq
    b = rows // (w.H * w.Nq)
    L = np.full(rows.shape, w.Nk, np.int64)
    if seqlens is not None:
        L = np.clip(np.asarray(seqlens, np.int64)[b], 0, w.Nk)
    hi = L.copy()
    if w.mask_kind & (W.MASK_CAUSAL | W.MASK_WINDOW):
        hi = np.minimum(hi, i + 1)
    lo = np.zeros_like(i)
    if w.mask_kind & W.MASK_WINDOW:
        lo = np.maximum(0, i - w.window + 1)
    return np.maximum(hi - lo, 0)


def oracle_sample(w, x, n_rows, seed=0):
    import oracle
    orc = oracle.Oracle()
    rng = np.random.default_rng(seed)
    rows = np.sort(rng.choice(w.B * w.H * w.Nq, size=n_rows, replace=False))
    qn, kn, vn = (x[n].float().numpy() for n in ("q", "k", "v"))
    sl = x.get("seqlens_k")
    sl = None if sl is None else sl.numpy()
    threads = oracle.default_threads()
    t0 = time.perf_counter()
    ro, rl = orc.attention(qn, kn, vn, w.scale, w.mask_kind, w.window, sl, rows=rows,
                           threads=threads)
    dt = time.perf_counter() - t0
    return rows, ro, rl, dt, threads


def cpu_baseline(w, x, o_gpu, lse_gpu, args, seconds):
    """The FP64 oracle, as it stands, on a bounded sample of rows of the
    same workload, timed on the host cores (about `seconds` of CPU work);
    also reports its agreement with the GPU output on those rows."""
    sl = x.get("seqlens_k")
    sl = None if sl is None else sl.numpy()
    # calibrate on a small sample, then size the sample to ~seconds
    rows, _, _, dt, _ = oracle_sample(w, x, 64, seed=1)
    n = int(min(w.B * w.H * w.Nq, max(64, 64 * seconds / max(dt, 1e-3))))
    rows, ro, rl, dt, threads = oracle_sample(w, x, n, seed=2)
    fl = 4.0 * w.d * float(row_visible_keys(w, rows, sl).sum())
    idx = torch.from_numpy(rows).to(o_gpu.device)
    got = o_gpu.float().reshape(-1, w.d)[idx].cpu().numpy()
    got_l = lse_gpu.reshape(-1)[idx].cpu().double().numpy()
    fin = np.isfinite(rl)
    return {"value": round(fl / dt / 1e12, 6), "unit": "TFLOP/s", "cores": threads,
            "kind": "oracle", "seconds": round(dt, 2),
            "sample": "%d random query rows (each with its visible keys) of the %s workload"
                      % (n, w.name),
            "max_abs_err_gpu_vs_oracle": float(np.abs(got - ro).max()),
            "max_abs_lse_err_gpu_vs_oracle": float(np.abs(got_l[fin] - rl[fin]).max())
            if fin.any() else 0.0,
            "lse_neginf_pattern_matches": bool(np.array_equal(np.isneginf(got_l), ~fin))}


def cpu_baseline_decode(w, x, o_gpu, lse_gpu, seconds):
    """The FP64 oracle on the decode workload's first heads (as many as fit in
    about `seconds` of CPU work, every key of each), in the decode metric's
    unit: algorithmic bytes of those heads per second."""
    import oracle
    orc = oracle.Oracle()
    threads = oracle.default_threads()

    def run(nh):
        qn, kn, vn = (x[n][:, :nh].float().numpy() for n in ("q", "k", "v"))
        t0 = time.perf_counter()
        ro, rl = orc.attention(qn, kn, vn, w.scale, 0, 0, None, threads=threads)
        return ro, rl, time.perf_counter() - t0

    _, _, dt1 = run(1)
    nh = int(min(w.H, max(1, seconds / max(dt1, 1e-3))))
    ro, rl, dt = run(nh)
    alg = 2 * w.B * nh * w.Nk * w.d * 2 + 2 * w.B * nh * w.d * 2 + w.B * nh * 4
    got = o_gpu[:, :nh].float().cpu().numpy()
    got_l = lse_gpu[:, :nh].cpu().double().numpy()
    return {"value": round(alg / dt / 1e9, 3), "unit": "GB/s", "cores": threads,
            "kind": "oracle", "seconds": round(dt, 2),
            "sample": "heads 0..%d of %d (all %d keys each) of the decode workload"
                      % (nh - 1, w.H, w.Nk),
            "max_abs_err_gpu_vs_oracle": float(np.abs(got - ro).max()),
            "max_abs_lse_err_gpu_vs_oracle": float(np.abs(got_l - rl).max())}


def cpu_baseline_backward(w, x, do, dq, dk, dv):
    """The FP64 backward oracle (numpy) on the first head of the workload
    (every query and key of it), in the backward metric's unit, with its
    normwise agreement with the GPU gradients of that head."""
    from oracle import backward as OB
    one = [x[n][:1, :1].float().numpy() for n in ("q", "k", "v")]
    t0 = time.perf_counter()
    rq, rk, rv = OB.attention_backward(*one, do[:1, :1].float().cpu().numpy(), w.scale,
                                       w.mask_kind, w.window)
    dt = time.perf_counter() - t0
    fl = 2.5 * 4.0 * w.d * w.Nq * w.Nk        # one head, no mask
    errs = {}
    for name, got, ref in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        g = got[:1, :1].float().cpu().numpy()
        errs["normwise_err_" + name] = float(np.abs(g - ref).max() / np.abs(ref).max())
    try:
        import threadpoolctl
        cores = max(p.get("num_threads", 1) for p in threadpoolctl.threadpool_info())
    except Exception:   # noqa: BLE001
        cores = len(os.sched_getaffinity(0))
    return dict({"value": round(fl / dt / 1e12, 6), "unit": "TFLOP/s", "cores": cores,
                 "kind": "oracle", "seconds": round(dt, 2),
                 "sample": "head 0 of %d (all %d queries and keys) of the %s backward"
                           % (w.H, w.Nq, w.name)}, **errs)


def cpu_baseline_softmax(x, y, lse, seconds):
    """The FP64 row-softmax oracle on the first rows of the workload (as many
    as fit in about `seconds`), in GB/s of the rows' algorithmic bytes, with
    its agreement with the GPU rows."""
    import oracle
    orc = oracle.Oracle()
    threads = oracle.default_threads()
    n = x.shape[1]

    def run(r):
        xs = x[:r].float().cpu().numpy()
        t0 = time.perf_counter()
        ry, rl = orc.softmax_rows(xs, threads=threads)
        return ry, rl, time.perf_counter() - t0

    _, _, dt1 = run(16)
    r = int(min(x.shape[0], max(16, 16 * seconds / max(dt1, 1e-3))))
    ry, rl, dt = run(r)
    alg = r * (2 * n * x.element_size() + 4)
    return {"value": round(alg / dt / 1e9, 3), "unit": "GB/s", "cores": threads, "kind": "oracle",
            "seconds": round(dt, 2),
            "sample": "rows 0..%d of %d (all %d values each)" % (r - 1, x.shape[0], n),
            "max_abs_err_gpu_vs_oracle": float(np.abs(y[:r].cpu().numpy() - ry).max()),
            "max_abs_lse_err_gpu_vs_oracle": float(np.abs(lse[:r].cpu().numpy() - rl).max())}


def run_reference(args, rank, world):
    """The oracle as the reference arm: each of the --steps steps a bounded
    sample of rows, sized so that all steps together take about
    --ref-seconds of CPU work (at most --ref-seconds-per-step each)."""
    w = W.PREFILL
    x = W.generate(w)
    _, _, _, dt0, _ = oracle_sample(w, x, 32, seed=1)
    per_step = min(args.ref_seconds_per_step, args.ref_seconds / max(args.steps, 1))
    n = int(max(8, 32 * per_step / max(dt0, 1e-3)))
    for s in range(args.warmup):
        oracle_sample(w, x, min(n, 64), seed=100 + s)
    total = 0.0
    threads = 1
    for s in range(args.steps):
        _, _, _, dt, threads = oracle_sample(w, x, n, seed=200 + s)
        total += dt
    fl = 4.0 * w.d * w.Nk * n
    value = fl * args.steps / total / 1e12
    return {"metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(total / args.steps * 1e3, 2), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": dict(w.describe(), parallelism="host cores"), "impl": "reference",
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": threads,
                             "kind": "oracle",
                             "sample": "%d random query rows per step (all %d keys each)" % (n, w.Nk)},
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-seconds-per-step", type=float, default=6.0)
    ap.add_argument("--ref-seconds", type=float, default=60.0,
                    help="CPU seconds the reference arm's timed steps take in all")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-chunks", type=int, default=4, help="head groups of the e2e pipeline")
    ap.add_argument("--e2e-slots", type=int, default=3, help="device buffer sets of the e2e pipeline")
    # profiling helpers: run one section, or a reduced size of it
    ap.add_argument("--no-naive", action="store_true",
                    help="skip the naive (score matrix in HBM) attention context measurement")
    ap.add_argument("--only", choices=["all", "prefill", "causal", "masked", "fp8", "backward",
                                       "decode", "softmax"], default="all")
    ap.add_argument("--heads", type=int, default=0, help="override H of the prefill workload")
    ap.add_argument("--decode-nk", type=int, default=0, help="override Nk of the decode workload")
    ap.add_argument("--batch", type=int, default=0,
                    help="override B of the causal and masked workloads")
    ap.add_argument("--softmax-rows", type=int, default=0,
                    help="override the row count of the softmax workload")
    ap.add_argument("--lib", default=None,
                    help="another build of libattn.so for the forward, E4M3 and backward sections (one "
                         "made by python -m online_softmax_02_gb300.build -D ... --out PATH)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(run_reference(args, rank, world)))
        return
    dist_on = world > 1
    if dist_on:
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        torch.distributed.init_process_group("nccl")
    try:
        res = run_ours(args, rank, world, dist_on)
        if rank == 0:
            print(json.dumps(res))
    finally:
        if dist_on:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
