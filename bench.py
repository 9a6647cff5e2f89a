"""Benchmark of the fused SDPA forward on GB300 (one JSON line on stdout).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl {gb300,reference}]

A step is one sdpa_forward call (the whole hot path) on the diffusion-
transformer self-attention workload of MLX PR #964 (B=2, H=38, Lq=Lk=4250,
D=64, fp16, scale 1/8, no mask; seeded N(0,1) inputs).  The value is the
algorithmic attention throughput, 4*D FLOPs per visible (query, key) pair,
over the K timed steps, timed with CUDA events on the launching stream.  The
inputs rotate over three copies (372 MB > 2 x L2) so that no step starts
with its inputs in L2.  With N > 1 (torchrun) every rank runs the same
workload on its own GPU (replicas; weak scaling) and the slowest rank's time
counts.

Besides the headline line the JSON carries: `e2e` (the same metric through
the C ABI with host buffers: pinned host->device copy of q, k, v and
device->host copy of o and lse inside the timed region), `roofline` of the
prefill kernel against the measured peak, `clocks` sampled during the timed
region, `cpu_baseline` (the float64 oracle on this host's cores over a
bounded sample of the same workload) and `secondary` measurements of the
other workloads (causal GQA prefill, fp32 prefill, both decode workloads).

`--impl reference` times the float64 CPU oracle as it stands (there is no
reference implementation to install: the pages carry no code for this path)
on the same workload, metric and unit.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "SDPA TFLOP/s (prefill) & KV-read GB/s (decode), % of GB300 roofline, 1 GPU"
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_BYTES = 129 * 1024 * 1024


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return PEAKS_FALLBACK, "fallback"


def kernel_source_hash(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "scaled_dot_product_fwd_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profile_traffic(name, files, launch_units=None):
    """DRAM bytes per launch from a committed ncu summary, or None when the
    summary is missing or the kernel source changed since it was taken."""
    p = os.path.join(ROOT, "profiles", name + ".json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    if d.get("source_hash") != kernel_source_hash(files):
        return None
    return d.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]
        return False

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(dist, secs, device):
    """The slowest rank's time (every rank gets it); `dist` None = one rank."""
    if dist is None:
        return secs
    import torch
    t = torch.tensor([float(secs)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(work_per_step, steps, world, secs, scale):
    """Throughput of the whole job: every rank runs `steps` steps of the same
    work (replicas, weak scaling); `secs` is the slowest rank's time."""
    return work_per_step * steps * world / secs / scale


# ------------------------------------------------------------------ GPU arm
def gpu_inputs(torch, w, copies, device):
    from scaled_dot_product_fwd_gb300 import workloads as W
    base = W.make_inputs(w)
    sets = []
    for c in range(copies):
        sets.append({k: (None if t is None else t.to(device)) for k, t in base.items()})
    return base, sets


def time_device(torch, fn, nsets, steps, warmup, stream, windows=None):
    """fn(i) launches step i (input set i % nsets); seconds of `steps` calls.

    With `windows` (a list), events recorded between groups of steps (up to
    10 groups) append each group's milliseconds per step to it; the total
    stays the time of exactly `steps` back-to-back calls."""
    for i in range(warmup):
        fn(i % nsets)
    torch.cuda.synchronize()
    nwin = min(10, steps) if windows is not None else 1
    bounds = [steps * g // nwin for g in range(nwin + 1)]
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(nwin + 1)]
    evs[0].record(stream)
    for g in range(nwin):
        for i in range(bounds[g], bounds[g + 1]):
            fn(i % nsets)
        evs[g + 1].record(stream)
    torch.cuda.synchronize()
    if windows is not None:
        for g in range(nwin):
            n = bounds[g + 1] - bounds[g]
            if n > 0:
                windows.append(evs[g].elapsed_time(evs[g + 1]) / n)
    return evs[0].elapsed_time(evs[-1]) / 1e3  # seconds


def run_workload(torch, S, w, steps, warmup, device, stream, copies=None, windows=None):
    """Device-timed seconds for `steps` calls on rotating input copies."""
    es = 4 if w.dtype == "float32" else 2
    per = (w.B * w.Hq * w.Lq * w.D + 2 * w.B * w.Hkv * w.Lk * w.D) * es
    if copies is None:
        copies = min(64, max(1, -(-2 * L2_BYTES // max(per, 1))))
    _, sets = gpu_inputs(torch, w, copies, device)
    Bq, Hq, Lq, D = sets[0]["q"].shape
    outs = [torch.empty_like(s["q"]) for s in sets]
    lses = [torch.empty((Bq, Hq, Lq), dtype=torch.float32, device=device) for s in sets]

    def fn(i):
        s = sets[i]
        S.sdpa_forward(s["q"], s["k"], s["v"], scale=w.scale, causal=w.causal,
                       sinks=s["sinks"], out=outs[i], lse=lses[i])

    secs = time_device(torch, fn, len(sets), steps, warmup, stream, windows)
    launches = S.sdpa_last_launch_count()  # kernels per call, from the library
    if S.sdpa_device_status() != 0:
        raise RuntimeError("device status set during %s" % w.name)
    return secs, copies, per, launches


def run_workload_graph(torch, S, w, calls, reps, device, copies=None):
    """Device-timed seconds per call for `calls` back-to-back calls captured in
    one CUDA graph on rotating input copies (no host launch overhead between
    calls), replayed `reps` times after warm-up."""
    es = 4 if w.dtype == "float32" else 2
    per = (w.B * w.Hq * w.Lq * w.D + 2 * w.B * w.Hkv * w.Lk * w.D) * es
    if copies is None:
        copies = min(64, max(1, -(-2 * L2_BYTES // max(per, 1))))
    _, sets = gpu_inputs(torch, w, copies, device)
    Bq, Hq, Lq, D = sets[0]["q"].shape
    outs = [torch.empty_like(s["q"]) for s in sets]
    lses = [torch.empty((Bq, Hq, Lq), dtype=torch.float32, device=device) for s in sets]

    def fn(i):
        s = sets[i % len(sets)]
        S.sdpa_forward(s["q"], s["k"], s["v"], scale=w.scale, causal=w.causal,
                       sinks=s["sinks"], out=outs[i % len(sets)], lse=lses[i % len(sets)])

    for i in range(max(3, len(sets))):  # warm-up outside the capture (workspace, attributes)
        fn(i)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream(device)
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            for i in range(calls):
                fn(i)
    torch.cuda.synchronize()
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    if S.sdpa_device_status() != 0:
        raise RuntimeError("device status set during %s" % w.name)
    return e0.elapsed_time(e1) / 1e3 / (reps * calls), copies


def run_e2e(torch, S, w, steps, warmup, device, stream):
    """Same metric with host buffers, through the public host-buffer call
    (sdpa_forward_host): every step copies q, k, v from pinned host memory to
    the GPU and o, lse back, overlapped piece by piece with the kernels; the
    CUDA events on the launching stream bracket all of it."""
    from scaled_dot_product_fwd_gb300 import workloads as W
    host = W.make_inputs(w)
    hq, hk, hv = (host[k].pin_memory() for k in ("q", "k", "v"))
    hs = host["sinks"].to(device) if host["sinks"] is not None else None
    B, Hq, Lq, D = hq.shape
    ho = torch.empty_like(hq).pin_memory()
    hl = torch.empty((B, Hq, Lq), dtype=torch.float32).pin_memory()
    pieces = 4 if w.Lq > 1 else 1

    def step(_):
        S.sdpa_forward_host(hq, hk, hv, scale=w.scale, causal=w.causal, sinks=hs, out=ho,
                            lse=hl, chunks=pieces, device=device)

    secs = time_device(torch, step, 1, steps, warmup, stream)
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv))
    d2h = ho.numel() * ho.element_size() + hl.numel() * hl.element_size()
    return secs, h2d, d2h


def work_per_row(w, total_rows):
    """Work of one query row in the workload's metric: FLOPs (prefill,
    TFLOP/s) or its share of the K/V bytes read once (decode, GB/s)."""
    if w.Lq == 1:
        return w.kv_bytes() / total_rows, 1e9, "GB/s"
    return w.flops() / total_rows, 1e12, "TFLOP/s"


def cpu_model():
    """The host CPU's model name (x86 /proc/cpuinfo 'model name', or the Arm
    implementer/part fields), else the platform's processor string."""
    try:
        with open("/proc/cpuinfo") as f:
            info = f.read()
        for key in ("model name", "Model"):
            for ln in info.splitlines():
                if ln.split(":")[0].strip() == key:
                    return ln.split(":", 1)[1].strip()
        impl = [ln.split(":", 1)[1].strip() for ln in info.splitlines()
                if ln.startswith("CPU implementer")]
        part = [ln.split(":", 1)[1].strip() for ln in info.splitlines()
                if ln.startswith("CPU part")]
        if impl and part:
            return "Arm implementer %s part %s" % (impl[0], part[0])
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


def cpu_baseline(w, target_s=12.0):
    """The float64 oracle on this host's cores over a bounded row sample,
    plus one thread on a smaller sample (rows per second per core)."""
    import numpy as np

    from oracle import oracle as orc
    from scaled_dot_product_fwd_gb300 import workloads as W
    inp = W.make_inputs(w)
    f = W.as_float64
    q, k, v = f(inp["q"]), f(inp["k"]), f(inp["v"])
    total = w.B * w.Hq * w.Lq
    rng = np.random.default_rng(3)
    work_row, scale, unit = work_per_row(w, total)
    n, done, elapsed = 256, 0, 0.0
    while elapsed < target_s and n <= total:
        rows = rng.integers(0, total, size=n)
        t0 = time.perf_counter()
        orc.sdpa(q, k, v, w.scale, w.causal, rows=rows)
        dt = time.perf_counter() - t0
        done += n
        elapsed += dt
        n = min(total, int(n * max(2.0, 1.5 * (target_s - elapsed) / max(dt, 1e-3))))
    rate = done * work_row / elapsed
    cores = orc.num_threads()
    # one thread, about 2 s
    orc.set_num_threads(1)
    try:
        rows1 = max(8, min(total, int(2.0 * done / elapsed / max(cores, 1))))
        t0 = time.perf_counter()
        orc.sdpa(q, k, v, w.scale, w.causal, rows=rng.integers(0, total, size=rows1))
        t1 = time.perf_counter() - t0
    finally:
        orc.set_num_threads(cores)
    return {"value": rate / scale, "unit": unit, "cores": cores, "kind": "oracle",
            "sample": "%d random query rows of %s (all keys each), %.1f s" % (done, w.name, elapsed),
            "cpu_model": cpu_model(),
            "single_thread": {"rows_per_s": round(rows1 / t1, 2),
                              "value": rows1 * work_row / t1 / scale, "unit": unit,
                              "sample": "%d random rows, %.1f s" % (rows1, t1)},
            "timer": "time.perf_counter around the oracle's C call"}


def secondary(torch, S, device, stream, peaks):
    """Other workloads, device-timed (for context; not the headline)."""
    from scaled_dot_product_fwd_gb300 import workloads as W
    out = {}
    for w, steps in ((W.CAUSAL_GQA, 100), (W.DIT_F32, 20), (W.PREFILL_D512, 20)):
        secs, copies, _, _ = run_workload(torch, S, w, steps, 3, device, stream)
        t = w.flops() * steps / secs / 1e12
        out[w.name] = {"value": round(t, 2), "unit": "TFLOP/s", "ms_per_call": secs / steps * 1e3,
                       "frac_of_bf16_peak": round(t / peaks["bf16_tflops"], 4)}
    # microsecond-long calls are timed as a CUDA graph of 20 calls
    per_call, copies = run_workload_graph(torch, S, W.TINY, 20, 25, device, copies=4)
    out[W.TINY.name] = {"value": round(W.TINY.flops() / per_call / 1e12, 3), "unit": "TFLOP/s",
                        "us_per_call": round(per_call * 1e6, 2), "input_copies": copies,
                        "timing": "CUDA graph of 20 calls, replayed"}
    for w, reps in ((W.DECODE_LONG, 10), (W.DECODE_D512[(1, "bfloat16", False)], 25),
                    (W.DECODE_D512[(2, "bfloat16", False)], 25),
                    (W.DECODE_D512[(1, "float16", True)], 25),
                    (W.DECODE_D512[(1, "float32", False)], 25)):
        per_call, copies = run_workload_graph(torch, S, w, 20, reps, device)
        g = w.kv_bytes() / per_call / 1e9
        out[w.name] = {"value": round(g, 1), "unit": "GB/s", "us_per_call": round(per_call * 1e6, 2),
                       "frac_of_hbm": round(g / peaks["hbm_gbs"], 4),
                       "input_copies": copies, "timing": "CUDA graph of 20 calls, replayed"}
    out["decode_kvcache_b8_cap32768_d128_bf16_ragged"] = run_kvcache_decode(torch, S, device,
                                                                             peaks)
    out.update(run_layout_variants(torch, S, device, peaks))
    out.update(run_backward(torch, S, device, peaks))
    return out


def run_backward(torch, S, device, peaks, names=None):
    """Backward pass (sdpa_backward: pre, main and post kernels; fp32: pre,
    dK/dV and dQ kernels) on the DiT fp16, causal GQA bf16 and DiT fp32
    shapes; TFLOP/s counts 2.5 x the forward's
    algorithmic FLOPs (S recomputed, dP, dV, dK, dQ: five products of the
    forward's two).  Synthetic N(0, 1) q, k, v, dO drawn on the device; o and
    lse from the forward."""
    from scaled_dot_product_fwd_gb300 import workloads as W
    g = torch.Generator(device=device).manual_seed(1)
    res = {}
    for w in (W.DIT_F16, W.CAUSAL_GQA, W.DIT_F32):
        if names and w.name not in names:
            continue
        dt = {"float16": torch.float16, "bfloat16": torch.bfloat16}.get(w.dtype, torch.float32)
        q = torch.randn(w.B, w.Hq, w.Lq, w.D, device=device, dtype=dt, generator=g)
        k = torch.randn(w.B, w.Hkv, w.Lk, w.D, device=device, dtype=dt, generator=g)
        v = torch.randn(w.B, w.Hkv, w.Lk, w.D, device=device, dtype=dt, generator=g)
        o, lse = S.sdpa_forward(q, k, v, scale=w.scale, causal=w.causal)
        d_o = torch.randn(o.shape, device=device, dtype=dt, generator=g)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)

        def call():
            S.sdpa_backward(q, k, v, o, lse, d_o, scale=w.scale, causal=w.causal, dq=dq, dk=dk,
                            dv=dv)

        for _ in range(3):
            call()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n = 10
        e0.record()
        for _ in range(n):
            call()
        e1.record()
        torch.cuda.synchronize()
        if S.sdpa_device_status() != 0:
            raise RuntimeError("device status set during the backward")
        sec = e0.elapsed_time(e1) / 1e3 / n
        t = 2.5 * w.flops() / sec / 1e12
        res[w.name + "_backward"] = {
            "value": round(t, 1), "unit": "TFLOP/s", "ms_per_call": round(sec * 1e3, 4),
            "frac_of_bf16_peak": round(t / peaks["bf16_tflops"], 4),
            "kernels_per_call": S.sdpa_last_launch_count()}
    return res


def run_layout_variants(torch, S, device, peaks):
    """The DiT prefill and the long decode on other input forms: [B, L, H, D]
    tensors seen through a transpose (strided q, k, v, o), a boolean key mask
    and an additive key mask.  Synthetic N(0, 1) data drawn on the device; prefill inputs rotate
    over 3 copies (> 2 x L2), the decode K/V (1 GiB) exceeds L2."""
    from scaled_dot_product_fwd_gb300 import workloads as W
    g = torch.Generator(device=device).manual_seed(0)
    res = {}

    def bshd(B, H, L, D, dt):
        return torch.randn(B, L, H, D, device=device, dtype=dt, generator=g).transpose(1, 2)

    def time_calls(calls, steps):
        for i in range(3):
            calls[i % len(calls)]()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for i in range(steps):
            calls[i % len(calls)]()
        e1.record()
        torch.cuda.synchronize()
        if S.sdpa_device_status() != 0:
            raise RuntimeError("device status set during a layout variant")
        return e0.elapsed_time(e1) / 1e3 / steps

    w = W.DIT_F16
    dt = torch.float16
    sets = [tuple(bshd(w.B, h, w.Lq, w.D, dt) for h in (w.Hq, w.Hkv, w.Hkv)) for _ in range(3)]
    outs = [torch.empty_like(st[0]) for st in sets]
    calls = [lambda st=st, o=o: S.sdpa_forward(*st, scale=w.scale, out=o, return_lse=False)
             for st, o in zip(sets, outs)]
    sec = time_calls(calls, 20)
    t = w.flops() / sec / 1e12
    res[w.name + "_bshd"] = {"value": round(t, 1), "unit": "TFLOP/s",
                             "ms_per_call": round(sec * 1e3, 4),
                             "frac_of_bf16_peak": round(t / peaks["bf16_tflops"], 4),
                             "layout": "q, k, v, o stored [B, L, H, D] (SDPA_FLAG_STRIDES)"}
    keep = torch.rand(w.B, 1, 1, w.Lk, device=device, generator=g) >= 0.1
    calls = [lambda st=st, o=o: S.sdpa_forward(*st, scale=w.scale, mask=keep, out=o,
                                               return_lse=False)
             for st, o in zip(sets, outs)]
    sec = time_calls(calls, 20)
    vis = int(keep.sum().item()) * w.Hq * w.Lq  # visible (query, key) pairs
    tv = 4 * w.D * vis / sec / 1e12
    res[w.name + "_bool_key_mask_bshd"] = {
        "value": round(tv, 1), "unit": "TFLOP/s", "ms_per_call": round(sec * 1e3, 4),
        "frac_of_bf16_peak": round(tv / peaks["bf16_tflops"], 4),
        "flops": "4 D per visible (query, key) pair (about 90 % of the keys kept)"}
    bias = torch.randn(w.B, 1, 1, w.Lk, device=device, generator=g).to(dt)
    hide = torch.rand(w.B, 1, 1, w.Lk, device=device, generator=g) < 0.1
    bias[hide] = float("-inf")
    calls = [lambda st=st, o=o: S.sdpa_forward(*st, scale=w.scale, mask=bias, out=o,
                                               return_lse=False)
             for st, o in zip(sets, outs)]
    sec = time_calls(calls, 20)
    vis = int((~hide).sum().item()) * w.Hq * w.Lq
    tv = 4 * w.D * vis / sec / 1e12
    res[w.name + "_additive_key_mask_bshd"] = {
        "value": round(tv, 1), "unit": "TFLOP/s", "ms_per_call": round(sec * 1e3, 4),
        "frac_of_bf16_peak": round(tv / peaks["bf16_tflops"], 4),
        "flops": "4 D per visible (query, key) pair (N(0, 1) bias, about 10 % -inf)"}
    del sets, outs, calls
    wd = W.DECODE_LONG
    q = torch.randn(wd.B, wd.Hq, 1, wd.D, device=device, dtype=torch.bfloat16, generator=g)
    k = bshd(wd.B, wd.Hkv, wd.Lk, wd.D, torch.bfloat16)
    v = bshd(wd.B, wd.Hkv, wd.Lk, wd.D, torch.bfloat16)
    o = torch.empty_like(q)
    gr = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream(device)
    S.sdpa_forward(q, k, v, scale=wd.scale, out=o, return_lse=False)
    torch.cuda.synchronize()
    with torch.cuda.stream(side):
        with torch.cuda.graph(gr, stream=side):
            for _ in range(20):
                S.sdpa_forward(q, k, v, scale=wd.scale, out=o, return_lse=False)
    torch.cuda.synchronize()
    sec = time_calls([gr.replay], 10) / 20
    gb = wd.kv_bytes() / sec / 1e9
    res[wd.name + "_kv_bshd"] = {
        "value": round(gb, 1), "unit": "GB/s", "us_per_call": round(sec * 1e6, 2),
        "frac_of_hbm": round(gb / peaks["hbm_gbs"], 4),
        "layout": "k, v stored [B, L, Hkv, D]: one bulk copy per key row",
        "timing": "CUDA graph of 20 calls, replayed"}
    return res


def run_kvcache_decode(torch, S, device, peaks):
    """Decode against a fixed-capacity KV cache with ragged per-batch lengths
    (B8 Hq32 Hkv8 D128 bf16, capacity 32768, lengths 32768 down to 4096):
    GB/s of the K/V rows the lengths cover, CUDA graph of 20 calls."""
    import numpy as np
    B, Hq, Hkv, D, cap = 8, 32, 8, 128, 32768
    lens = [32768, 28672, 24576, 20480, 16384, 12288, 8192, 4096]
    rng = np.random.default_rng(0)
    q = torch.from_numpy(rng.standard_normal((B, Hq, 1, D), dtype=np.float32)).to(torch.bfloat16)
    kc = torch.from_numpy(rng.standard_normal((B, Hkv, cap, D), dtype=np.float32)).to(torch.bfloat16)
    vc = torch.from_numpy(rng.standard_normal((B, Hkv, cap, D), dtype=np.float32)).to(torch.bfloat16)
    q, kc, vc = q.to(device), kc.to(device), vc.to(device)
    tk = torch.tensor(lens, dtype=torch.int32, device=device)
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, 1), dtype=torch.float32, device=device)

    def call():
        S.sdpa_forward(q, kc, vc, scale=D ** -0.5, kv_len=cap, seq_lens_kv=tk, out=o, lse=lse)

    for _ in range(3):
        call()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream(device)
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            for _ in range(20):
                call()
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(10):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    if S.sdpa_device_status() != 0:
        raise RuntimeError("device status set during the KV-cache decode")
    per_call = e0.elapsed_time(e1) / 1e3 / 200
    used = sum(lens) * Hkv * D * 2 * 2
    gbs = used / per_call / 1e9
    return {"value": round(gbs, 1), "unit": "GB/s", "us_per_call": round(per_call * 1e6, 2),
            "kv_bytes_used": used, "frac_of_hbm": round(gbs / peaks["hbm_gbs"], 4),
            "timing": "CUDA graph of 20 calls, replayed (the K/V rows used, 604 MB, exceed L2)"}


def gb300_arm(args):
    import torch

    import scaled_dot_product_fwd_gb300 as S
    from scaled_dot_product_fwd_gb300 import workloads as W
    world, rank, local = dist_setup(args)
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    import __graft_entry__
    if rank == 0 or world == 1:
        __graft_entry__.build()
    if dist is not None:
        dist.barrier()
    S.load_library()
    peaks, peak_kind = load_peaks()
    w = W.NAMED[args.workload]
    stream = torch.cuda.current_stream(device)

    # --- timed region: K steps, device time, max over ranks
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    windows = []
    with ClockSampler(local) as clk:
        secs, copies, per, per_call_launches = run_workload(torch, S, w, args.steps, args.warmup,
                                                            device, stream, windows=windows)
    secs = max_over_ranks(dist, secs, device)
    if dist is not None:
        dist.barrier()
    flops = w.flops()
    per_launch = secs / args.steps
    e2e_steps = max(3, args.steps // 10)
    e2e_secs, h2d, d2h = run_e2e(torch, S, w, e2e_steps, args.warmup, device, stream)
    if w.Lq == 1:
        # decode: KV-read GB/s, HBM roofline of the split-KV pass (its launch
        # and the combine's together: one step)
        work, unit, scale = w.kv_bytes(), "GB/s", 1e9
        bound, peak, peak_name = "hbm", peaks["hbm_gbs"], " (HBM copy)"
        sustained = peaks["hbm_gbs"]
        if w.D == 512 and w.dtype != "float32" and w.Hq // w.Hkv * w.Lq <= 16:
            # the tensor-core pass (head_dim 512, fp16/bf16, up to 16 rows per kv head)
            traffic = profile_traffic("decode_tc_" + w.name, ["decode_tc.cu", "ptx.cuh"])
        elif w.D == 128 and w.dtype != "float32" and w.Hq // w.Hkv * w.Lq <= 16:
            # the streaming tensor-core pass at head_dim 128
            traffic = profile_traffic("decode_tc128_" + w.name, ["decode_tc128.cu", "ptx.cuh"])
        else:
            traffic = profile_traffic("decode_split_" + w.name,
                                      ["decode.cuh", "decode_combine.cu", "ptx.cuh"])
    else:
        work, unit, scale = flops, "TFLOP/s", 1e12
        bound, peak, peak_name = "tensor", peaks["bf16_tflops"], " (bf16 dense, burst)"
        sustained = peaks["bf16_tflops_sustained"]
        if w.dtype == "float32" and w.D != 64:  # fp32 FMA tiles
            traffic = profile_traffic("prefill_f32_" + w.name, ["prefill_f32.cu"])
        elif w.D == 512:  # two CTAs per query tile, each half of O
            traffic = profile_traffic("prefill_d512_" + w.name, ["prefill_d512.cu", "ptx.cuh"])
        else:  # tensor-core kernel (fp32 at D = 64 as bf16 hi/lo parts)
            tu = "prefill_tc.cu" if w.dtype == "float32" else "prefill_tc_d%d.cu" % w.D
            traffic = profile_traffic("prefill_tc_" + w.name, ["prefill_tc.cuh", tu, "ptx.cuh"])
    launches = per_call_launches * args.steps
    value = whole_job_rate(work, args.steps, world, secs, scale)
    achieved = work / per_launch / scale
    e2e_secs = max_over_ranks(dist, e2e_secs, device)
    e2e_value = whole_job_rate(work, e2e_steps, world, e2e_secs, scale)
    result = {
        "metric": METRIC, "value": round(value, 3), "unit": unit, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(secs / args.steps * 1e3, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": {"float16": "f16", "bfloat16": "bf16", "float32": "f32"}[w.dtype],
        "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "Lq": w.Lq,
                   "Lk": w.Lk, "D": w.D, "causal": w.causal,
                   "flops_per_step": flops,
                   "l2": "inputs rotate over %d copies (%d MB > 2 x L2)" % (
                       copies, copies * per // 10**6),
                   "parallelism": "replicas" if world > 1 else "single"},
        "gpu_launches": launches,
        "step_ms_spread": {"windows": len(windows),
                           "median": round(statistics.median(windows), 5),
                           "min": round(min(windows), 5), "max": round(max(windows), 5),
                           "note": "ms per step of each of up to 10 consecutive groups of "
                                   "the K timed steps (same run as value)"},
        "roofline": {"bound": bound, "achieved": round(achieved, 2),
                     "peak": peak, "unit": unit,
                     "frac": round(achieved / peak, 4),
                     "traffic": traffic, "peak_source": peak_kind + peak_name,
                     "frac_of_sustained": round(achieved / sustained, 4)},
        "clocks": clk.summary(),
        "e2e": {"value": round(e2e_value, 3), "unit": unit, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "method": "C call sdpa_forward_host (include/sdpa.h) through ctypes: pinned "
                          "host q, k, v in, o, lse out; one cudaMemcpyAsync per piece and "
                          "tensor on the library's copy streams, overlapped with the other "
                          "pieces' kernels"},
    }
    if rank == 0 and not args.no_secondary:
        result["secondary"] = secondary(torch, S, device, stream, peaks)
    if rank == 0 and not args.no_cpu and world == 1:
        result["cpu_baseline"] = cpu_baseline(w)
    if rank == 0:
        print(json.dumps(result), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


def reference_arm(args):
    world, rank, local = dist_setup(args)
    if rank != 0:
        return
    from oracle import oracle as orc
    from scaled_dot_product_fwd_gb300 import workloads as W
    import numpy as np
    orc.build()
    w = W.NAMED[args.workload]
    inp = W.make_inputs(w)
    f = W.as_float64
    q, k, v = f(inp["q"]), f(inp["k"]), f(inp["v"])
    total = w.B * w.Hq * w.Lq
    work_row, scale, unit = work_per_row(w, total)
    rng = np.random.default_rng(5)
    # size one step so that warmup + steps take about a minute
    t0 = time.perf_counter()
    orc.sdpa(q, k, v, w.scale, w.causal, rows=rng.integers(0, total, size=128))
    per_row = (time.perf_counter() - t0) / 128
    rows = int(max(1, min(total, 60.0 / max(args.steps + args.warmup, 1) / per_row)))
    for _ in range(args.warmup):
        orc.sdpa(q, k, v, w.scale, w.causal, rows=rng.integers(0, total, size=rows))
    t0 = time.perf_counter()
    for _ in range(args.steps):
        orc.sdpa(q, k, v, w.scale, w.causal, rows=rng.integers(0, total, size=rows))
    secs = time.perf_counter() - t0
    value = rows * work_row * args.steps / secs / scale
    sample = "%d random query rows of %s per step (all keys each)" % (rows, w.name)
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": unit,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": secs / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "Lq": w.Lq,
                   "Lk": w.Lk, "D": w.D, "causal": w.causal},
        "cpu_baseline": {"value": value, "unit": unit, "cores": orc.num_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--workload", default="dit_b2_h38_l4250_d64_f16")
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--backward-only", action="store_true",
                    help="time only the backward pass workloads and print them (a profiling "
                         "target; not the benchmark line)")
    ap.add_argument("--backward-workloads", default="",
                    help="with --backward-only: comma-separated workload names (default: all)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.backward_only:
        import torch
        import scaled_dot_product_fwd_gb300 as S
        torch.cuda.set_device(0)
        peaks, _ = load_peaks()
        names = [n for n in args.backward_workloads.split(",") if n]
        print(json.dumps(run_backward(torch, S, "cuda", peaks, names)), flush=True)
        return
    if args.impl == "reference":
        reference_arm(args)
    else:
        gb300_arm(args)


if __name__ == "__main__":
    main()
