#!/usr/bin/env python
"""Benchmark of the GB300 attention hot path (one JSON line on rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl gqa|reference]

Default workload: PLaMo-3-shaped local-layer prefill (B=2, T=S=8192, 64 query / 8 KV
heads, d=128, window 2048, RoPE base 1e4).  One step = one pass of the prefill path:
K rotated once (gqa_rope_apply) + the tcgen05 attention kernel with Q rotated on load
(gqa_attn_prefill with k_is_rotated=1) -- exactly the two launches gqa_attn_prefill makes
for pre-RoPE keys.  `value` = effective TFLOP/s (visible (query, key) pairs only,
4 d FLOP each per query head) with inputs resident in HBM, L2 flushed before every timed
step.  `e2e` = the same metric through one gqa_attn_prefill call with host buffers:
pinned Q/K/V copied in and O copied out inside the timed region.

Other workloads (--workload): plamo3_global_prefill (T=32768, YaRN), and
plamo3_decode_batch32 (kv_append + split-KV decode, metric KV GB/s).  On the default run
the other two are also measured and reported under "extra".

Multi-GPU (torchrun): every rank runs its own replica of the workload (the units are
independent sequences/heads, no collective on the data path); value = units of all
ranks / max-over-ranks time ("scaling": "weak").

--impl reference: the fp64 CPU oracle (the only reference this path has) timed on the
host cores on a bounded sample of the same workload, same metric and unit.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = ("prefill effective attention TFLOP/s (window & global); decode KV GB/s, "
          "% roofline")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 256 << 20
_INPUT_CACHE = {}


# ----------------------------------------------------------------------------------------
# environment
# ----------------------------------------------------------------------------------------

def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def code_sha256(path: str) -> str:
    """SHA-256 of a C/CUDA source's code: comments, trailing blanks and empty lines
    removed, so that editing a comment keeps a measurement of the code valid."""
    import re
    with open(path) as f:
        src = f.read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    lines = [ln.rstrip() for ln in src.splitlines()]
    return hashlib.sha256("\n".join(ln for ln in lines if ln).encode()).hexdigest()


def traffic_record(kernel: str, workload: str):
    """DRAM bytes per launch of `kernel` on `workload` from a committed ncu capture
    (profiles/traffic.json), valid only while the kernel source's code is identical to
    the one profiled (code_sha256); None otherwise."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        rec = json.load(f).get(kernel, {}).get(workload)
    if not rec:
        return None
    sha = code_sha256(os.path.join(ROOT, "global_causal_gqa_gb300", "csrc", rec["source"]))
    return rec["bytes_per_launch"] if rec.get("code_sha256") == sha else None


def kernel_name(L) -> str:
    from global_causal_gqa_gb300 import accounting as acc
    return acc.prefill_kernel_name(L.d, L.T, L.S, L.window)


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms while running."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = os.path.join("/tmp", f"gqa_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------------------
# timing helpers
# ----------------------------------------------------------------------------------------

class Timer:
    """Per-step CUDA events on the launching stream; L2 flushed (untimed) before each step."""

    def __init__(self, torch, stream, n_marks: int):
        self.torch = torch
        self.stream = stream
        self.n_marks = n_marks
        self.flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
        self.records = []

    def run(self, steps: int, step_fn, timed: bool = True):
        torch = self.torch
        for _ in range(steps):
            self.flush.fill_(1)
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(self.n_marks)]
            marks = iter(ev)

            def mark():
                next(marks).record(self.stream)

            step_fn(mark)
            if timed:
                self.records.append(ev)

    def durations_ms(self):
        """[steps][segments] durations between consecutive marks."""
        self.torch.cuda.synchronize()
        return [[a.elapsed_time(b) for a, b in zip(ev[:-1], ev[1:])] for ev in self.records]


def load_phase(timer, step, seconds: float = 1.0):
    """Untimed steps for about `seconds` right before the timed region, so the clock
    sampler (one sample per 200 ms) sees the GPU under this load; the reported clocks
    cover this phase and the timed steps."""
    t_end = time.perf_counter() + seconds
    while time.perf_counter() < t_end:
        timer.run(1, step, timed=False)
        timer.torch.cuda.synchronize()


def dist_setup(args):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(world, value: float) -> float:
    """The largest of the ranks' values (the step time every rank reports is the slowest
    rank's); NCCL reduces a device tensor, gloo (CPU runs) a host one."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------------------
# prefill
# ----------------------------------------------------------------------------------------

def prefill_setup(layer):
    import torch
    import global_causal_gqa_gb300 as gqa
    from workloads import prefill_inputs
    x = prefill_inputs(layer)
    st = {"x": x, "q": x.q.cuda(), "k": x.k.cuda(), "v": x.v.cuda()}
    st["o"] = torch.empty_like(st["q"])
    d, r = layer.d, layer.rope
    w = gqa.gqa_rope_inv_freq(d, r.base, r.yarn_factor, r.yarn_L0, r.beta_fast, r.beta_slow,
                              r.rotate_fraction)
    st["table"] = torch.empty(layer.S * d, dtype=torch.float32, device="cuda")
    gqa.gqa_rope_table_build(st["table"], w, d, r.amp, layer.S)
    st["wsb"] = gqa.gqa_prefill_workspace_bytes(layer.B, layer.Hkv, layer.S, d)
    st["ws"] = torch.empty(st["wsb"], dtype=torch.uint8, device="cuda")
    return st


def bench_prefill(name, layers, steps: int, warmup: int, stream, peaks, peak_src, world,
                  with_e2e: bool, clocks_index=None):
    """One step = every layer of the workload in sequence, each = K rotated once
    (gqa_rope_apply) + the attention kernel (gqa_attn_prefill, k_is_rotated=1)."""
    import torch
    import global_causal_gqa_gb300 as gqa
    from global_causal_gqa_gb300 import accounting as acc
    if not isinstance(layers, (list, tuple)):
        layers = [layers]
    sts = [prefill_setup(L) for L in layers]
    flops = sum(acc.prefill_flops(L.B, L.Hq, L.T, L.S, L.d, L.window) for L in layers)
    timer = Timer(torch, stream, 2 * len(layers) + 1)

    def step(mark):
        mark()
        for L, st in zip(layers, sts):
            gqa.gqa_rope_apply(st["k"], st["ws"], L.B, L.Hkv, L.S, L.d, 0, st["table"], L.S,
                               stream)
            mark()
            gqa.gqa_attn_prefill(st["q"], st["ws"], st["v"], st["o"], None, L.B, L.T, L.S,
                                 L.Hq, L.Hkv, L.d, L.window, L.scale, st["table"], L.S, 1,
                                 None, 0, stream)
            mark()

    timer.run(warmup, step, timed=False)
    torch.cuda.synchronize()
    assert gqa.gqa_get_device_status(stream) == 0
    barrier(world)
    torch.cuda.synchronize()
    sampler = ClockSampler(clocks_index) if clocks_index is not None else None
    if sampler:
        sampler.__enter__()
        load_phase(timer, step)
    t0 = time.perf_counter()
    timer.run(steps, step)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    barrier(world)
    if sampler:
        sampler.__exit__(None, None, None)
    st_code = gqa.gqa_get_device_status(stream)
    assert st_code == 0, f"device status {st_code}"
    dur = timer.durations_ms()
    step_ms = statistics.mean(sum(d) for d in dur)
    rope_ms = statistics.mean(sum(d[0::2]) for d in dur)
    kern_ms = statistics.mean(sum(d[1::2]) for d in dur)
    per_layer = [statistics.mean(d[2 * i + 1] for d in dur) for i in range(len(layers))]
    step_ms_max = max_over_ranks(world, step_ms)
    value = world * flops / (step_ms_max * 1e-3) / 1e12
    peak = peaks["bf16_tflops"]
    # roofline of the dominant kernel: the layer with the largest device time
    dom = max(range(len(layers)), key=lambda i: per_layer[i])
    Ld = layers[dom]
    dom_flops = acc.prefill_flops(Ld.B, Ld.Hq, Ld.T, Ld.S, Ld.d, Ld.window)
    achieved = dom_flops / (per_layer[dom] * 1e-3) / 1e12
    dom_wl = name if len(layers) == 1 else f"{name}[layer {dom}]"
    out = {
        "value": value, "unit": "TFLOP/s", "ms_per_step": step_ms_max,
        "kernel_ms": {"rope_k": rope_ms, "prefill": kern_ms},
        "flops_per_step": flops, "wall_s": wall,
        "roofline": {"bound": "tensor", "kernel": kernel_name(Ld), "achieved": achieved,
                     "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                     "peak_source": f"bf16_tflops (burst, {peak_src})",
                     "traffic": traffic_record(kernel_name(Ld), dom_wl)},
        "gpu_launches": 2 * len(layers) * steps,
        "clocks": sampler.summary() if sampler else None,
    }
    if len(layers) > 1:
        out["roofline"]["layer"] = dom
        all_tf = flops / (kern_ms * 1e-3) / 1e12
        out["roofline"]["all_attention_kernels"] = {"achieved": all_tf, "frac": all_tf / peak}
        out["per_layer"] = [
            {"d": L.d, "window": L.window, "kernel": kernel_name(L), "ms": ms,
             "tflops": acc.prefill_flops(L.B, L.Hq, L.T, L.S, L.d, L.window) / (ms * 1e-3) / 1e12}
            for L, ms in zip(layers, per_layer)]
    if with_e2e:
        out["e2e"] = e2e_prefill(layers[0], sts[0], steps, warmup, stream,
                                 acc.prefill_flops(layers[0].B, layers[0].Hq, layers[0].T,
                                                   layers[0].S, layers[0].d, layers[0].window))
        if len(layers) > 1:
            out["e2e"]["note"] = "first layer only"
    return out


def e2e_prefill(L, st, steps, warmup, stream, flops):
    """One step through the public call with host buffers: pinned Q/K/V in, O out.  The
    step is cut into independent chunks (a batch element and one KV head with its query
    group), each one gqa_attn_prefill call on the caller's stream; later chunks' inputs
    copy in on one stream and earlier chunks' outputs copy out on another while a chunk
    computes, as a serving loop would overlap its transfers.  The host inputs are laid out
    chunk after chunk (a chunk's Q heads, K and V side by side, as a serving loop would
    gather a request's tensors), so each chunk comes in with one copy; the device tensors
    have the same layout and each call gets its chunk's pointers.  Measured on the local
    prefill: 246 TFLOP/s with the copies and the whole call in series, 389 / 411 / 414
    with 4 / 8 / 16 chunks and three copies per chunk."""
    import torch
    import global_causal_gqa_gb300 as gqa
    x = st["x"]
    G = L.Hq // L.Hkv
    parts = [(b, g) for b in range(L.B) for g in range(L.Hkv)]
    qn, kn = G * L.T * L.d, L.S * L.d          # elements of a chunk's Q and of its K (= V)
    cn = qn + 2 * kn
    hin = torch.empty(len(parts) * cn, dtype=torch.bfloat16).pin_memory()
    for c, (b, g) in enumerate(parts):
        hin[c * cn: c * cn + qn].copy_(x.q[b, G * g: G * (g + 1)].reshape(-1))
        hin[c * cn + qn: c * cn + qn + kn].copy_(x.k[b, g].reshape(-1))
        hin[c * cn + qn + kn: (c + 1) * cn].copy_(x.v[b, g].reshape(-1))
    din = torch.empty_like(hin, device="cuda")
    oh = torch.empty_like(x.q).pin_memory()
    h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()
    timer = Timer(torch, stream, 2)
    whole = st["o"].clone()   # the device-timed single call's output, same inputs

    def step(mark):
        mark()
        start = torch.cuda.Event()
        start.record(stream)
        h2d.wait_event(start)
        d2h.wait_event(start)
        landed = []
        with torch.cuda.stream(h2d):
            for c in range(len(parts)):
                din[c * cn: (c + 1) * cn].copy_(hin[c * cn: (c + 1) * cn], non_blocking=True)
                e = torch.cuda.Event()
                e.record(h2d)
                landed.append(e)
        for c, ((b, g), e) in enumerate(zip(parts, landed)):
            stream.wait_event(e)
            qd = din[c * cn: c * cn + qn]
            kd = din[c * cn + qn: c * cn + qn + kn]
            vd = din[c * cn + qn + kn: (c + 1) * cn]
            od = st["o"][b, G * g: G * (g + 1)]
            gqa.gqa_attn_prefill(qd, kd, vd, od, None, 1, L.T, L.S, G, 1, L.d, L.window,
                                 L.scale, st["table"], L.S, 0, st["ws"], st["wsb"], stream)
            done = torch.cuda.Event()
            done.record(stream)
            with torch.cuda.stream(d2h):
                d2h.wait_event(done)
                oh[b, G * g: G * (g + 1)].copy_(od, non_blocking=True)
        out = torch.cuda.Event()
        out.record(d2h)
        stream.wait_event(out)
        mark()

    timer.run(max(1, warmup), step, timed=False)
    timer.run(steps, step)
    ms = statistics.mean(a for (a,) in timer.durations_ms())
    if not torch.equal(oh, whole.cpu()):
        raise SystemExit("end-to-end chunked output differs from the single call's")
    nb = lambda t: t.numel() * t.element_size()  # noqa: E731
    return {"value": flops / (ms * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": ms,
            "h2d_bytes_per_step": nb(hin), "d2h_bytes_per_step": nb(oh),
            "pipeline": f"{len(parts)} public calls per step (batch element x KV head), "
                        "one copy in per call (its Q, K and V side by side) and one out, on "
                        "two more streams overlapping the compute"}


# ----------------------------------------------------------------------------------------
# decode
# ----------------------------------------------------------------------------------------

def decode_setup(w):
    import numpy as np
    import torch
    import global_causal_gqa_gb300 as gqa
    from workloads import decode_inputs
    x = decode_inputs(w)
    st = {"x": x, "q": x.q.cuda(), "k_new": x.k_new.cuda(), "v_new": x.v_new.cuda(),
          "kc": [t.cuda() for t in x.k_cache]}
    # a shared K/V layer has one cache per sequence (its descriptors' v is never read)
    st["vc"] = st["kc"] if w.kv_shared else [t.cuda() for t in x.v_cache]
    tables = {}
    for r in set(x.rope):
        n = max(x.cap[i] for i in range(w.nseq) if x.rope[i] == r)
        wf = gqa.gqa_rope_inv_freq(w.d, r.base, r.yarn_factor, r.yarn_L0, r.beta_fast,
                                   r.beta_slow, r.rotate_fraction)
        t = torch.empty(n * w.d, dtype=torch.float32, device="cuda")
        gqa.gqa_rope_table_build(t, wf, w.d, r.amp, n)
        tables[r] = (t, n)
    st["tables"] = tables
    a = gqa.make_kv_descs(st["kc"], st["vc"], [tables[r][0] for r in x.rope], x.cap,
                          x.count_before, x.is_ring, [tables[r][1] for r in x.rope])
    st["descs0"] = torch.from_numpy(a.view(np.uint8).copy()).cuda()
    st["descs"] = st["descs0"].clone()
    st["max_len"] = max(w.global_len_range[1], w.window)
    st["o"] = torch.empty_like(st["q"])
    st["wsb"] = gqa.gqa_decode_workspace_bytes(w.nseq, w.Hq, w.Hkv, w.d, st["max_len"])
    st["ws"] = torch.empty(st["wsb"], dtype=torch.uint8, device="cuda")
    st["retained"] = [min(c + 1, cap) if ring else c + 1
                      for c, cap, ring in zip(x.count_before, x.cap, x.is_ring)]
    if w.kv_shared:
        # one cache per sequence holding Zn = N_1(Z) of the drawn rows (normalised once,
        # untimed); the query and key gains of the layer
        from workloads import norm_gains
        for i, zc in enumerate(st["kc"]):
            gqa.gqa_qk_norm_rope_kv_shared(None, zc, None, zc, None, 1, 0, w.Hkv, x.cap[i], w.d,
                                           0, None, None, 1e-6, None, 0)
        st["q_gamma"] = torch.from_numpy(norm_gains(w.d, w.seed + 1)).float().cuda()
        st["k_gamma"] = torch.from_numpy(norm_gains(w.d, w.seed + 2)).float().cuda()
        st["q_out"] = torch.empty_like(st["q"])
    return st


def decode_step_calls(w, st, stream, mark=None):
    """The step's two calls: append the new token (plain K/V, or the shared projection's
    normalised row plus the normalised query), then the decode attention."""
    import global_causal_gqa_gb300 as gqa
    mark = mark or (lambda: None)
    if w.kv_shared:
        gqa.gqa_kv_shared_append(st["descs"], w.nseq, st["q"], st["k_new"], w.Hq, w.Hkv, w.d,
                                 st["q_gamma"], 1e-6, st["q_out"], None, stream)
        mark()
        gqa.gqa_attn_decode_kv_shared(st["q_out"], st["descs"], w.nseq, w.Hq, w.Hkv, w.d,
                                      w.scale, st["k_gamma"], st["max_len"], st["o"], None,
                                      st["ws"], st["wsb"], stream)
    else:
        gqa.gqa_kv_append(st["descs"], w.nseq, st["k_new"], st["v_new"], w.Hkv, w.d, None,
                          stream)
        mark()
        gqa.gqa_attn_decode(st["q"], st["descs"], w.nseq, w.Hq, w.Hkv, w.d, w.scale,
                            st["max_len"], st["o"], None, st["ws"], st["wsb"], stream)


def bench_decode(w, steps, warmup, stream, peaks, peak_src, world, with_e2e, clocks_index=None):
    import torch
    import global_causal_gqa_gb300 as gqa
    from global_causal_gqa_gb300 import accounting as acc
    st = decode_setup(w)
    kv_bytes = acc.decode_kv_bytes(st["retained"], w.Hkv, w.d, kv_shared=w.kv_shared)
    qo_bytes = 2 * w.nseq * w.Hq * w.d * 2
    timer = Timer(torch, stream, 3)

    def step(mark):
        # every step starts from the same cache state (descriptor counts restored, untimed)
        st["descs"].copy_(st["descs0"], non_blocking=True)
        mark()
        decode_step_calls(w, st, stream, mark)
        mark()

    timer.run(warmup, step, timed=False)
    torch.cuda.synchronize()
    assert gqa.gqa_get_device_status(stream) == 0
    barrier(world)
    sampler = ClockSampler(clocks_index) if clocks_index is not None else None
    if sampler:
        sampler.__enter__()
        load_phase(timer, step)
    timer.run(steps, step)
    torch.cuda.synchronize()
    barrier(world)
    if sampler:
        sampler.__exit__(None, None, None)
    assert gqa.gqa_get_device_status(stream) == 0
    dur = timer.durations_ms()
    step_ms = max_over_ranks(world, statistics.mean(a + b for a, b in dur))
    dec_ms = statistics.mean(b for _, b in dur)
    value = world * kv_bytes / (step_ms * 1e-3) / 1e9
    peak = peaks["hbm_gbs"]
    achieved = (kv_bytes + qo_bytes) / (dec_ms * 1e-3) / 1e9
    out = {
        "value": value, "unit": "GB/s", "ms_per_step": step_ms,
        "kernel_ms": {"kv_append": statistics.mean(a for a, _ in dur), "decode": dec_ms},
        "kv_bytes_per_step": kv_bytes,
        "roofline": {"bound": "hbm", "kernel": "decode_partial_kernel + decode_combine_kernel",
                     "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_source": f"hbm_gbs ({peak_src})",
                     "traffic": traffic_record("decode_partial_kernel", w.name)},
        "gpu_launches": 3 * steps,
        "clocks": sampler.summary() if sampler else None,
    }
    if with_e2e:
        out["e2e"] = e2e_decode(w, st, steps, warmup, stream, kv_bytes)
    return out


def e2e_decode(w, st, steps, warmup, stream, kv_bytes):
    """Host query and new K/V rows in, host output out; the caches stay resident (they are
    the model's state between steps, not a per-step input)."""
    import torch
    import global_causal_gqa_gb300 as gqa
    x = st["x"]
    # host inputs of one step: the query and the new token's rows (K and V, or the shared
    # projection's Z alone)
    ins = [(x.q, st["q"]), (x.k_new, st["k_new"])]
    if not w.kv_shared:
        ins.append((x.v_new, st["v_new"]))
    ins = [(h.pin_memory(), dev) for h, dev in ins]
    oh = torch.empty_like(x.q).pin_memory()
    timer = Timer(torch, stream, 2)

    def step(mark):
        st["descs"].copy_(st["descs0"], non_blocking=True)
        mark()
        for h, dev in ins:
            dev.copy_(h, non_blocking=True)
        decode_step_calls(w, st, stream)
        oh.copy_(st["o"], non_blocking=True)
        mark()

    timer.run(max(1, warmup), step, timed=False)
    timer.run(steps, step)
    ms = statistics.mean(a for (a,) in timer.durations_ms())
    nb = lambda t: t.numel() * t.element_size()  # noqa: E731
    return {"value": kv_bytes / (ms * 1e-3) / 1e9, "unit": "GB/s", "ms_per_step": ms,
            "h2d_bytes_per_step": sum(nb(h) for h, _ in ins), "d2h_bytes_per_step": nb(oh)}


# ----------------------------------------------------------------------------------------
# whole-model decode step (every layer of the hybrid decoder, CUDA graph)
# ----------------------------------------------------------------------------------------

def decode_model_stack(w):
    """The whole-model decode step's layers (7 local ring layers then 1 global linear
    layer per period), with caches and inputs drawn on the device (synthetic N(0,1),
    seeded), as a LayerStack whose descriptors live in one buffer."""
    import torch
    import global_causal_gqa_gb300 as gqa
    from global_causal_gqa_gb300.model_step import Layer, LayerStack
    gen = torch.Generator(device="cuda").manual_seed(w.seed)
    rnd = lambda *shape: torch.randn(*shape, generator=gen, device="cuda").to(torch.bfloat16)  # noqa: E731
    tables = {}
    for is_g, rope, n in ((True, w.rope_global, w.N), (False, w.rope_local, w.W)):
        f = gqa.gqa_rope_inv_freq(w.d, rope.base, rope.yarn_factor, rope.yarn_L0, rope.beta_fast,
                                  rope.beta_slow, rope.rotate_fraction)
        t = torch.empty(n * w.d, dtype=torch.float32, device="cuda")
        gqa.gqa_rope_table_build(t, f, w.d, rope.amp, n)
        tables[is_g] = (t, n)
    layers = []
    for l in range(w.layers):
        is_g = (l % w.period) == w.period - 1
        cap = w.N if is_g else w.W
        tab, tlen = tables[is_g]
        layers.append(Layer(k_cache=rnd(w.nseq, w.Hkv, cap, w.d),
                            v_cache=rnd(w.nseq, w.Hkv, cap, w.d),
                            q=rnd(w.nseq, w.Hq, w.d), k_new=rnd(w.nseq, w.Hkv, w.d),
                            v_new=rnd(w.nseq, w.Hkv, w.d),
                            o=torch.empty(w.nseq, w.Hq, w.d, dtype=torch.bfloat16,
                                          device="cuda"),
                            table=tab, table_len=tlen, is_ring=not is_g,
                            count_before=[w.N - 1] * w.nseq))
    return LayerStack(layers, w.Hq, w.Hkv, w.d, w.scale, max_len=w.N)


def bench_decode_model(w, steps, warmup, stream, peaks, peak_src):
    """One step = kv_append + decode for every layer, captured once in a CUDA graph and
    replayed; every layer's counts are restored by a single copy at the start of each
    replay, so each step appends into the same slots.
    Reported against the pages' byte model: K and V read once per (sequence, KV head),
    4 Hkv d [n_global N + n_local min(N, W)] bytes per sequence."""
    import torch
    import global_causal_gqa_gb300 as gqa
    from global_causal_gqa_gb300 import accounting as acc
    stack = decode_model_stack(w)
    n_g = w.layers // w.period
    n_l = w.layers - n_g
    bytes_step = w.nseq * 2 * 2 * w.Hkv * w.d * (n_g * w.N + n_l * min(w.N, w.W))
    assert bytes_step == w.nseq * acc.kv_bytes_per_token(w.layers, w.Hkv, w.d, w.N, w.W)
    body = stack.step

    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")

    def timed(run, n):
        out = []
        for _ in range(n):
            flush.fill_(1)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            run()
            e1.record()
            out.append((e0, e1))
        torch.cuda.synchronize()
        return statistics.mean(a.elapsed_time(b) for a, b in out)

    for _ in range(warmup):
        body()
    torch.cuda.synchronize()
    assert gqa.gqa_get_device_status() == 0
    eager_ms = timed(body, steps)
    graph = stack.capture()
    for _ in range(warmup):
        graph.replay()
    torch.cuda.synchronize()
    graph_ms = timed(graph.replay, steps)
    assert gqa.gqa_get_device_status() == 0
    peak = peaks["hbm_gbs"]
    predicted_ms = bytes_step / (peak * 1e9) * 1e3
    return {
        "value": bytes_step / (graph_ms * 1e-3) / 1e9, "unit": "GB/s", "ms_per_step": graph_ms,
        "eager_ms_per_step": eager_ms, "kv_bytes_per_step": bytes_step,
        "byte_model": {"bytes_per_token": bytes_step // w.nseq,
                       "predicted_ms_at_peak": predicted_ms,
                       "measured_over_predicted": graph_ms / predicted_ms},
        "roofline": {"bound": "hbm", "kernel": "64 x (kv_append_kernel + decode_partial_kernel "
                     "+ decode_combine_kernel), one CUDA graph",
                     "achieved": bytes_step / (graph_ms * 1e-3) / 1e9, "peak": peak,
                     "unit": "GB/s", "frac": (bytes_step / (graph_ms * 1e-3) / 1e9) / peak,
                     "peak_source": f"hbm_gbs ({peak_src})", "traffic": None},
        "gpu_launches": 3 * w.layers * steps,
    }


# ----------------------------------------------------------------------------------------
# CPU oracle (cpu_baseline leg and --impl reference)
# ----------------------------------------------------------------------------------------

def oracle_prefill_sample(layer, target_s: float, seed: int = 0):
    """Times the fp64 oracle on a seeded sample of query rows of `layer`, sized to take
    about target_s seconds.  Returns (TFLOP/s counted like the GPU metric, info)."""
    import numpy as np
    import oracle
    from global_causal_gqa_gb300 import accounting as acc
    from workloads import prefill_inputs
    orc = oracle.default()
    key = ("prefill", layer)
    if key not in _INPUT_CACHE:
        _INPUT_CACHE[key] = prefill_inputs(layer)
    x = _INPUT_CACHE[key]
    r = layer.rope
    w = orc.inv_freq(layer.d, r.base, r.yarn_factor, r.yarn_L0, r.beta_fast, r.beta_slow,
                     r.rotate_fraction)
    rng = np.random.default_rng(seed)

    def run(n):
        # rows of one (batch, KV head) group so the per-group key rotation is shared
        G = layer.Hq // layer.Hkv
        b, g = int(rng.integers(layer.B)), int(rng.integers(layer.Hkv))
        rows = np.stack([np.full(n, b), g * G + rng.integers(0, G, n),
                         rng.integers(0, layer.T, n)], 1).astype(np.int32)
        t0 = time.perf_counter()
        orc.attention(x.q, x.k, x.v, window=layer.window, scale=layer.scale, w=w,
                      amp=r.amp, rows=rows)
        dt = time.perf_counter() - t0
        off = layer.S - layer.T
        pairs = sum(min(off + int(t) + 1, layer.window) if layer.window > 0 else off + int(t) + 1
                    for t in rows[:, 2])
        return dt, 4 * layer.d * pairs, n

    # each call rotates its group's keys once, then pays per row: fit both costs from two
    # calls, then run batches of at most 100k rows until about target_s has been spent
    dt1, _, n1 = run(64)
    dt2, _, n2 = run(1024)
    per_row = max((dt2 - dt1) / (n2 - n1), 1e-7)
    batch = int(min(100000, max(1024, (target_s - dt1) / per_row)))
    dt = fl = n = 0
    while dt < 0.8 * target_s:
        d_i, f_i, n_i = run(batch)
        dt, fl, n = dt + d_i, fl + f_i, n + n_i
    return fl / dt / 1e12, {"rows": n, "seconds": dt}


def oracle_decode_sample(w, target_s: float, seed: int = 0):
    """Times the oracle decode step on a subset of the sequences; GB/s of K/V covered."""
    import oracle
    from global_causal_gqa_gb300 import accounting as acc
    from workloads import decode_inputs
    orc = oracle.default()
    key = ("decode", w.name)
    if key not in _INPUT_CACHE:
        _INPUT_CACHE[key] = decode_inputs(w)
    x = _INPUT_CACHE[key]
    ws = [orc.inv_freq(w.d, r.base, r.yarn_factor, r.yarn_L0, r.beta_fast, r.beta_slow,
                       r.rotate_fraction) for r in x.rope]
    order = list(range(w.nseq - 1, -1, -1))   # rings first, then global sequences

    if w.kv_shared:
        from workloads import norm_gains
        gq, gk = norm_gains(w.d, w.seed + 1), norm_gains(w.d, w.seed + 2)

    def run(idx):
        sub = lambda a: [a[i] for i in idx]  # noqa: E731
        t0 = time.perf_counter()
        if w.kv_shared:
            orc.decode_step_kv_shared(x.q[idx], x.k_new[idx], sub(x.k_cache), sub(x.cap),
                                      sub(x.count_before), sub(x.is_ring), sub(ws),
                                      [r.amp for r in sub(x.rope)], q_gamma=gq, k_gamma=gk,
                                      eps=1e-6, scale=w.scale)
        else:
            orc.decode_step(x.q[idx], x.k_new[idx], x.v_new[idx], sub(x.k_cache),
                            sub(x.v_cache), sub(x.cap), sub(x.count_before), sub(x.is_ring),
                            sub(ws), [r.amp for r in sub(x.rope)], w.scale)
        dt = time.perf_counter() - t0
        ret = [min(x.count_before[i] + 1, x.cap[i]) if x.is_ring[i] else x.count_before[i] + 1
               for i in idx]
        return dt, acc.decode_kv_bytes(ret, w.Hkv, w.d, kv_shared=w.kv_shared)

    dt, b = run(order[:1])
    k = 1
    while k < len(order) and dt < target_s / 2:
        k = min(len(order), k * 2)
        dt, b = run(order[:k])
    return b / dt / 1e9, {"sequences": k, "seconds": dt}


def cpu_baseline(workload_name, layer_or_w, is_decode, target_s=12.0):
    cores = os.cpu_count()
    if is_decode:
        v, info = oracle_decode_sample(layer_or_w, target_s)
        return {"value": v, "unit": "GB/s", "cores": cores, "kind": "oracle",
                "sample": f"{info['sequences']} of {layer_or_w.nseq} sequences of "
                          f"{workload_name} (fp64, {info['seconds']:.1f} s)"}
    v, info = oracle_prefill_sample(layer_or_w, target_s)
    return {"value": v, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"{info['rows']} random query rows of {workload_name} "
                      f"(fp64, {info['seconds']:.1f} s)"}


def run_reference(args, wl, world, rank):
    if rank != 0:
        return
    from workloads import DecodeWorkload
    is_decode = isinstance(wl, DecodeWorkload)
    target = wl if is_decode else wl.layers[0]
    per_step = float(os.environ.get("GQA_REF_STEP_SECONDS", "3"))
    vals, secs = [], []
    for i in range(args.warmup + args.steps):
        if is_decode:
            v, info = oracle_decode_sample(target, per_step, seed=i)
        else:
            v, info = oracle_prefill_sample(target, per_step, seed=i)
        if i >= args.warmup:
            vals.append(v)
            secs.append(info["seconds"])
    value = statistics.mean(vals)
    unit = "GB/s" if is_decode else "TFLOP/s"
    sample = (f"each step: {info.get('sequences', info.get('rows'))} "
              f"{'sequences' if is_decode else 'random query rows'} of {wl.name}, fp64")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": unit,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * statistics.mean(secs), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {**config_of(wl), "parallelism": f"host cores x{os.cpu_count()}"},
            "cpu_baseline": {"value": value, "unit": unit, "cores": os.cpu_count(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def config_of(wl):
    from workloads import DecodeWorkload
    if isinstance(wl, DecodeWorkload):
        return {"workload": wl.name, "nseq": wl.nseq, "n_global": wl.n_global,
                "n_local": wl.n_local, "Hq": wl.Hq, "Hkv": wl.Hkv, "d": wl.d,
                "global_len": list(wl.global_len_range), "window": wl.window,
                "kv_shared": wl.kv_shared, "scale": wl.scale,
                "l2": "flushed before every timed step (256 MiB write)"}
    L = wl.layers[0]
    cfg = {"workload": wl.name, "layers": len(wl.layers), "B": L.B, "T": L.T, "S": L.S,
           "Hq": L.Hq, "Hkv": L.Hkv, "d": L.d, "window": L.window,
           "rope_base": L.rope.base, "yarn_factor": L.rope.yarn_factor,
           "l2": "flushed before every timed step (256 MiB write)"}
    if len(wl.layers) > 1:
        cfg["layer_shapes"] = [{"d": x.d, "Hq": x.Hq, "Hkv": x.Hkv, "window": x.window,
                                "rope_base": x.rope.base,
                                "rotate_fraction": x.rope.rotate_fraction} for x in wl.layers]
    return cfg


# ----------------------------------------------------------------------------------------

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="plamo3_local_prefill")
    ap.add_argument("--impl", choices=["gqa", "reference"], default="gqa")
    ap.add_argument("--no-extra", action="store_true", help="skip the other workloads")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--layer", type=int, default=None,
                    help="time only this layer of a multi-layer prefill workload (profiling)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)

    from workloads import DecodeModelWorkload, DecodeWorkload, get_workload
    wl = get_workload(args.workload)
    if isinstance(wl, DecodeModelWorkload):
        raise SystemExit(f"{wl.name} is reported in the extras of the default run only")
    if args.layer is not None:
        import dataclasses
        wl = dataclasses.replace(wl, name=f"{wl.name}[layer {args.layer}]",
                                 layers=(wl.layers[args.layer],))
        args.no_extra = True
    world, rank, local = dist_setup(args)

    if args.impl == "reference":
        run_reference(args, wl, world, rank)
        return

    import torch
    import global_causal_gqa_gb300 as gqa
    torch.cuda.set_device(local)
    if gqa.gqa_device_check() != 0:
        raise SystemExit("this build runs on sm_103 (GB300) only")
    stream = torch.cuda.current_stream()
    peaks, peak_src = load_peaks()
    is_decode = isinstance(wl, DecodeWorkload)
    clock_idx = local
    if is_decode:
        main_res = bench_decode(wl, args.steps, args.warmup, stream, peaks, peak_src, world,
                                True, clock_idx)
    else:
        main_res = bench_prefill(wl.name, list(wl.layers), args.steps, args.warmup, stream,
                                 peaks, peak_src, world, True, clock_idx)

    extra = []
    if world == 1 and not args.no_extra:
        for name in ("plamo3_local_prefill", "plamo3_global_prefill", "plamo3_decode_batch32",
                     "gemma4_period_6layer", "gemma4_decode_global",
                     "gemma4_decode_global_kv_shared", "gemma4_decode_local",
                     "plamo3_decode_64layer"):
            if name == wl.name:
                continue
            other = get_workload(name)
            ks, kw = min(args.steps, 10), 3
            if isinstance(other, DecodeModelWorkload):
                r = bench_decode_model(other, ks, kw, stream, peaks, peak_src)
            elif isinstance(other, DecodeWorkload):
                r = bench_decode(other, ks, kw, stream, peaks, peak_src, 1, False)
            else:
                r = bench_prefill(name, list(other.layers), ks, kw, stream, peaks, peak_src, 1,
                                  False)
            r.pop("clocks", None)
            extra.append({"workload": name, "steps": ks, "warmup": kw, **r})

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        target = wl if is_decode else wl.layers[0]
        cpu = cpu_baseline(wl.name, target, is_decode)

    if rank == 0:
        line = {
            "metric": METRIC, "value": main_res["value"], "unit": main_res["unit"],
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": main_res["ms_per_step"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) bf16)",
            "config": {**config_of(wl), "parallelism": f"replicas x{world}"},
            "roofline": main_res["roofline"], "cpu_baseline": cpu, "e2e": main_res["e2e"],
            "gpu_launches": main_res["gpu_launches"], "clocks": main_res["clocks"],
            "kernel_ms": main_res["kernel_ms"], "extra": extra,
        }
        if "per_layer" in main_res:
            line["per_layer"] = main_res["per_layer"]
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
