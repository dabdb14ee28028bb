#!/usr/bin/env python3
"""Benchmark of the NVFP4 paged-KV hot path on one GB300 (or N replicas).

A step is one pass of the path over the 16K-token causal prefill workload:
append the 16,384 tokens' K and V (8 kv heads, shuffled slot order) into the
NVFP4 cache, then run the A4Q paged prefill (32 q heads) over it.  The
headline value is prefill TFLOP/s per step (4*D FLOPs per visible causal
(query, key) pair per q head).  The same run also reports, each timed alone
with L2 flushed: append GB/s, the A4Q prefill in both modes and the
dequant-ahead variant at 16K, the other workloads of the benchmark matrix
(4 x 128 queries over 2K keys; 8 x 16-query tails over 16,400 keys, in GB/s
of cache read; 32,768 + 7,001 tokens, append and prefill), paged decode GB/s
on the batch-32 decode workload (kv_len ~ U[1K, 32K]), the measured A4Q error
against a BF16 query and against exact attention, and the CPU oracle's rate
on the host cores with its parity against the kernel's output.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
For N > 1 launch with torch.distributed.run; every rank runs an independent
replica (the path has no exchange step) and rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
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

from nvfp4_paged_kv_append_gb300 import workloads as W  # noqa: E402

METRIC = "A4Q NVFP4-KV paged prefill TFLOP/s @16K; append & decode HBM GB/s"
APPEND_BYTES_PER_TOKEN_HEAD = 2 * (256 + 72)     # K and V: bf16 read + codes/scales written
CACHE_BYTES_PER_TOKEN_HEAD = 2 * 72              # K and V codes + scales read by decode
L2_FLUSH_BYTES = 256 << 20
FP4_OVER_BF16 = 13.5 / 2.25                       # nominal dense FP4 : BF16 tensor ratio


# ---------------------------------------------------------------------------- helpers
def env_int(name, default):
    try:
        return int(os.environ.get(name, default))
    except ValueError:
        return default


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def physical_gpu_index() -> int:
    local = env_int("LOCAL_RANK", 0)
    cvd = os.environ.get("CUDA_VISIBLE_DEVICES")
    if cvd:
        parts = [p.strip() for p in cvd.split(",")]
        if local < len(parts) and parts[local].isdigit():
            return int(parts[local])
        return 0
    return local


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def prefill_flops_split(wl: W.Workload):
    """(QK FLOPs on FP4, PV FLOPs on 16-bit) for the A4Q path."""
    f = wl.flops()
    return f / 2, f / 2


def prefill_roof_s(wl: W.Workload, peaks, a4q=True) -> float:
    """Tensor-roofline time of one prefill: QK at the FP4 rate and PV at the
    16-bit rate (A4Q, a4q True), both at the 16-bit rate (dequant-ahead, a4q
    False), or both at the FP4 rate (a4q "fp4": the FP4 PV experiment)."""
    f_qk, f_pv = prefill_flops_split(wl)
    p16 = peaks["bf16_tflops"] * 1e12
    if a4q == "fp4":
        return (f_qk + f_pv) / (p16 * FP4_OVER_BF16)
    return (f_qk / (p16 * FP4_OVER_BF16) + f_pv / p16) if a4q else (f_qk + f_pv) / p16


# Issue cost of one tcgen05.mma by a single thread issuing back to back (one
# CTA, SM clock stamps; a probe on this GB300): block-scaled FP4 at M = 128,
# N = 128, K = 64 and f16 at M = 128, N = 128, K = 16 both take 68 cycles, so
# at M = 128 an FP4 instruction does 4x the f16 work, not the nominal 6x.
MMA_ISSUE_CYCLES = {"fp4_m128_n128_k64": 68, "f16_m128_n128_k16": 68}


def fp4_issue_note(wl: W.Workload, peaks, achieved_tflops: float) -> dict:
    """The measured M = 128 issue rate beside the nominal ratio the
    roofline uses, and the fraction the headline would have at that rate."""
    ratio = (64 / MMA_ISSUE_CYCLES["fp4_m128_n128_k64"]) / (16 / MMA_ISSUE_CYCLES["f16_m128_n128_k16"])
    f_qk, f_pv = prefill_flops_split(wl)
    p16 = peaks["bf16_tflops"] * 1e12
    t = f_qk / (p16 * ratio) + f_pv / p16
    return {"probe": "one thread issuing back to back, one CTA, cta_group::1 (M = 256 over a CTA pair not built)",
            "cycles": MMA_ISSUE_CYCLES, "fp4_over_bf16_at_m128": ratio,
            "frac_at_that_ratio": round(achieved_tflops / (wl.flops() / t / 1e12), 4)}


def host_cores() -> int:
    """Host cores this process may run on (its affinity mask)."""
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


_INPUTS = {}


def inputs_of(cfg: str) -> W.Inputs:
    """Seeded inputs of a named workload, generated once per run."""
    if cfg not in _INPUTS:
        _INPUTS[cfg] = W.make_inputs(W.CONFIGS[cfg]())
    return _INPUTS[cfg]


# ---------------------------------------------------------------------------- our arm
class Bench:
    def __init__(self, dev):
        from nvfp4_paged_kv_append_gb300 import binding as nk
        self.nk = nk
        self.dev = dev
        self.flush_buf = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        self.stream = torch.cuda.current_stream(dev)

    def flush(self):
        self.flush_buf.fill_(1.0)

    def time_fn(self, fn, steps, warmup, flush=True):
        """Per-call device time (ms) with CUDA events on the launching stream,
        L2 flushed before every call (outside the events)."""
        for _ in range(warmup):
            if flush:
                self.flush()
            fn()
        torch.cuda.synchronize(self.dev)
        times = []
        for _ in range(steps):
            if flush:
                self.flush()
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record(self.stream)
            fn()
            e.record(self.stream)
            times.append((s, e))
        torch.cuda.synchronize(self.dev)
        return [s.elapsed_time(e) for s, e in times]


def time_graph(nk_bench, fn, steps, warmup=3):
    """Per-replay device time (ms) of `fn` captured once into a CUDA graph
    (no host launch gaps inside the events); L2 flushed before every replay,
    outside the events.  Returns None if the capture is not possible."""
    try:
        fn()
        torch.cuda.synchronize(nk_bench.dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        torch.cuda.synchronize(nk_bench.dev)
        return nk_bench.time_fn(g.replay, steps, warmup)
    except Exception as e:  # pragma: no cover - reported in the JSON line
        print(f"graph timing unavailable: {e}", file=sys.stderr)
        return None


def setup_prefill(nk, dev, inp):
    wl = inp.wl
    order = W.shuffled_append_order(inp.wl.total_kv)
    k = inp.k[order].contiguous().to(dev)
    v = inp.v[order].contiguous().to(dev)
    slots = inp.slot_mapping[order].contiguous().to(dev)
    cache = nk.Cache(inp.num_pages, wl.num_kv_heads, inp.k_global, inp.v_global, device=dev)
    q = inp.q.to(dev)
    pt, kvl, qo = inp.page_table.to(dev), inp.kv_lens.to(dev), inp.qo_indptr.to(dev)
    out = torch.empty_like(q)
    # room for repack mode (V dequantized once per KV tile) and the schedule-only size
    ws = torch.empty(nk.nvfp4_workspace_bytes(nk.OP_PREFILL, wl.batch, wl.num_q_heads, wl.num_kv_heads,
                                              wl.total_q, pt.shape[1] * 16), dtype=torch.uint8, device=dev)
    ws_min = torch.empty(nk.nvfp4_workspace_bytes(nk.OP_PREFILL, wl.batch, wl.num_q_heads, wl.num_kv_heads,
                                                  wl.total_q, 0), dtype=torch.uint8, device=dev)
    return dict(inp=inp, k=k, v=v, slots=slots, cache=cache, q=q, pt=pt, kvl=kvl, qo=qo, out=out, ws=ws,
                ws_min=ws_min)


def run_ours(args, rank, world, dev):
    nk_bench = Bench(dev)
    nk = nk_bench.nk
    peaks = measured_peaks()
    inp = inputs_of(args.config)
    wl = inp.wl
    P = setup_prefill(nk, dev, inp)

    def append():
        nk.nvfp4_kv_append(P["k"], P["v"], P["slots"], P["cache"])

    def prefill(variant=nk.VARIANT_A4Q, ws="ws"):
        nk.nvfp4_paged_prefill(P["q"], P["cache"], P["pt"], P["kvl"], P["qo"], causal=wl.causal,
                               sm_scale=inp.sm_scale, variant=variant, out=P["out"], workspace=P[ws])

    def plan(variant=nk.VARIANT_A4Q, ws="ws"):
        nk.nvfp4_paged_prefill_plan(P["cache"], wl.total_q, wl.num_q_heads, P["pt"], P["kvl"], P["qo"], P[ws],
                                    causal=wl.causal, variant=variant)

    def attend(variant=nk.VARIANT_A4Q, ws="ws"):
        nk.nvfp4_paged_prefill_run(P["q"], P["cache"], P["pt"], P["kvl"], P["qo"], P[ws], causal=wl.causal,
                                   sm_scale=inp.sm_scale, variant=variant, out=P["out"])

    def step():
        append()
        prefill()

    # correctness guard before timing: the library must report a clean status
    step()
    torch.cuda.synchronize(dev)
    st = nk.nvfp4kv_get_device_status()
    if st != 0:
        raise RuntimeError(f"device status {st} after the first step")

    flops = wl.flops()
    f_qk, f_pv = prefill_flops_split(wl)

    # ---- headline: K timed steps, barrier + synchronize on both sides.
    # Clocks are sampled from the warm-up through the component timings.
    clocks = ClockSampler(physical_gpu_index())
    clocks.start()
    time.sleep(0.3)
    for _ in range(args.warmup):
        nk_bench.flush()
        step()
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    t_wall0 = time.perf_counter()
    ev = []
    for _ in range(args.steps):
        nk_bench.flush()
        s, m, r, e = (torch.cuda.Event(enable_timing=True) for _ in range(4))
        s.record(nk_bench.stream)
        append()
        m.record(nk_bench.stream)
        plan()     # schedule + repack pre-pass
        r.record(nk_bench.stream)
        attend()   # the attention kernel alone
        e.record(nk_bench.stream)
        ev.append((s, m, r, e))
    torch.cuda.synchronize(dev)
    t_wall = time.perf_counter() - t_wall0
    step_ms = [s.elapsed_time(e) for s, m, r, e in ev]
    app_ms = [s.elapsed_time(m) for s, m, r, e in ev]
    pre_ms = [m.elapsed_time(e) for s, m, r, e in ev]
    plan_ms = [m.elapsed_time(r) for s, m, r, e in ev]
    attn_ms = [r.elapsed_time(e) for s, m, r, e in ev]
    ms = max_over_ranks(statistics.mean(step_ms), world, dev)
    value = whole_job_tflops(flops, world, ms)

    # the A4Q output of the last timed step, for the oracle's parity check
    a4q_out = P["out"].float().cpu() if rank == 0 and not args.no_cpu_baseline else None

    # ---- components (each timed alone, L2 flushed before every call)
    K = max(min(args.steps, 50), 5)
    app = nk_bench.time_fn(append, K, 3)
    app_g = time_graph(nk_bench, append, K)
    pre = nk_bench.time_fn(prefill, K, 3)
    dqa = nk_bench.time_fn(lambda: prefill(nk.VARIANT_DQ_AHEAD), K, 3)
    pre_ik = nk_bench.time_fn(lambda: prefill(nk.VARIANT_A4Q, "ws_min"), K, 3)
    dqa_ik = nk_bench.time_fn(lambda: prefill(nk.VARIANT_DQ_AHEAD, "ws_min"), K, 3)
    fp4pv = nk_bench.time_fn(lambda: prefill(nk.VARIANT_A4Q_FP4PV), K, 3)
    app_bytes = APPEND_BYTES_PER_TOKEN_HEAD * wl.total_kv * wl.num_kv_heads
    comps = {
        "append": dict(gbs_entry(app, app_bytes, peaks, app_g), copy_same_bytes=copy_reference(nk_bench, app_bytes, K)),
        "prefill_a4q": tflops_entry(pre, wl, peaks, True, "V repacked once per KV tile"),
        "prefill_a4q_inkernel": tflops_entry(pre_ik, wl, peaks, True, "V dequantized in the kernel"),
        "prefill_dq_ahead": tflops_entry(dqa, wl, peaks, False, "K and V repacked once per KV tile"),
        "prefill_dq_ahead_inkernel": tflops_entry(dqa_ik, wl, peaks, False, "K and V dequantized in the kernel"),
        "prefill_a4q_fp4pv": tflops_entry(fp4pv, wl, peaks, "fp4", FP4PV_MODE),
    }
    if not args.no_matrix:
        comps["shortq"] = shortq_component(nk, nk_bench, dev, K, peaks)
        comps["tails"] = tails_component(nk, nk_bench, dev, K, peaks)
        comps["prefill32k"] = long_component(nk, nk_bench, dev, K, peaks)
    comps["decode"] = decode_component(nk, nk_bench, dev, K)
    if not args.no_matrix:
        comps["fp8"] = fp8_component(nk, nk_bench, dev, K, peaks, comps)
    clk = clocks.stop()

    # the dominant kernel: the attention launch, timed inside the timed steps
    achieved = flops / (statistics.mean(attn_ms) * 1e-3) / 1e12
    p16 = peaks["bf16_tflops"]
    peak_eff = flops / prefill_roof_s(wl, peaks) / 1e12

    # ---- end to end through the public API with host buffers
    e2e = e2e_measure(nk, nk_bench, dev, P, wl, args) if not args.no_e2e else None

    result = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "nvfp4(e2m1+e4m3) QK, f16 PV, f32 accum", "data": "synthetic",
        "config": bench_config(wl, world),
        "step_breakdown_ms": {"append": round(statistics.mean(app_ms), 4), "prefill": round(statistics.mean(pre_ms), 4),
                              "prefill_plan_and_repack": round(statistics.mean(plan_ms), 4),
                              "prefill_attention": round(statistics.mean(attn_ms), 4)},
        "roofline": {"bound": "tensor", "kernel": "nvfp4_prefill_a4q_2cta_sm103_kernel", "achieved": round(achieved, 2),
                     "peak": round(peak_eff, 2), "unit": "TFLOP/s", "frac": round(achieved / peak_eff, 4),
                     "traffic": prefill_traffic_bytes(),
                     "peak_basis": f"t = F_QK/(bf16 x {FP4_OVER_BF16:g}) + F_PV/bf16 with bf16 = {p16} TFLOP/s "
                                   f"({peaks['source']} burst)",
                     "fp4_mma_issue": fp4_issue_note(wl, peaks, achieved)},
        "components": comps,
        "e2e": e2e,
        "gpu_launches": 4 * args.steps,  # append, schedule, repack pre-pass, attention
        "clocks": clk,
        "wall_s_timed_loop": round(t_wall, 3),
    }
    if not args.no_accuracy:
        result["a4q_error"] = a4q_error_report(nk, dev)
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(args.cpu_seconds, a4q_out)
    return result


def copy_reference(nk_bench, nbytes, K):
    """A plain device copy that moves the same number of bytes (nbytes/2 read
    + nbytes/2 written), timed like the components: what a transfer of this
    size reaches on this GPU, launch, ramp and drain included."""
    src = torch.empty(nbytes // 2, dtype=torch.uint8, device=nk_bench.dev).fill_(1)
    dst = torch.empty_like(src)
    t = statistics.mean(nk_bench.time_fn(lambda: dst.copy_(src), K, 3))
    gbs = nbytes / (t * 1e-3) / 1e9
    return {"ms": round(t, 4), "GB/s": round(gbs, 1), "frac_of_hbm": round(gbs / measured_peaks()["hbm_gbs"], 4),
            "what": "torch copy of nbytes/2 (same bytes moved), L2 flushed before every call"}


def gbs_entry(times, nbytes, peaks, graph_times=None):
    """Component entry of an HBM-bound call: mean time, algorithmic GB/s and
    the fraction of the measured copy bandwidth (and the same replayed from a
    CUDA graph, when given)."""
    t = statistics.mean(times)
    gbs = nbytes / (t * 1e-3) / 1e9
    e = {"ms": round(t, 4), "GB/s": round(gbs, 1), "frac_of_hbm": round(gbs / peaks["hbm_gbs"], 4), "bytes": nbytes}
    if graph_times:
        tg = statistics.mean(graph_times)
        g = nbytes / (tg * 1e-3) / 1e9
        e.update({"graph_ms": round(tg, 4), "graph_GB/s": round(g, 1), "graph_frac_of_hbm": round(g / peaks["hbm_gbs"], 4)})
    return e


def tflops_entry(times, wl, peaks, a4q, mode):
    """Component entry of a prefill: mean time, TFLOP/s and the fraction of
    its tensor roofline (mixed FP4/16-bit for A4Q, 16-bit for dequant-ahead)."""
    t = statistics.mean(times)
    roof = "FP4 QK + FP4 PV" if a4q == "fp4" else "FP4 QK + 16-bit PV" if a4q else "16-bit QK + PV"
    return {"workload": wl.name, "ms": round(t, 4), "TFLOP/s": round(wl.flops() / (t * 1e-3) / 1e12, 2),
            "frac_of_roofline": round(prefill_roof_s(wl, peaks, a4q) / (t * 1e-3), 4),
            "roofline": roof, "mode": mode}


class PrefillCase:
    """A workload's cache (built by the library's append) and its prefill
    buffers, for the component timings."""

    def __init__(self, nk, dev, inp, shuffled_append=False):
        self.nk, self.inp = nk, inp
        wl = inp.wl
        order = W.shuffled_append_order(wl.total_kv) if shuffled_append else torch.arange(wl.total_kv)
        self.k = inp.k[order].contiguous().to(dev)
        self.v = inp.v[order].contiguous().to(dev)
        self.slots = inp.slot_mapping[order].contiguous().to(dev)
        self.cache = nk.Cache(inp.num_pages, wl.num_kv_heads, inp.k_global, inp.v_global, device=dev)
        self.append()
        self.q = inp.q.to(dev)
        self.pt, self.kvl, self.qo = inp.page_table.to(dev), inp.kv_lens.to(dev), inp.qo_indptr.to(dev)
        self.out = torch.empty_like(self.q)
        self.ws = torch.empty(nk.nvfp4_workspace_bytes(nk.OP_PREFILL, wl.batch, wl.num_q_heads, wl.num_kv_heads,
                                                       wl.total_q, self.pt.shape[1] * 16),
                              dtype=torch.uint8, device=dev)

    def append(self):
        self.nk.nvfp4_kv_append(self.k, self.v, self.slots, self.cache)

    def prefill(self, variant):
        wl = self.inp.wl
        self.nk.nvfp4_paged_prefill(self.q, self.cache, self.pt, self.kvl, self.qo, causal=wl.causal,
                                    sm_scale=self.inp.sm_scale, variant=variant, out=self.out, workspace=self.ws)


FP4PV_MODE = ("experiment: A4Q QK, then P coded to NVFP4 per 16 keys and V re-coded once per 128-key tile "
              "along tokens, PV on block-scaled FP4 MMA (one CTA per SM)")


def shortq_component(nk, nk_bench, dev, K, peaks):
    """Batch 4 x q 128 at the end of kv 2,048, 32/8 heads, permuted pages (the
    repack comparison shape; four q tiles per kv head): A4Q runs the in-kernel
    mode (repack needs eight q tiles per kv head for A4Q), dequant-ahead the
    repack mode (two)."""
    c = PrefillCase(nk, dev, inputs_of("shortq"))
    wl = c.inp.wl
    a = nk_bench.time_fn(lambda: c.prefill(nk.VARIANT_A4Q), K, 3)
    d = nk_bench.time_fn(lambda: c.prefill(nk.VARIANT_DQ_AHEAD), K, 3)
    f = nk_bench.time_fn(lambda: c.prefill(nk.VARIANT_A4Q_FP4PV), K, 3)
    return {"a4q": tflops_entry(a, wl, peaks, True, "in-kernel"),
            "dq_ahead": tflops_entry(d, wl, peaks, False, "repack"),
            "a4q_fp4pv": tflops_entry(f, wl, peaks, "fp4", FP4PV_MODE)}


def tails_component(nk, nk_bench, dev, K, peaks):
    """Chunked-prefill tails: 8 requests x 16 new queries over 16,400 cached
    tokens, 32/8 heads.  One q tile per (request, kv head), so the in-kernel
    mode runs; bound by reading the cache: GB/s of cache bytes read."""
    c = PrefillCase(nk, dev, inputs_of("tails"))
    wl = c.inp.wl
    kv_bytes = CACHE_BYTES_PER_TOKEN_HEAD * wl.total_kv * wl.num_kv_heads
    res = {}
    for name, variant in (("a4q", nk.VARIANT_A4Q), ("dq_ahead", nk.VARIANT_DQ_AHEAD)):
        t = nk_bench.time_fn(lambda: c.prefill(variant), K, 3)
        e = gbs_entry(t, kv_bytes, peaks)
        e["TFLOP/s"] = round(wl.flops() / (statistics.mean(t) * 1e-3) / 1e12, 2)
        e["mode"] = "in-kernel (one q tile per request and kv head)"
        res[name] = e
    res["workload"] = wl.name
    return res


def long_component(nk, nk_bench, dev, K, peaks):
    """32,768 + 7,001 tokens in one batch, 64/8 heads: the append of all
    39,769 tokens (GB/s) and the A4Q prefill (TFLOP/s, repack mode)."""
    c = PrefillCase(nk, dev, inputs_of("prefill32k"), shuffled_append=True)
    wl = c.inp.wl
    app = nk_bench.time_fn(c.append, K, 3)
    pre = nk_bench.time_fn(lambda: c.prefill(nk.VARIANT_A4Q), max(3, K // 4), 2)
    res = {"workload": wl.name,
           "append": gbs_entry(app, APPEND_BYTES_PER_TOKEN_HEAD * wl.total_kv * wl.num_kv_heads, peaks),
           "prefill_a4q": tflops_entry(pre, wl, peaks, True, "repack")}
    res["append"]["copy_same_bytes"] = copy_reference(nk_bench, res["append"]["bytes"], K)
    del c
    torch.cuda.empty_cache()
    return res


def decode_component(nk, nk_bench, dev, K):
    wl = W.decode_batch()
    inp = W.make_inputs(wl)
    cache = nk.Cache(inp.num_pages, wl.num_kv_heads, inp.k_global, inp.v_global, device=dev)
    nk.nvfp4_kv_append(inp.k.to(dev), inp.v.to(dev), inp.slot_mapping.to(dev), cache)
    q, pt, kvl = inp.q.to(dev), inp.page_table.to(dev), inp.kv_lens.to(dev)
    out = torch.empty_like(q)
    ws = torch.empty(nk.nvfp4_workspace_bytes(nk.OP_DECODE, wl.batch, wl.num_q_heads, wl.num_kv_heads, 0,
                                              pt.shape[1] * 16), dtype=torch.uint8, device=dev)

    def dec():
        nk.nvfp4_paged_decode(q, cache, pt, kvl, sm_scale=inp.sm_scale, out=out, workspace=ws)

    t = nk_bench.time_fn(dec, K, 3)
    tg = time_graph(nk_bench, dec, K)
    e = gbs_entry(t, CACHE_BYTES_PER_TOKEN_HEAD * wl.total_kv * wl.num_kv_heads, measured_peaks(), tg)
    e["workload"] = wl.name
    return e


FP8_APPEND_BYTES_PER_TOKEN_HEAD = 2 * (256 + 128)  # K and V: bf16 read + one code byte per value written
FP8_CACHE_BYTES_PER_TOKEN_HEAD = 2 * 128           # K and V codes read by decode


def fp8_component(nk, nk_bench, dev, K, peaks, comps):
    """The FP8 (E4M3) comparison cache on the same shapes: append and prefill
    of the 16K workload, decode of the batch-32 workload, and the NVFP4 / FP8
    time ratios ("NVFP4 KV cache A4Q prefill explained", section "Build the
    benchmark matrix": FP8 and the NVFP4 paths on the same revision)."""
    inp = inputs_of("prefill16k")
    wl = inp.wl
    ks, vs = W.fp8_scale(inp.k), W.fp8_scale(inp.v)
    order = W.shuffled_append_order(wl.total_kv)
    k, v, slots = (inp.k[order].contiguous().to(dev), inp.v[order].contiguous().to(dev),
                   inp.slot_mapping[order].contiguous().to(dev))
    cache = nk.Fp8Cache(inp.num_pages, wl.num_kv_heads, ks, vs, device=dev)
    q, pt, kvl, qo = inp.q.to(dev), inp.page_table.to(dev), inp.kv_lens.to(dev), inp.qo_indptr.to(dev)
    out = torch.empty_like(q)
    ws = torch.empty(nk.fp8_workspace_bytes(nk.OP_PREFILL, wl.batch, wl.num_q_heads, wl.num_kv_heads, wl.total_q,
                                            pt.shape[1] * 16), dtype=torch.uint8, device=dev)
    app = nk_bench.time_fn(lambda: nk.fp8_kv_append(k, v, slots, cache), K, 3)
    pre = nk_bench.time_fn(lambda: nk.fp8_paged_prefill(q, cache, pt, kvl, qo, causal=True, sm_scale=inp.sm_scale,
                                                        out=out, workspace=ws), K, 3)
    res = {"format": "E4M3, one fp32 scale per tensor (amax/448), 128 B per (token, kv head) per tensor",
           "append": gbs_entry(app, FP8_APPEND_BYTES_PER_TOKEN_HEAD * wl.total_kv * wl.num_kv_heads, peaks),
           "prefill": tflops_entry(pre, wl, peaks, False, "BF16 query; K/V converted once per 128-key tile, "
                                                          "BF16 QK + FP16 PV")}
    del k, v, slots, cache, q, out, ws
    torch.cuda.empty_cache()
    dwl = W.decode_batch()
    dinp = W.make_inputs(dwl)
    dcache = nk.Fp8Cache(dinp.num_pages, dwl.num_kv_heads, W.fp8_scale(dinp.k), W.fp8_scale(dinp.v), device=dev)
    nk.fp8_kv_append(dinp.k.to(dev), dinp.v.to(dev), dinp.slot_mapping.to(dev), dcache)
    dq, dpt, dkvl = dinp.q.to(dev), dinp.page_table.to(dev), dinp.kv_lens.to(dev)
    dout = torch.empty_like(dq)
    dws = torch.empty(nk.fp8_workspace_bytes(nk.OP_DECODE, dwl.batch, dwl.num_q_heads, dwl.num_kv_heads, 0,
                                             dpt.shape[1] * 16), dtype=torch.uint8, device=dev)
    dec = nk_bench.time_fn(lambda: nk.fp8_paged_decode(dq, dcache, dpt, dkvl, sm_scale=dinp.sm_scale, out=dout,
                                                       workspace=dws), K, 3)
    res["decode"] = gbs_entry(dec, FP8_CACHE_BYTES_PER_TOKEN_HEAD * dwl.total_kv * dwl.num_kv_heads, peaks)
    res["decode"]["workload"] = dwl.name
    res["nvfp4_over_fp8_time"] = {
        "append_16k": round(comps["append"]["ms"] / res["append"]["ms"], 3),
        "prefill_16k_a4q": round(comps["prefill_a4q"]["ms"] / res["prefill"]["ms"], 3),
        "prefill_16k_dq_ahead": round(comps["prefill_dq_ahead"]["ms"] / res["prefill"]["ms"], 3),
        "decode_b32": round(comps["decode"]["ms"] / res["decode"]["ms"], 3),
        "pages_context": "SM120 with FlashInfer: prefill 16K stock 21.0 / A4Q 18.0 vs FP8 11.1 ms; "
                         "decode 9.63 vs 12.35 us; append 8.39 vs 3.01 us (other hardware)"}
    return res


def e2e_measure(nk, nk_bench, dev, P, wl, args):
    """Host (pinned) inputs copied in, append + prefill through the public
    API, output copied back: every step's copies are inside the timed
    region.  Steps are pipelined the way a server runs them: the inputs of
    step i+1 are copied in (one stream) while step i computes (another) and
    the output of step i-1 is copied out (a third), with double-buffered
    device inputs and outputs."""
    inp = P["inp"]
    order = W.shuffled_append_order(inp.wl.total_kv)
    hk = inp.k[order].contiguous().pin_memory()
    hv = inp.v[order].contiguous().pin_memory()
    hs = inp.slot_mapping[order].contiguous().pin_memory()
    hq = inp.q.contiguous().pin_memory()
    hpt, hkv, hqo = inp.page_table.pin_memory(), inp.kv_lens.pin_memory(), inp.qo_indptr.pin_memory()
    ho = torch.empty(hq.shape, dtype=torch.bfloat16).pin_memory()
    host_in = (hk, hv, hs, hq, hpt, hkv, hqo)
    dev_in = [tuple(torch.empty_like(t, device=dev) for t in host_in) for _ in range(2)]
    dev_out = [torch.empty_like(P["out"]) for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = ho.numel() * ho.element_size()
    s_in, s_comp, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    in_ready = [torch.cuda.Event() for _ in range(2)]
    comp_done = [torch.cuda.Event() for _ in range(2)]
    out_done = [torch.cuda.Event() for _ in range(2)]

    def step(i):
        buf = i % 2
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(comp_done[buf])  # step i-2 no longer reads these inputs
            for d, h in zip(dev_in[buf], host_in):
                d.copy_(h, non_blocking=True)
            in_ready[buf].record(s_in)
        with torch.cuda.stream(s_comp):
            s_comp.wait_event(in_ready[buf])
            if i >= 2:
                s_comp.wait_event(out_done[buf])  # step i-2's output has been copied out
            dk, dv, ds, dq, dpt, dkv, dqo = dev_in[buf]
            nk.nvfp4_kv_append(dk, dv, ds, P["cache"])
            nk.nvfp4_paged_prefill(dq, P["cache"], dpt, dkv, dqo, causal=wl.causal, sm_scale=inp.sm_scale,
                                   out=dev_out[buf], workspace=P["ws"])
            comp_done[buf].record(s_comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(comp_done[buf])
            ho.copy_(dev_out[buf], non_blocking=True)
            out_done[buf].record(s_out)

    def run(n):
        for i in range(n):
            step(i)
        for st in (s_in, s_comp, s_out):
            torch.cuda.current_stream(dev).wait_stream(st)

    run(3)  # warm-up
    torch.cuda.synchronize(dev)
    n = max(args.steps, 3)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    for st in (s_in, s_comp, s_out):
        st.wait_stream(torch.cuda.current_stream(dev))
    run(n)
    t1.record()
    torch.cuda.synchronize(dev)
    ms = t0.elapsed_time(t1) / n
    return {"value": round(wl.flops() / (ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s", "ms_per_step": round(ms, 4),
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "pipeline": "copy-in of step i+1, compute of step i and copy-out of step i-1 on three streams",
            "l2": "not flushed: every step moves 201 MB in and 134 MB out, more than the 129 MB L2"}


def bench_config(wl, world):
    """The `config` object of the JSON line (the same for both arms)."""
    return {"workload": wl.name, "batch": wl.batch, "seq_len": wl.q_lens[0], "q_heads": wl.num_q_heads,
            "kv_heads": wl.num_kv_heads, "head_dim": 128, "page_size": 16, "causal": wl.causal,
            "step": "append(K,V 16384 tok, shuffled slots) + A4Q paged prefill (repack mode)",
            "flops_per_step": wl.flops(), "l2": "flushed (256 MB write) before every timed step, outside the events",
            "parallelism": f"replicas x{world}"}


# ---------------------------------------------------------------------------- A4Q accuracy
# Measured accuracy of the A4Q query ("NVFP4 KV cache A4Q prefill explained",
# section "Make query accuracy a release gate": lengths, head shapes, causal
# masks and scale outliers are checked, the query scale scheme -- single or
# dual level -- is a recorded choice, and long contexts amplify score error).
# Every output compared comes from the library's kernels:
#   o_a4q    A4Q prefill (query quantized to NVFP4 inside the kernel),
#   o_bf16q  dequant-ahead prefill (BF16 query) on the same NVFP4 cache,
# and o_exact is softmax attention in float64 (plain torch on the host) over
# the UNQUANTIZED bf16 Q, K and V.  So o_a4q - o_bf16q is what the query
# quantization adds, o_bf16q - o_exact is the NVFP4 cache alone, and
# o_a4q - o_exact the whole A4Q path.
Q_SCHEMES = {
    "per_row": "dual level per (token, head) row: g_row = amax_row/2688 (q_global_scale 0, the default)",
    "per_tensor": "dual level per tensor: one g = amax(Q)/2688 for every row",
    "single_level": "single level: g = 1, the E4M3 block scales alone",
}


def q_scale_for(scheme: str, q: torch.Tensor) -> float:
    """The q_global_scale argument that selects `scheme` for query tensor q."""
    if scheme == "per_row":
        return 0.0
    if scheme == "single_level":
        return 1.0
    amax = np.float32(q.float().abs().max().item())
    return float(np.float32(amax / np.float32(2688.0)))


def exact_rows(inp: W.Inputs, rows):
    """float64 softmax attention over the unquantized bf16 values for the
    given (request, position) rows: {(b, i): [Hq, D] numpy}."""
    wl = inp.wl
    G = wl.group
    out = {}
    by_req = {}
    for b, i in rows:
        by_req.setdefault(b, set()).add(i)
    for b, positions in by_req.items():
        pos = torch.tensor(sorted(positions), dtype=torch.int64)
        q_len, kv_len = wl.q_lens[b], wl.kv_lens[b]
        k0 = int(inp.kv_indptr[b])
        qrows = inp.q[int(inp.qo_indptr[b]) + pos].to(torch.float64)          # [n, Hq, D]
        k = inp.k[k0:k0 + kv_len].to(torch.float64)                             # [kv, Hkv, D]
        v = inp.v[k0:k0 + kv_len].to(torch.float64)
        last = (kv_len - q_len + pos) if wl.causal else torch.full_like(pos, kv_len - 1)
        mask = torch.arange(kv_len)[None, :] > last[:, None]                   # [n, kv]
        o = torch.empty(len(pos), wl.num_q_heads, wl.head_dim, dtype=torch.float64)
        for h in range(wl.num_kv_heads):
            s = torch.einsum("ngd,kd->ngk", qrows[:, h * G:(h + 1) * G, :], k[:, h, :]) * inp.sm_scale
            p = torch.softmax(s.masked_fill(mask[:, None, :], -math.inf), dim=-1)
            o[:, h * G:(h + 1) * G, :] = torch.einsum("ngk,kd->ngd", p, v[:, h, :])
        for r, i in enumerate(pos.tolist()):
            out[(b, i)] = o[r].numpy()
    return out


def err_stats(got: dict, ref: dict):
    """max-abs and relative Frobenius of got - ref over the rows of ref."""
    d = np.stack([got[k] - ref[k] for k in ref])
    r = np.stack([ref[k] for k in ref])
    return {"max_abs": round(float(np.abs(d).max()), 6),
            "rel_fro": round(float(np.linalg.norm(d) / max(np.linalg.norm(r), 1e-30)), 6)}


def kernel_rows(out: torch.Tensor, inp: W.Inputs, rows):
    o = out.float().cpu().numpy().astype(np.float64)
    return {(b, i): o[int(inp.qo_indptr[b]) + i] for b, i in rows}


def accuracy_run(nk, dev, inp, rows, schemes=("per_row",), fp4pv=False):
    """Kernel outputs on `rows` of one workload: the BF16-query dequant-ahead
    prefill and the A4Q prefill under each query scale scheme (and the FP4 PV
    experiment)."""
    c = PrefillCase(nk, dev, inp)
    res = {}
    c.prefill(nk.VARIANT_DQ_AHEAD)
    res["bf16q"] = kernel_rows(c.out, inp, rows)
    for sch in schemes:
        wl = inp.wl
        nk.nvfp4_paged_prefill(c.q, c.cache, c.pt, c.kvl, c.qo, causal=wl.causal, sm_scale=inp.sm_scale,
                               variant=nk.VARIANT_A4Q, out=c.out, workspace=c.ws,
                               q_global_scale=q_scale_for(sch, inp.q))
        res[sch] = kernel_rows(c.out, inp, rows)
    if fp4pv:
        c.prefill(nk.VARIANT_A4Q_FP4PV)
        res["fp4pv"] = kernel_rows(c.out, inp, rows)
    torch.cuda.synchronize(dev)
    st = nk.nvfp4kv_get_device_status()
    if st != 0:
        raise RuntimeError(f"device status {st} in the accuracy run")
    del c
    torch.cuda.empty_cache()
    return res


def a4q_error_report(nk, dev):
    """The a4q_error object of the benchmark line: the A4Q error on sampled
    rows of the outlier config (every row), the 16K and the 32K + 7K configs,
    then the query scale schemes x context length."""
    per = {}
    for cfg, rows_of in (("tiny", lambda wl: [(b, i) for b in range(wl.batch) for i in range(wl.q_lens[b])]),
                         ("prefill16k", lambda wl: W.sample_rows(wl, 6)),
                         ("prefill32k", lambda wl: W.sample_rows(wl, 3))):
        inp = inputs_of(cfg)
        rows = rows_of(inp.wl)
        k = accuracy_run(nk, dev, inp, rows, fp4pv=True)
        ex = exact_rows(inp, rows)
        per[cfg] = {"workload": inp.wl.name, "values": inp.wl.dist, "rows": len(rows),
                    "a4q_vs_bf16q": err_stats(k["per_row"], k["bf16q"]),
                    "a4q_vs_exact": err_stats(k["per_row"], ex), "bf16q_vs_exact": err_stats(k["bf16q"], ex),
                    "fp4pv_vs_a4q": err_stats(k["fp4pv"], k["per_row"]), "fp4pv_vs_exact": err_stats(k["fp4pv"], ex)}
    sweep = {}
    for L in (1024, 4096, 16384, 32768):
        wl = W.Workload(f"tail_q64_kv{L}_h32x8_outliers", [64], [L], 32, 8, dist="outliers", seed=L)
        inp = W.make_inputs(wl)
        rows = W.sample_rows(wl, 6)
        k = accuracy_run(nk, dev, inp, rows, tuple(Q_SCHEMES))
        ex = exact_rows(inp, rows)
        e = {"rows": len(rows), "bf16q_vs_exact": err_stats(k["bf16q"], ex)}
        for sch in Q_SCHEMES:
            e[sch] = {"vs_exact": err_stats(k[sch], ex), "vs_bf16q": err_stats(k[sch], k["bf16q"])}
        sweep[str(L)] = e
    return {"q_scheme": Q_SCHEMES["per_row"] + "; then one E4M3 scale per 16 values (nearest even) and E2M1 "
                                               "codes (nearest even), the cache's block codec",
            "outputs": "o_a4q: A4Q kernel; o_bf16q: dequant-ahead kernel (BF16 query) on the same NVFP4 cache; "
                       "o_fp4pv: the FP4 PV experiment (A4Q QK, NVFP4 P, V re-coded along tokens); "
                       "o_exact: float64 attention on the unquantized bf16 Q, K, V",
            "configs": per,
            "q_scheme_x_kv_len": {"workload": "64-query tail at the end of kv_len keys, 32/8 heads, N(0,1) with "
                                              "2% of the channels x8; seeded rows",
                                  "schemes": Q_SCHEMES, "by_kv_len": sweep}}


# ---------------------------------------------------------------------------- oracle arm
_ORACLE = {}


def oracle_setup():
    """CPU oracle state for the 16K workload: the full cache written by the
    oracle's append, and kv head 0 decoded (setup, timed separately)."""
    if _ORACLE:
        return _ORACLE
    import oracle
    wl = W.full_prefill_16k()
    inp = W.make_inputs(wl)
    pools = oracle.Pools(inp.num_pages, wl.num_kv_heads)
    t0 = time.perf_counter()
    oracle.kv_append(pools, inp.k.float().numpy(), inp.v.float().numpy(), inp.slot_mapping.numpy(),
                     inp.k_global, inp.v_global)
    t_app = time.perf_counter() - t0
    kd = oracle.gather_decode(pools, "k", inp.page_table[0].numpy(), wl.kv_lens[0], 0, inp.k_global)
    vd = oracle.gather_decode(pools, "v", inp.page_table[0].numpy(), wl.kv_lens[0], 0, inp.v_global)
    _ORACLE.update(dict(wl=wl, inp=inp, kd=kd, vd=vd, q=inp.q.float().numpy(), append_s=t_app,
                        append_gbs=APPEND_BYTES_PER_TOKEN_HEAD * wl.total_kv * wl.num_kv_heads / t_app / 1e9))
    return _ORACLE


def oracle_rows(seconds: float, workers: int, collect: bool = False):
    """The oracle as it stands: A4Q attention for seeded query rows of the
    four q heads of kv head 0 of the 16K workload, on `workers` host threads
    (each runs independent rows; the C oracle releases the interpreter lock),
    until `seconds` have passed.  Returns (TFLOP/s, rows, seconds, results)
    with results a list of (positions, q head, o) when `collect`."""
    import concurrent.futures as cf

    import oracle
    o = oracle_setup()
    wl, inp = o["wl"], o["inp"]
    t0 = time.perf_counter()

    def worker(idx):
        rng = np.random.default_rng(1000 + idx)
        flops, rows, res = 0.0, 0, []
        while time.perf_counter() - t0 < seconds:
            pos = np.sort(rng.integers(0, wl.q_lens[0], 8)).astype(np.int32)
            for gq in range(wl.group):
                qd = oracle.decode_q_a4q(o["q"][pos, gq, :])
                out, _ = oracle.attention_rows(qd, pos, wl.q_lens[0], o["kd"], o["vd"], True, inp.sm_scale)
                flops += float(np.sum(4.0 * 128 * (pos.astype(np.float64) + 1)))
                rows += len(pos)
                if collect:
                    res.append((pos, gq, out))
        return flops, rows, res

    with cf.ThreadPoolExecutor(max_workers=workers) as ex:
        parts = list(ex.map(worker, range(workers)))
    dt = time.perf_counter() - t0
    flops = sum(p[0] for p in parts)
    rows = sum(p[1] for p in parts)
    return flops / dt / 1e12, rows, dt, [r for p in parts for r in p[2]]


def half_bf16_ulp(x):
    a = np.maximum(np.abs(x), 2.0 ** -126)
    return np.ldexp(1.0, np.floor(np.log2(a)).astype(np.int64) - 8)


def cpu_baseline(seconds, gpu_out=None):
    """The oracle timed on the host's cores; when the kernel's output of the
    same workload is given, the oracle rows are also compared with it (raw
    max-abs, max-abs beyond the half bf16 ulp of the stored output, relative
    Frobenius)."""
    cores = host_cores()
    v, rows, dt, res = oracle_rows(seconds, cores, collect=gpu_out is not None)
    o = oracle_setup()
    out = {"value": round(v, 9), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
           "sample": f"{rows} causal A4Q query rows of the 16K workload (q heads 0-3) in {dt:.1f} s on "
                     f"{cores} threads; oracle append of all 16,384 tokens x 8 heads took {o['append_s']:.1f} s "
                     f"({o['append_gbs']:.3f} GB/s)"}
    if gpu_out is not None and res:
        g = gpu_out.numpy().astype(np.float64)
        d, r = [], []
        for pos, gq, ref in res:
            d.append(g[pos, gq, :] - ref)
            r.append(ref)
        d, r = np.concatenate(d), np.concatenate(r)
        out["parity_vs_kernel"] = {
            "rows": int(d.shape[0]), "kernel": "nvfp4_prefill_a4q_2cta_sm103_kernel (last timed step)",
            "max_abs_raw": round(float(np.abs(d).max()), 6),
            "max_abs_beyond_half_bf16_ulp": round(float(np.maximum(np.abs(d) - half_bf16_ulp(r), 0).max()), 6),
            "rel_fro": round(float(np.linalg.norm(d) / max(np.linalg.norm(r), 1e-30)), 7),
            "tolerance": {"max_abs": 2e-2, "rel_fro": 1e-2}}
    return out


def run_reference(args, rank, world):
    if rank != 0:
        return None
    cores = host_cores()
    per_step = min(args.cpu_seconds, 150.0 / (args.steps + args.warmup))
    oracle_setup()
    vals, times = [], []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        v, rows, dt, _ = oracle_rows(per_step, cores)
        if i >= args.warmup:
            vals.append(v)
            times.append(time.perf_counter() - t0)
    value = statistics.mean(vals)
    o = oracle_setup()
    desc = (f"each step: causal A4Q query rows of the 16K workload for {per_step:.1f} s on {cores} threads; "
            f"oracle append of the full cache took {o['append_s']:.1f} s")
    return {"impl": "reference", "metric": METRIC, "value": round(value, 9), "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(statistics.mean(times) * 1e3, 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": dict(bench_config(W.full_prefill_16k(), world), sample="bounded CPU sample per step"),
            "cpu_baseline": {"value": round(value, 9), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": round(value, 9), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# ---------------------------------------------------------------------------- ncu traffic
# DRAM read + write of one attention launch (nvfp4_prefill_a4q_2cta_sm103_kernel,
# 16K causal, 32/8 heads) from one ncu capture, keyed by a digest of the
# kernel's sources as captured: once they change the figure no longer
# describes the kernel and is reported as null.
PREFILL_TRAFFIC = {"sources": ["prefill_a4q.cu", "prefill_common.cuh", "kernels.cuh", "codec.cuh", "ptx.cuh"],
                   "sha256_16": "df2d22427fde6e94", "bytes": 183289344 + 89786880}


def prefill_sources_digest() -> str:
    import hashlib
    h = hashlib.sha256()
    for name in PREFILL_TRAFFIC["sources"]:
        with open(os.path.join(ROOT, "nvfp4_paged_kv_append_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def prefill_traffic_bytes():
    return PREFILL_TRAFFIC["bytes"] if prefill_sources_digest() == PREFILL_TRAFFIC["sha256_16"] else None


# ---------------------------------------------------------------------------- ranks
def max_over_ranks(ms: float, world: int, dev=None) -> float:
    """The step time of the job: the slowest rank's (MAX all-reduce; the
    tensor lives on the GPU under NCCL and on the CPU under gloo)."""
    if world <= 1:
        return ms
    on_gpu = torch.distributed.get_backend() == "nccl"
    t = torch.tensor([ms], dtype=torch.float64, device=dev if on_gpu else "cpu")
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(flops_per_rank_step: float, world: int, ms: float) -> float:
    """Replicas: every rank processes one full step of the workload, so the
    job does world x the FLOPs in the slowest rank's time."""
    return flops_per_rank_step * world / (ms * 1e-3) / 1e12


# ---------------------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="prefill16k", choices=sorted(W.CONFIGS))
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-accuracy", action="store_true", help="skip the A4Q accuracy report")
    ap.add_argument("--no-matrix", action="store_true", help="skip the other workloads' component timings")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    world = env_int("WORLD_SIZE", 1)
    rank = env_int("RANK", 0)
    local = env_int("LOCAL_RANK", 0)
    if args.impl == "reference":
        if world > 1:
            torch.distributed.init_process_group("gloo")
        res = run_reference(args, rank, world)
        if rank == 0:
            print(json.dumps(res), flush=True)
        if world > 1:
            torch.distributed.destroy_process_group()
        return
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=dev)
    from nvfp4_paged_kv_append_gb300 import build
    build.build()
    res = run_ours(args, rank, world, dev)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
