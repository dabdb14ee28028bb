#!/usr/bin/env python3
"""Benchmark of the NVFP4 paged-KV hot path on one GB300 (or N replicas).

A step is one pass of the path over the 16K-token causal prefill workload:
append the 16,384 tokens' K and V (8 kv heads, shuffled slot order) into the
NVFP4 cache, then run the A4Q paged prefill (32 q heads) over it.  The
headline value is prefill TFLOP/s per step (4*D FLOPs per visible causal
(query, key) pair per q head).  The same run also reports append GB/s, A4Q
prefill alone, the dequant-ahead variant, and paged decode GB/s on the batch-32
decode workload (kv_len ~ U[1K, 32K]).

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


def setup_prefill(nk, dev, wl):
    inp = W.make_inputs(wl)
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
    wl = W.CONFIGS[args.config]()
    P = setup_prefill(nk, dev, wl)
    inp = P["inp"]

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

    # ---- components (each timed alone, L2 flushed before every call)
    K = max(min(args.steps, 50), 5)
    app = nk_bench.time_fn(append, K, 3)
    app_g = time_graph(nk_bench, append, K)
    pre = nk_bench.time_fn(prefill, K, 3)
    dqa = nk_bench.time_fn(lambda: prefill(nk.VARIANT_DQ_AHEAD), K, 3)
    pre_ik = nk_bench.time_fn(lambda: prefill(nk.VARIANT_A4Q, "ws_min"), K, 3)
    dqa_ik = nk_bench.time_fn(lambda: prefill(nk.VARIANT_DQ_AHEAD, "ws_min"), K, 3)
    app_bytes = APPEND_BYTES_PER_TOKEN_HEAD * wl.total_kv * wl.num_kv_heads
    dec = decode_component(nk, nk_bench, dev, K)
    clk = clocks.stop()

    pre_avg = statistics.mean(pre)
    # the dominant kernel: the attention launch, timed inside the timed steps
    achieved = flops / (statistics.mean(attn_ms) * 1e-3) / 1e12
    p16 = peaks["bf16_tflops"]
    t_roof = f_qk / (p16 * FP4_OVER_BF16 * 1e12) + f_pv / (p16 * 1e12)
    peak_eff = flops / t_roof / 1e12

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
                                   f"({peaks['source']} burst)"},
        "components": {
            "append": {"ms": round(statistics.mean(app), 4),
                       "GB/s": round(app_bytes / (statistics.mean(app) * 1e-3) / 1e9, 1),
                       "frac_of_hbm": round(app_bytes / (statistics.mean(app) * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
                       "graph_ms": round(statistics.mean(app_g), 4) if app_g else None,
                       "graph_GB/s": round(app_bytes / (statistics.mean(app_g) * 1e-3) / 1e9, 1) if app_g else None,
                       "graph_frac_of_hbm": round(app_bytes / (statistics.mean(app_g) * 1e-3) / 1e9 / peaks["hbm_gbs"], 4)
                       if app_g else None,
                       "bytes": app_bytes},
            "prefill_a4q": {"ms": round(pre_avg, 4), "TFLOP/s": round(flops / (pre_avg * 1e-3) / 1e12, 2),
                            "mode": "V repacked once per KV tile"},
            "prefill_a4q_inkernel": {"ms": round(statistics.mean(pre_ik), 4),
                                     "TFLOP/s": round(flops / (statistics.mean(pre_ik) * 1e-3) / 1e12, 2),
                                     "mode": "V dequantized in the kernel"},
            "prefill_dq_ahead": {"ms": round(statistics.mean(dqa), 4),
                                 "TFLOP/s": round(flops / (statistics.mean(dqa) * 1e-3) / 1e12, 2),
                                 "frac_of_bf16": round(flops / (statistics.mean(dqa) * 1e-3) / 1e12 / p16, 4),
                                 "mode": "K and V repacked once per KV tile"},
            "prefill_dq_ahead_inkernel": {"ms": round(statistics.mean(dqa_ik), 4),
                                          "TFLOP/s": round(flops / (statistics.mean(dqa_ik) * 1e-3) / 1e12, 2)},
            "decode": dec,
        },
        "e2e": e2e,
        "gpu_launches": 4 * args.steps,  # append, schedule, repack pre-pass, attention
        "clocks": clk,
        "wall_s_timed_loop": round(t_wall, 3),
    }
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
    return result


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
    peaks = measured_peaks()
    bytes_ = CACHE_BYTES_PER_TOKEN_HEAD * wl.total_kv * wl.num_kv_heads
    gbs = bytes_ / (statistics.mean(t) * 1e-3) / 1e9
    out = {"workload": wl.name, "ms": round(statistics.mean(t), 4), "GB/s": round(gbs, 1),
           "frac_of_hbm": round(gbs / peaks["hbm_gbs"], 4), "bytes": bytes_}
    if tg:
        g = bytes_ / (statistics.mean(tg) * 1e-3) / 1e9
        out.update({"graph_ms": round(statistics.mean(tg), 4), "graph_GB/s": round(g, 1),
                    "graph_frac_of_hbm": round(g / peaks["hbm_gbs"], 4)})
    return out


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
                        append_gbs=APPEND_BYTES_PER_TOKEN_HEAD * wl.total_kv * wl.num_kv_heads / t_app / 1e9,
                        rng=np.random.default_rng(0)))
    return _ORACLE


def oracle_rows(seconds: float):
    """The oracle as it stands: A4Q attention for seeded query rows of the
    four q heads of kv head 0 until `seconds` have passed.  Returns
    (TFLOP/s, rows, seconds)."""
    import oracle
    o = oracle_setup()
    wl, inp = o["wl"], o["inp"]
    flops, rows = 0.0, 0
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < seconds:
        pos = np.sort(o["rng"].integers(0, wl.q_lens[0], 8)).astype(np.int32)
        for gq in range(wl.group):
            qd = oracle.decode_q_a4q(o["q"][pos, gq, :])
            oracle.attention_rows(qd, pos, wl.q_lens[0], o["kd"], o["vd"], True, inp.sm_scale)
            flops += float(np.sum(4.0 * 128 * (pos.astype(np.float64) + 1)))
            rows += len(pos)
    dt = time.perf_counter() - t0
    return flops / dt / 1e12, rows, dt


def cpu_baseline(seconds):
    v, rows, dt = oracle_rows(seconds)
    o = oracle_setup()
    return {"value": round(v, 9), "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
            "sample": f"{rows} causal A4Q query rows of the 16K workload (q heads 0-3) in {dt:.1f} s; "
                      f"oracle append of all 16,384 tokens x 8 heads took {o['append_s']:.1f} s "
                      f"({o['append_gbs']:.3f} GB/s)"}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    per_step = min(args.cpu_seconds, 150.0 / (args.steps + args.warmup))
    oracle_setup()
    vals, times = [], []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        v, rows, dt = oracle_rows(per_step)
        if i >= args.warmup:
            vals.append(v)
            times.append(time.perf_counter() - t0)
    value = statistics.mean(vals)
    o = oracle_setup()
    desc = (f"each step: causal A4Q query rows of the 16K workload for {per_step:.1f} s on one core; "
            f"oracle append of the full cache took {o['append_s']:.1f} s")
    return {"impl": "reference", "metric": METRIC, "value": round(value, 9), "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(statistics.mean(times) * 1e3, 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": dict(bench_config(W.full_prefill_16k(), world), sample="bounded CPU sample per step"),
            "cpu_baseline": {"value": round(value, 9), "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": round(value, 9), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# ---------------------------------------------------------------------------- ncu traffic
# DRAM read + write of one attention launch (nvfp4_prefill_a4q_2cta_sm103_kernel,
# 16K causal, 32/8 heads) from the ncu capture summarised in
# profiles/prefill_a4q_16k_ncu.md, keyed by the digest of the kernel source it
# was taken on: once that source changes the figure no longer describes the
# kernel and is reported as null.
PREFILL_TRAFFIC = {"source": "prefill_a4q.cu", "sha256_16": "9d235b9533aab863", "bytes": 184646400 + 95481344}


def prefill_traffic_bytes():
    import hashlib
    src = os.path.join(ROOT, "nvfp4_paged_kv_append_gb300", "csrc", PREFILL_TRAFFIC["source"])
    with open(src, "rb") as f:
        dig = hashlib.sha256(f.read()).hexdigest()[:16]
    return PREFILL_TRAFFIC["bytes"] if dig == PREFILL_TRAFFIC["sha256_16"] else None


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
