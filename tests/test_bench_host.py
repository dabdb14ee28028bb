"""The benchmark's accounting against closed forms, on the CPU: the work of
the 16K causal prefill, its tensor roofline, and the algorithmic bytes of
append and decode that the bandwidth fractions divide by ("NVFP4 KV cache
prefill vs decode performance", section "NVFP4 stores 4.5 bits per value
before padding": 64 code bytes and 8 scale bytes per 128-value row)."""
import math

import pytest

import bench
from nvfp4_paged_kv_append_gb300 import workloads as W

PEAKS = {"bf16_tflops": 1913.3, "hbm_gbs": 6653.3}


def test_causal_prefill_flops_16k():
    """Bottom-right causal with q_len = kv_len = n: query i sees i + 1 keys,
    n (n + 1) / 2 pairs per q head; QK and PV are 2 D flops per pair each."""
    wl = W.full_prefill_16k()
    n, d, hq = 16384, 128, 32
    pairs = n * (n + 1) // 2
    assert wl.visible_pairs() == pairs
    assert wl.flops() == 4 * d * pairs * hq == 2_199_157_473_280
    f_qk, f_pv = bench.prefill_flops_split(wl)
    assert f_qk == f_pv == wl.flops() / 2


def test_causal_prefill_flops_ragged_tails():
    """A tail of q tokens at the end of kv cached tokens: query i sees
    kv - q + 1 + i keys."""
    wl = W.Workload("t", [16, 3], [100, 7], 8, 2)
    expect = sum(sum(kv - q + 1 + i for i in range(q)) for q, kv in ((16, 100), (3, 7)))
    assert wl.visible_pairs() == expect
    assert wl.flops() == 4 * 128 * expect * 8


def test_prefill_roofline_mixed_precision():
    """A4Q: QK at the FP4 rate (6x bf16), PV at the bf16 rate; 670 us at 16K
    for a 1913.3 TFLOP/s bf16 peak."""
    wl = W.full_prefill_16k()
    half = wl.flops() / 2
    p16 = PEAKS["bf16_tflops"] * 1e12
    t = bench.prefill_roof_s(wl, PEAKS, True)
    assert t == pytest.approx(half / (6 * p16) + half / p16, rel=1e-12)
    assert t == pytest.approx(670.5e-6, rel=1e-3)
    assert bench.prefill_roof_s(wl, PEAKS, False) == pytest.approx(2 * half / p16, rel=1e-12)
    assert bench.prefill_roof_s(wl, PEAKS, "fp4") == pytest.approx(2 * half / (6 * p16), rel=1e-12)
    e = bench.tflops_entry([1.2], wl, PEAKS, True, "m")
    assert e["frac_of_roofline"] == pytest.approx(t / 1.2e-3, abs=1e-4)
    assert e["TFLOP/s"] == pytest.approx(wl.flops() / 1.2e-3 / 1e12, abs=0.01)


def test_cache_and_append_bytes():
    """Per (token, kv head): a cached row of K or V is 64 code bytes + 8 scale
    bytes (128 values at 4.5 bits); the append reads 256 bf16 bytes of each
    and writes its 72."""
    assert bench.CACHE_BYTES_PER_TOKEN_HEAD == 2 * (128 * 4.5 / 8)
    assert bench.APPEND_BYTES_PER_TOKEN_HEAD == 2 * (128 * 2) + bench.CACHE_BYTES_PER_TOKEN_HEAD
    assert bench.APPEND_BYTES_PER_TOKEN_HEAD * 16384 * 8 == 85_983_232
    wl = W.decode_batch()
    assert sum(wl.kv_lens) == 429_798
    assert bench.CACHE_BYTES_PER_TOKEN_HEAD * sum(wl.kv_lens) * wl.num_kv_heads == 495_127_296
    e = bench.gbs_entry([0.1], 495_127_296, PEAKS)
    assert e["GB/s"] == pytest.approx(495_127_296 / 1e-4 / 1e9, abs=0.1)
    assert e["frac_of_hbm"] == pytest.approx(e["GB/s"] / PEAKS["hbm_gbs"], abs=1e-4)
    assert math.isclose(bench.FP4_OVER_BF16, 6.0)


def test_fp4_issue_note():
    """At the measured M = 128 issue costs (68 cycles for FP4 K = 64 and for
    f16 K = 16) an FP4 instruction does 4x the f16 work; the headline's
    fraction at that ratio uses the same roofline form with 4 in place of 6."""
    wl = W.full_prefill_16k()
    note = bench.fp4_issue_note(wl, PEAKS, 1835.76)
    assert note["fp4_over_bf16_at_m128"] == 4.0
    half = wl.flops() / 2
    p16 = PEAKS["bf16_tflops"] * 1e12
    t4 = half / (4 * p16) + half / p16
    assert note["frac_at_that_ratio"] == pytest.approx(1835.76e12 / (wl.flops() / t4), abs=1e-4)
    assert note["frac_at_that_ratio"] > 1835.76e12 * bench.prefill_roof_s(wl, PEAKS) / wl.flops()
