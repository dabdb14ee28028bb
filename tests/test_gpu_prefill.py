"""Paged prefill on the GPU against the oracle.  A4Q is compared with the
oracle's A4Q query (same per-row quantization), the dequant-ahead variant with
the BF16 query; max-abs <= 2e-2 and relative Frobenius <= 1e-2 ("NVFP4 KV
cache A4Q prefill explained", sections "Quantize Q instead of expanding K",
"Compare A4Q with dequantize-ahead repacking", "Make query accuracy a release
gate")."""
import numpy as np
import pytest
import torch

from nvfp4_paged_kv_append_gb300 import workloads as W

from . import _gpu as G

pytestmark = pytest.mark.gpu

VARIANTS = [(0, "a4q"), (1, "bf16")]


def _check(inp, cache, pools, variant, q_mode, causal=True, rows=None, mode="auto", ref=None):
    got, lse, status = G.run_prefill(inp, cache, variant, causal=causal, mode=mode)
    assert status == 0
    if ref is None:
        ref = G.oracle_prefill(pools, inp, q_mode, causal=causal, rows=rows)
    mx, fro, n = G.compare_rows(got, ref, inp.qo_indptr)
    lerr = G.compare_lse(lse, ref, inp.qo_indptr)
    assert mx <= G.MAX_ABS and fro <= G.REL_FRO, (mx, fro, n)
    assert lerr <= 2e-3, lerr
    return got, ref


@pytest.mark.parametrize("mode", ["auto", "inkernel"])
@pytest.mark.parametrize("variant,q_mode", VARIANTS)
@pytest.mark.parametrize("cfg", ["tiny", "small_ragged"])
def test_prefill_full_parity(cfg, variant, q_mode, mode):
    """Every row; "auto" runs the repack pre-pass for dequant-ahead (these
    batches average two or more q tiles per kv head) and the in-kernel mode
    for A4Q (fewer than eight), "inkernel" dequantizes V in the kernel."""
    inp = G.inputs(cfg)
    cache = G.gpu_cache(inp)
    _check(inp, cache, G.pools_for(cfg), variant, q_mode, mode=mode)


@pytest.mark.parametrize("variant,q_mode", VARIANTS)
def test_prefill_noncausal_and_groups(variant, q_mode):
    for group, hkv in [(1, 3), (8, 1), (16, 2)]:
        wl = W.Workload(f"nc_g{group}", [70, 3], [150, 40], group * hkv, hkv, causal=False, seed=group)
        inp = W.make_inputs(wl)
        cache = G.gpu_cache(inp, fill=0x7F)   # junk in unused slots must not leak
        _check(inp, cache, G.oracle_pools(inp), variant, q_mode, causal=False)


@pytest.mark.parametrize("variant,q_mode", VARIANTS)
def test_prefill_zero_length_and_edge_rows(variant, q_mode):
    """A request with q_len 0, one with q_len 1 over a long cache, a zero
    query row, kv_len not a multiple of the page or tile size."""
    wl = W.Workload("edge", [0, 1, 129, 5], [0, 300, 129, 1000], 4, 2, seed=6)
    inp = W.make_inputs(wl)
    q = inp.q.clone()
    q[3] = 0
    inp.q = q
    cache = G.gpu_cache(inp, fill=0x7F)
    _check(inp, cache, G.oracle_pools(inp), variant, q_mode)


@pytest.mark.parametrize("mode", ["auto", "inkernel"])
@pytest.mark.parametrize("variant,q_mode", VARIANTS)
def test_prefill_shortq_longkv(variant, q_mode, mode):
    """batch 4, q 128 at the end of kv 2048, 32/8 heads, permuted pages: all
    rows of request 0 and one row of every 128-row q tile of the others."""
    inp = G.inputs("shortq")
    cache = G.gpu_cache(inp)
    rows = sorted(set([(0, i) for i in range(128)] + W.tile_rows(inp.wl)))
    ref = G.oracle_prefill_cached("shortq", q_mode, rows)
    _check(inp, cache, None, variant, q_mode, mode=mode, ref=ref)


@pytest.mark.parametrize("variant,q_mode", VARIANTS)
def test_prefill_tails(variant, q_mode):
    """8 requests x 16 new queries over 16,400 cached tokens (sampled rows)."""
    inp = G.inputs("tails")
    cache = G.gpu_cache(inp)
    rows = [(b, i) for b in (0, 7) for i in range(16)] + W.sample_rows(inp.wl, 2)
    _check(inp, cache, G.pools_for("tails"), variant, q_mode, rows=rows)


@pytest.mark.parametrize("mode", ["auto", "inkernel"])
@pytest.mark.parametrize("variant,q_mode", VARIANTS)
def test_prefill_full_16k_sampled(variant, q_mode, mode):
    """The 16K causal configuration at full size, as the benchmark runs it
    (cache built by the CUDA append in shuffled order).  One seeded query
    position inside every 128-row q tile (32 tokens x 4 grouped heads), so
    every (q tile, kv head) work item of the schedule is checked: 512
    positions x 32 heads."""
    inp = G.inputs("prefill16k")
    cache = G.gpu_cache(inp, append_order=W.shuffled_append_order(inp.wl.total_kv))
    rows = W.tile_rows(inp.wl)
    assert len({(b, i // 32) for b, i in rows}) == 16384 // 32
    ref = G.oracle_prefill_cached("prefill16k", q_mode, rows)
    _check(inp, cache, None, variant, q_mode, mode=mode, ref=ref)


@pytest.mark.parametrize("variant,q_mode", VARIANTS)
def test_prefill_long_ragged_every_tile(variant, q_mode):
    """32,768 + 7,001 tokens in one batch, 64/8 heads (16 tokens per 128-row
    q tile): one seeded query position in every q tile of both requests,
    both variants (repack mode)."""
    inp = G.inputs("prefill32k")
    cache = G.gpu_cache(inp)
    rows = W.tile_rows(inp.wl)
    tiles = {(b, i // 16) for b, i in rows}
    assert len(tiles) == 32768 // 16 + (7001 + 15) // 16
    ref = G.oracle_prefill_cached("prefill32k", q_mode, rows)
    _check(inp, cache, None, variant, q_mode, ref=ref)


@pytest.mark.parametrize("mode", ["auto", "inkernel"])
@pytest.mark.parametrize("variant,q_mode", VARIANTS)
def test_prefill_group1_repack(variant, q_mode, mode):
    """One query head per kv head (G = 1): 128 tokens per q tile.  Two
    requests average eight and a half q tiles per kv head, so "auto" runs the
    repack-mode kernels (the two-CTA kernel for A4Q); every row is checked."""
    wl = W.Workload("g1_repack", [1100, 1000], [1200, 1000], 3, 3, seed=17)
    assert G.repack_mode_expected(wl, variant)
    inp = W.make_inputs(wl)
    cache = G.gpu_cache(inp, fill=0x7F)
    _check(inp, cache, G.oracle_pools(inp), variant, q_mode, mode=mode)


@pytest.mark.parametrize("variant,q_mode", VARIANTS)
def test_prefill_many_short_items(variant, q_mode):
    """120 requests of 128 queries over 128-240 keys, 32/4 heads (16 tokens
    per q tile, eight q tiles per kv head): 3,840 work items of one to three
    KV tiles, about 12 per CTA of the two-CTA kernel, in repack mode.  Each
    CTA stages the Q tile of its next item while it runs the current one (two
    Q buffers, reused every other item; an item of one tile releases its
    buffer at its first QK); every row is checked."""
    rng = np.random.default_rng(23)
    kv = [int(x) for x in rng.integers(128, 241, size=120)]
    wl = W.Workload("many_short", [128] * 120, kv, 32, 4, seed=23)
    assert G.repack_mode_expected(wl, variant)
    inp = W.make_inputs(wl)
    cache = G.gpu_cache(inp, fill=0x7F)
    _check(inp, cache, G.oracle_pools(inp), variant, q_mode)


@pytest.mark.parametrize("mode", ["auto", "inkernel"])
@pytest.mark.parametrize("variant,q_mode", VARIANTS)
@pytest.mark.parametrize("group", [32, 64, 128])
def test_prefill_wide_groups(group, variant, q_mode, mode):
    """GQA ratios up to the largest the library accepts (128: one query token
    per 128-row q tile), causal, ragged; every row against the oracle.  The
    requests average eight or more q tiles per kv head, so "auto" runs repack
    mode (the two-CTA kernel for A4Q)."""
    hkv = 2 if group == 32 else 1
    wl = W.Workload(f"wide_g{group}", [80, 20, 1], [100, 133, 1], group * hkv, hkv, seed=group)
    assert G.repack_mode_expected(wl, variant)
    inp = W.make_inputs(wl)
    cache = G.gpu_cache(inp, fill=0x7F)
    _check(inp, cache, G.oracle_pools(inp), variant, q_mode, mode=mode)


def test_a4q_is_closer_to_its_own_reference():
    """The A4Q kernel really quantizes Q: its output is nearer the oracle's A4Q
    result than the BF16-query result, and the gap between the two oracle
    results (the A4Q error) is reported."""
    inp = G.inputs("tiny")
    cache = G.gpu_cache(inp)
    pools = G.pools_for("tiny")
    got, _, _ = G.run_prefill(inp, cache, 0)
    ra = G.oracle_prefill(pools, inp, "a4q")
    rb = G.oracle_prefill(pools, inp, "bf16")
    to_a, _, _ = G.compare_rows(got, ra, inp.qo_indptr)
    to_b, _, _ = G.compare_rows(got, rb, inp.qo_indptr)
    a4q_err = max(float(np.abs(ra[k][0] - rb[k][0]).max()) for k in ra)
    print(f"A4Q vs BF16-Q max-abs error (oracle): {a4q_err:.4g}; kernel to A4Q ref {to_a:.3g}, to BF16 ref {to_b:.3g}")
    assert to_a < to_b


def test_prefill_bad_page_and_shape_flagged():
    b = G.nk()
    inp = W.make_inputs(W.Workload("bad", [20], [40], 4, 2, seed=3))
    cache = G.gpu_cache(inp)
    pt = inp.page_table.clone()
    pt[0, 1] = inp.num_pages + 100                 # out of range: skipped + flagged
    o = b.nvfp4_paged_prefill(inp.q.to(G.dev()), cache, pt.to(G.dev()), inp.kv_lens.to(G.dev()),
                              inp.qo_indptr.to(G.dev()), sm_scale=inp.sm_scale)
    torch.cuda.synchronize()
    assert b.nvfp4kv_get_device_status() == -6
    assert torch.isfinite(o.float()).all()
    kvl = inp.kv_lens.clone()
    kvl[0] = 10                                     # causal with q_len 20 > kv_len 10
    b.nvfp4_paged_prefill(inp.q.to(G.dev()), cache, inp.page_table.to(G.dev()), kvl.to(G.dev()),
                          inp.qo_indptr.to(G.dev()), sm_scale=inp.sm_scale)
    torch.cuda.synchronize()
    assert b.nvfp4kv_get_device_status() == -2


@pytest.mark.parametrize("mode", ["auto", "inkernel"])
@pytest.mark.parametrize("variant", [0, 1])
def test_plan_then_run_equals_single_call(variant, mode):
    """nvfp4_paged_prefill_plan + nvfp4_paged_prefill_run produce the same bytes
    as nvfp4_paged_prefill, in repack and in-kernel mode, and a plan can be
    reused by several runs over the same cache."""
    b = G.nk()
    inp = G.inputs("shortq")
    cache = G.gpu_cache(inp)
    d = G.dev()
    q, pt, kvl, qo = inp.q.to(d), inp.page_table.to(d), inp.kv_lens.to(d), inp.qo_indptr.to(d)
    ws = G.prefill_workspace(inp, mode)
    ref = b.nvfp4_paged_prefill(q, cache, pt, kvl, qo, sm_scale=inp.sm_scale, variant=variant, workspace=ws)
    ws2 = G.prefill_workspace(inp, mode)
    b.nvfp4_paged_prefill_plan(cache, inp.wl.total_q, inp.wl.num_q_heads, pt, kvl, qo, ws2, variant=variant)
    for _ in range(2):
        got = b.nvfp4_paged_prefill_run(q, cache, pt, kvl, qo, ws2, sm_scale=inp.sm_scale, variant=variant)
        torch.cuda.synchronize()
        assert b.nvfp4kv_get_device_status() == 0
        assert torch.equal(got.view(torch.int16), ref.view(torch.int16))


@pytest.mark.parametrize("variant,q_mode", VARIANTS)
def test_prefill_zero_query_rows_repack_mode(variant, q_mode):
    """All-zero query rows (a per-row Q scale of 0) in repack mode, on the
    causal diagonal tiles where keys are masked: the output is the mean of
    the visible V rows, never NaN."""
    wl = W.Workload("zero_rows_repack", [256, 256], [2048, 1024], 32, 8, seed=31)
    assert G.repack_mode_expected(wl, variant)  # eight q tiles per kv head
    inp = W.make_inputs(wl)
    zero_tokens = [0, 5, 127, 256 + 64, 256 + 255]
    inp.q[zero_tokens] = 0
    cache = G.gpu_cache(inp)
    rows = [(0, i) for i in range(128)] + [(1, 64), (1, 255), (0, 200), (0, 255)]
    got, _ = _check(inp, cache, G.oracle_pools(inp), variant, q_mode, rows=rows, mode="auto")
    assert np.isfinite(got).all()


@pytest.mark.parametrize("mode", ["auto", "inkernel"])
@pytest.mark.parametrize("scheme", ["per_tensor", "single_level"])
@pytest.mark.parametrize("cfg", ["tiny", "shortq"])
def test_prefill_query_scale_schemes(cfg, scheme, mode):
    """The A4Q query with one scale for every row (q_global_scale > 0): a
    per-tensor dual-level scale fl32(amax(Q)/2688), or 1 (single level), in
    both kernel modes, against the oracle's query coded with the same scale
    ("NVFP4 KV cache A4Q prefill explained", section "Make query accuracy a
    release gate": the scheme is a recorded choice)."""
    b = G.nk()
    inp = G.inputs(cfg)
    qf = inp.q.float().numpy()
    g = float(np.float32(np.float32(np.abs(qf).max()) / np.float32(2688.0))) if scheme == "per_tensor" else 1.0
    cache = G.gpu_cache(inp)
    d = G.dev()
    lse = torch.empty(inp.wl.total_q, inp.wl.num_q_heads, device=d)
    o = b.nvfp4_paged_prefill(inp.q.to(d), cache, inp.page_table.to(d), inp.kv_lens.to(d), inp.qo_indptr.to(d),
                              sm_scale=inp.sm_scale, variant=0, lse=lse, workspace=G.prefill_workspace(inp, mode),
                              q_global_scale=g)
    torch.cuda.synchronize()
    assert b.nvfp4kv_get_device_status() == 0
    rows = None if cfg == "tiny" else W.tile_rows(inp.wl)
    ref = G.oracle.paged_attention(G.pools_for(cfg), qf, inp.qo_indptr, inp.kv_lens, inp.page_table,
                                   inp.wl.num_q_heads, inp.k_global, inp.v_global, True, inp.sm_scale,
                                   q_mode="a4q", rows=rows, q_scale=g)
    mx, fro, n = G.compare_rows(o.float().cpu().numpy(), ref, inp.qo_indptr)
    assert mx <= G.MAX_ABS and fro <= G.REL_FRO, (mx, fro, n)
    assert G.compare_lse(lse.cpu().numpy(), ref, inp.qo_indptr) <= 2e-3


SPLIT_CASES = [
    # (name, q_lens, kv_lens, Hq, Hkv, causal): fewer (request, q tile, kv
    # head) units than the kernel's CTAs, long KV: the KV range is split
    ("split_g4_causal", [5, 40], [3000, 2500], 8, 2, True),
    ("split_g1_noncausal", [3, 17], [1800, 2200], 2, 2, False),
    ("split_g16_causal", [2, 9], [2600, 1500], 32, 2, True),
    ("split_g4_repack", [300, 260], [2600, 2300], 8, 2, True),   # repack mode (>= 2 q tiles per kv head)
]


@pytest.mark.parametrize("variant,q_mode", VARIANTS)
@pytest.mark.parametrize("case", SPLIT_CASES, ids=[c[0] for c in SPLIT_CASES])
def test_prefill_split_kv(case, variant, q_mode):
    """Few work units over long KV ranges: with room in the workspace each
    unit's KV range is cut into parts merged by log-sum-exp; every row
    against the oracle, and the same rows without the split (schedule-only
    workspace) agree with it too."""
    name, ql, kl, hq, hkv, causal = case
    inp = W.make_inputs(W.Workload(name, ql, kl, hq, hkv, causal=causal, seed=len(name)))
    cache = G.gpu_cache(inp, fill=0x7F)
    pools = G.oracle_pools(inp)
    ref = G.oracle_prefill(pools, inp, q_mode, causal=causal)
    _check(inp, cache, pools, variant, q_mode, causal=causal, mode="auto", ref=ref)
    _check(inp, cache, pools, variant, q_mode, causal=causal, mode="inkernel", ref=ref)
