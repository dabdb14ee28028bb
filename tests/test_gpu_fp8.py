"""The FP8 (E4M3) comparison cache on the GPU against the oracle: append
bytes bit for bit, prefill (BF16 query) and decode within max-abs 2e-2 and
relative Frobenius 1e-2 of the fp64 oracle on the same codes ("NVFP4 KV cache
A4Q prefill explained", section "Build the benchmark matrix": FP8 and the
NVFP4 paths on the same revision; "NVFP4 KV cache prefill vs decode
performance", section "A worked per-token cache estimate": one byte per
value)."""
import numpy as np
import pytest
import torch

from nvfp4_paged_kv_append_gb300 import workloads as W

from . import _gpu as G

pytestmark = pytest.mark.gpu

_FP8 = {}


def fp8_scales(inp):
    return W.fp8_scale(inp.k), W.fp8_scale(inp.v)


def gpu_fp8_cache(inp, fill=0, append_order=None):
    b = G.nk()
    ks, vs = fp8_scales(inp)
    c = b.Fp8Cache(inp.num_pages, inp.wl.num_kv_heads, ks, vs, device=G.dev(), fill=fill)
    k, v, s = inp.k, inp.v, inp.slot_mapping
    if append_order is not None:
        k, v, s = k[append_order], v[append_order], s[append_order]
    b.fp8_kv_append(k.contiguous().to(G.dev()), v.contiguous().to(G.dev()), s.contiguous().to(G.dev()), c)
    return c


def oracle_fp8_pools(inp, fill=0):
    ks, vs = fp8_scales(inp)
    pools = G.oracle.FP8Pools(inp.num_pages, inp.wl.num_kv_heads, fill=fill)
    G.oracle.fp8_kv_append(pools, inp.k.float().numpy(), inp.v.float().numpy(), inp.slot_mapping.numpy(), ks, vs)
    return pools


def fp8_pools_for(cfg):
    if cfg not in _FP8:
        _FP8[cfg] = oracle_fp8_pools(G.inputs(cfg))
    return _FP8[cfg]


def oracle_fp8_attention(pools, inp, causal=True, rows=None):
    ks, vs = fp8_scales(inp)
    return G.oracle.paged_attention(pools, inp.q.float().numpy(), inp.qo_indptr, inp.kv_lens, inp.page_table,
                                    inp.wl.num_q_heads, ks, vs, causal, inp.sm_scale, q_mode="bf16", rows=rows)


@pytest.mark.parametrize("cfg", ["tiny", "small_ragged", "shortq"])
def test_fp8_append_bit_exact(cfg):
    inp = G.inputs(cfg)
    cache = gpu_fp8_cache(inp, append_order=W.shuffled_append_order(inp.wl.total_kv))
    pools = fp8_pools_for(cfg)
    assert np.array_equal(cache.k_data.cpu().numpy(), pools.k_data)
    assert np.array_equal(cache.v_data.cpu().numpy(), pools.v_data)
    assert G.nk().nvfp4kv_get_device_status() == 0


def test_fp8_append_extremes_and_padding():
    """Saturation far above the scale, tiny negatives (signed zero), zero
    rows and skipped slots, bit for bit."""
    wl = W.Workload("fp8_edge", [1], [96], 2, 2, seed=13)
    inp = W.make_inputs(wl, with_q=False)
    k = inp.k.float()
    k[0] = 0.0
    k[1] *= 1e-30
    k[2, :, :16] = 3.0e4             # far above amax/448 of the rest: saturates at 448
    k[3, 0, 5] = -1e-3
    inp.k = k.to(torch.bfloat16)
    ks, vs = fp8_scales(W.make_inputs(wl, with_q=False))  # scales from the unmodified tensors
    slots = inp.slot_mapping.clone()
    slots[10:14] = -1
    inp.slot_mapping = slots
    b = G.nk()
    c = b.Fp8Cache(inp.num_pages, 2, ks, vs, device=G.dev())
    b.fp8_kv_append(inp.k.to(G.dev()), inp.v.to(G.dev()), slots.to(G.dev()), c)
    pools = G.oracle.FP8Pools(inp.num_pages, 2)
    G.oracle.fp8_kv_append(pools, inp.k.float().numpy(), inp.v.float().numpy(), slots.numpy(), ks, vs)
    assert np.array_equal(c.k_data.cpu().numpy(), pools.k_data)
    assert np.array_equal(c.v_data.cpu().numpy(), pools.v_data)


def test_fp8_append_full_16k():
    inp = G.inputs("prefill16k")
    cache = gpu_fp8_cache(inp, append_order=W.shuffled_append_order(inp.wl.total_kv))
    pools = fp8_pools_for("prefill16k")
    assert np.array_equal(cache.k_data.cpu().numpy(), pools.k_data)
    assert np.array_equal(cache.v_data.cpu().numpy(), pools.v_data)


def _prefill(inp, cache, causal=True):
    b = G.nk()
    d = G.dev()
    lse = torch.full((inp.wl.total_q, inp.wl.num_q_heads), float("nan"), device=d)
    o = b.fp8_paged_prefill(inp.q.to(d), cache, inp.page_table.to(d), inp.kv_lens.to(d), inp.qo_indptr.to(d),
                            causal=causal, sm_scale=inp.sm_scale, lse=lse)
    torch.cuda.synchronize()
    assert b.nvfp4kv_get_device_status() == 0
    return o.float().cpu().numpy(), lse.cpu().numpy()


def _check(got, lse, ref, inp):
    mx, fro, n = G.compare_rows(got, ref, inp.qo_indptr)
    assert mx <= G.MAX_ABS and fro <= G.REL_FRO, (mx, fro, n)
    assert G.compare_lse(lse, ref, inp.qo_indptr) <= 2e-3


@pytest.mark.parametrize("cfg", ["tiny", "small_ragged"])
def test_fp8_prefill_full_parity(cfg):
    inp = G.inputs(cfg)
    got, lse = _prefill(inp, gpu_fp8_cache(inp))
    _check(got, lse, oracle_fp8_attention(fp8_pools_for(cfg), inp), inp)


def test_fp8_prefill_groups_noncausal_junk():
    """G = 1, 8, 16, non-causal, pools filled with 0x7F (an E4M3 NaN) outside
    the written slots: nothing unwritten may reach the output."""
    for group, hkv in [(1, 3), (8, 1), (16, 2)]:
        wl = W.Workload(f"fp8_nc_g{group}", [70, 3], [150, 40], group * hkv, hkv, causal=False, seed=group)
        inp = W.make_inputs(wl)
        got, lse = _prefill(inp, gpu_fp8_cache(inp, fill=0x7F), causal=False)
        assert np.isfinite(got).all()
        _check(got, lse, oracle_fp8_attention(oracle_fp8_pools(inp), inp, causal=False), inp)


def test_fp8_prefill_16k_every_tile():
    """The 16K causal workload: one seeded row in every 128-row q tile."""
    inp = G.inputs("prefill16k")
    cache = gpu_fp8_cache(inp, append_order=W.shuffled_append_order(inp.wl.total_kv))
    rows = W.tile_rows(inp.wl)
    got, lse = _prefill(inp, cache)
    _check(got, lse, oracle_fp8_attention(fp8_pools_for("prefill16k"), inp, rows=rows), inp)


def _decode(wl, fill=0, sample=None):
    inp = W.make_inputs(wl)
    b = G.nk()
    cache = gpu_fp8_cache(inp, fill=fill)
    lse = torch.full((wl.batch, wl.num_q_heads), float("nan"), device=G.dev())
    o = b.fp8_paged_decode(inp.q.to(G.dev()), cache, inp.page_table.to(G.dev()), inp.kv_lens.to(G.dev()),
                           sm_scale=inp.sm_scale, lse=lse)
    torch.cuda.synchronize()
    assert b.nvfp4kv_get_device_status() == 0
    reqs = range(wl.batch) if sample is None else sample
    rows = [(r, 0) for r in reqs if wl.kv_lens[r] > 0]
    ref = oracle_fp8_attention(oracle_fp8_pools(inp), inp, causal=False, rows=rows)
    got = o.float().cpu().numpy()
    mx, fro, _ = G.compare_rows(got, ref, inp.qo_indptr)
    return mx, fro, G.compare_lse(lse.cpu().numpy(), ref, inp.qo_indptr), got


@pytest.mark.parametrize("group", [1, 2, 4, 8, 16])
def test_fp8_decode_groups(group):
    wl = W.Workload(f"fp8_dec_g{group}", [1] * 5, [1, 17, 128, 129, 700], 2 * group, 2, seed=group)
    mx, fro, lerr, _ = _decode(wl)
    assert mx <= G.MAX_ABS and fro <= G.REL_FRO, (mx, fro)
    assert lerr <= 1e-3, lerr


def test_fp8_decode_junk_pool_and_splits():
    """Unwritten pool bytes are 0x7F (an E4M3 NaN); lengths cross the unit and
    split boundaries."""
    wl = W.Workload("fp8_dec_junk", [1] * 4, [33, 1025, 2049, 3000], 8, 2, dist="outliers", seed=4)
    mx, fro, lerr, got = _decode(wl, fill=0x7F)
    assert np.isfinite(got).all()
    assert mx <= G.MAX_ABS and fro <= G.REL_FRO, (mx, fro)


def test_fp8_decode_full_size_all_requests():
    """The batch-32 decode workload (kv_len ~ U[1K, 32K], 32/8 heads), every
    request against the oracle."""
    mx, fro, lerr, _ = _decode(W.decode_batch())
    assert mx <= G.MAX_ABS and fro <= G.REL_FRO, (mx, fro)
    assert lerr <= 1e-3


def test_fp8_prefill_split_kv():
    """FP8 prefill with few units over long KV (the KV range is split and
    merged): every row against the oracle."""
    wl = W.Workload("fp8_split", [5, 40], [3000, 2500], 8, 2, seed=23)
    inp = W.make_inputs(wl)
    got, lse = _prefill(inp, gpu_fp8_cache(inp, fill=0x7F))
    _check(got, lse, oracle_fp8_attention(oracle_fp8_pools(inp), inp), inp)
