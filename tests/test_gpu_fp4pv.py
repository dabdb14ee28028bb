"""The FP4 PV experiment on the GPU against the oracle's readings X1..X5: the
token-major V re-layout bit for bit, and the prefill variant (A4Q QK, FP4 P x
token-major FP4 V) within the attention tolerance of the oracle's FP4 PV
attention on the same codes.  The pages keep PV wide because the V block
scales run along the head dimension while PV reduces over tokens ("NVFP4 KV
cache A4Q prefill explained", sections "Why NVFP4 KV cache A4Q prefill
exists" and "Compare A4Q with dequantize-ahead repacking")."""
import numpy as np
import pytest
import torch

import oracle
from nvfp4_paged_kv_append_gb300 import workloads as W

from . import _gpu as G

pytestmark = pytest.mark.gpu


def oracle_token_major(pools, page_ids):
    """X1 page by page on the oracle's pools: the 16 slots decoded without
    the tensor scale, re-coded along tokens."""
    n, H, D = len(page_ids), pools.Hkv, pools.D
    codes = np.zeros((n, H, D, 8), np.uint8)
    scales = np.zeros((n, H, D), np.uint8)
    for i, p in enumerate(page_ids):
        for h in range(H):
            x = oracle.dequantize_rows(pools.v_data[p, h], pools.v_scale[p, h], g=1.0).astype(np.float32)
            codes[i, h], scales[i, h] = oracle.v_token_major_page(x)
    return codes, scales


@pytest.mark.parametrize("cfg", ["tiny", "small_ragged"])
def test_v_token_major_bit_exact(cfg):
    inp = G.inputs(cfg)
    cache = G.gpu_cache(inp, append_order=W.shuffled_append_order(inp.wl.total_kv))
    ids = torch.randperm(inp.num_pages, generator=torch.Generator().manual_seed(3)).to(torch.int32)
    b = G.nk()
    codes, scales = b.nvfp4_v_token_major(cache, ids.to(G.dev()))
    torch.cuda.synchronize()
    assert b.nvfp4kv_get_device_status() == 0
    want_c, want_s = oracle_token_major(G.pools_for(cfg), ids.tolist())
    np.testing.assert_array_equal(codes.cpu().numpy(), want_c)
    np.testing.assert_array_equal(scales.cpu().numpy(), want_s)


def test_v_token_major_bad_page_id():
    """An id outside the pool gives zero blocks and flags the device status."""
    inp = G.inputs("tiny")
    cache = G.gpu_cache(inp)
    b = G.nk()
    ids = torch.tensor([0, -1, inp.num_pages, 1], dtype=torch.int32, device=G.dev())
    codes, scales = b.nvfp4_v_token_major(cache, ids)
    torch.cuda.synchronize()
    assert b.nvfp4kv_get_device_status() == b.NVFP4KV_ERR_DEVICE_INDEX
    assert b.nvfp4kv_get_device_status() == 0  # reading the status clears it
    c = codes.cpu().numpy()
    assert not c[1].any() and not c[2].any() and not scales.cpu().numpy()[1:3].any()
    want_c, _ = oracle_token_major(G.pools_for("tiny"), [0, 1])
    np.testing.assert_array_equal(c[[0, 3]], want_c)


def run_fp4pv(inp, cache, causal=True):
    return G.run_prefill(inp, cache, G.nk().VARIANT_A4Q_FP4PV, causal=causal)


# P's codes are decisions taken on scores that the kernel computes in fp32
# (block-scaled MMA) and the oracle in fp64; the two differ by about 1e-5
# relative in p.  A decision within this relative distance of a rounding
# boundary may go either way, and the oracle's slack bounds what that moves.
SLACK_EPS = 2.0 ** -12


def oracle_fp4pv(pools, inp, causal=True, rows=None):
    return oracle.paged_attention(pools, inp.q.float().numpy(), inp.qo_indptr, inp.kv_lens, inp.page_table,
                                  inp.wl.num_q_heads, inp.k_global, inp.v_global, causal, inp.sm_scale,
                                  q_mode="a4q", rows=rows, pv="fp4", slack_eps=SLACK_EPS)


def _check(got, lse, status, ref, inp):
    assert status == 0
    mx, fro, n, raw, slack = G.compare_rows_slack(got, ref, inp.qo_indptr)
    assert mx <= G.MAX_ABS and fro <= G.REL_FRO, (mx, fro, n, raw, slack)
    assert G.compare_lse(lse, ref, inp.qo_indptr) <= 2e-3


@pytest.mark.parametrize("cfg", ["tiny", "small_ragged"])
def test_fp4pv_prefill_full_parity(cfg):
    inp = G.inputs(cfg)
    got, lse, status = run_fp4pv(inp, G.gpu_cache(inp))
    _check(got, lse, status, oracle_fp4pv(G.pools_for(cfg), inp), inp)


def test_fp4pv_prefill_groups_noncausal_junk():
    """G = 1, 8, 16, non-causal, pools filled with 0xFF outside the written
    slots (slots past kv_len of a last page must count as zeros in the
    token-major blocks)."""
    for group, hkv in [(1, 3), (8, 1), (16, 2)]:
        wl = W.Workload(f"fp4pv_nc_g{group}", [70, 3], [150, 41], group * hkv, hkv, causal=False, seed=group)
        inp = W.make_inputs(wl)
        got, lse, status = run_fp4pv(inp, G.gpu_cache(inp, fill=0xFF), causal=False)
        assert np.isfinite(got).all()
        _check(got, lse, status, oracle_fp4pv(G.oracle_pools(inp), inp, causal=False), inp)


@pytest.mark.parametrize("group", [32, 64, 128])
def test_fp4pv_prefill_wide_groups(group):
    """GQA ratios up to the largest the library accepts (128: one query token
    per 128-row q tile), causal, ragged, junk-filled pools; every row."""
    hkv = 2 if group == 32 else 1
    wl = W.Workload(f"fp4pv_wide_g{group}", [21, 5, 1], [40, 133, 1], group * hkv, hkv, seed=group)
    inp = W.make_inputs(wl)
    got, lse, status = run_fp4pv(inp, G.gpu_cache(inp, fill=0xFF))
    assert np.isfinite(got).all()
    _check(got, lse, status, oracle_fp4pv(G.oracle_pools(inp), inp), inp)


def test_fp4pv_prefill_shortq_sampled():
    """4 x 128 queries over 2,048 keys (the pages' repack case), sampled rows."""
    inp = G.inputs("shortq")
    rows = W.sample_rows(inp.wl, 6)
    got, lse, status = run_fp4pv(inp, G.gpu_cache(inp))
    _check(got, lse, status, oracle_fp4pv(G.pools_for("shortq"), inp, rows=rows), inp)


def test_fp4pv_prefill_16k_every_tile():
    """The 16K causal workload: one seeded row in every 128-row q tile."""
    inp = G.inputs("prefill16k")
    cache = G.gpu_cache(inp, append_order=W.shuffled_append_order(inp.wl.total_kv))
    rows = W.tile_rows(inp.wl)
    got, lse, status = run_fp4pv(inp, cache)
    _check(got, lse, status, oracle_fp4pv(G.pools_for("prefill16k"), inp, rows=rows), inp)


@pytest.mark.parametrize("cfg", ["tiny", "small_ragged"])
def test_fp4pv_error_against_wide_pv(cfg):
    """The experiment's accuracy cost, on the outlier workload and on normal
    values: against the exact attention on the unquantized values, FP4 PV is
    further off than the wide PV of the A4Q variant, by at most 0.15 in
    relative Frobenius norm (FP4 P has one mantissa bit; V is coded twice)."""
    inp = G.inputs(cfg)
    cache = G.gpu_cache(inp)
    b = G.nk()
    got4, _, s4 = run_fp4pv(inp, cache)
    got16, _, s16 = G.run_prefill(inp, cache, b.VARIANT_A4Q)
    assert s4 == 0 and s16 == 0
    rows = W.sample_rows(inp.wl, 24)
    exact = oracle.dense_attention(inp.q.float().numpy(), inp.qo_indptr, inp.k.float().numpy(),
                                   inp.v.float().numpy(), inp.kv_indptr, inp.wl.num_q_heads, True, inp.sm_scale, rows)
    _, fro4, _ = G.compare_rows(got4, exact, inp.qo_indptr)
    _, fro16, _ = G.compare_rows(got16, exact, inp.qo_indptr)
    assert fro16 < fro4 <= fro16 + 0.15, (fro16, fro4)


def test_fp4pv_needs_repack_workspace():
    """Without room for its records the variant is refused."""
    inp = G.inputs("tiny")
    cache = G.gpu_cache(inp)
    b = G.nk()
    d = G.dev()
    args = (inp.q.to(d), cache, inp.page_table.to(d), inp.kv_lens.to(d), inp.qo_indptr.to(d))
    with pytest.raises(b.NvFp4Error) as e:
        b.nvfp4_paged_prefill(*args, variant=b.VARIANT_A4Q_FP4PV, workspace=G.prefill_workspace(inp, "inkernel"))
    assert e.value.code == b.NVFP4KV_ERR_WORKSPACE
