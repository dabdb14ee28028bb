"""Cache append on the GPU against the oracle: packed codes and scale bytes
must match bit for bit ("NVFP4 KV cache prefill vs decode performance",
section "NVFP4 stores 4.5 bits per value before padding")."""
import numpy as np
import pytest
import torch

from nvfp4_paged_kv_append_gb300 import workloads as W

from . import _gpu as G

pytestmark = pytest.mark.gpu


def _assert_same(cache, pools):
    for name in ("k_data", "k_scale", "v_data", "v_scale"):
        got = getattr(cache, name).cpu().numpy()
        ref = getattr(pools, name)
        bad = np.argwhere(got != ref)
        assert bad.size == 0, f"{name}: {len(bad)} bytes differ, first at {bad[:3].tolist()}"


@pytest.mark.parametrize("cfg", ["tiny", "small_ragged", "shortq"])
def test_append_bit_exact(cfg):
    inp = G.inputs(cfg)
    order = W.shuffled_append_order(inp.wl.total_kv)
    cache = G.gpu_cache(inp, append_order=order)
    _assert_same(cache, G.pools_for(cfg))
    assert G.nk().nvfp4kv_get_device_status() == 0


def test_append_bit_exact_full_16k():
    """The 16K-token configuration at full size, tokens appended in shuffled order."""
    inp = G.inputs("prefill16k")
    cache = G.gpu_cache(inp, append_order=W.shuffled_append_order(inp.wl.total_kv))
    _assert_same(cache, G.pools_for("prefill16k"))


def test_append_sampled_full_40k():
    """32,768 + 7,001 tokens, 8 kv heads: every token on the GPU; the oracle
    writes a seeded sample of 3,000 tokens and those slots are compared."""
    inp = W.make_inputs(W.long_prefill_ragged(), with_q=False)
    cache = G.gpu_cache(inp)
    idx = torch.randperm(inp.wl.total_kv, generator=torch.Generator().manual_seed(3))[:3000].numpy()
    pools = G.oracle_pools(inp, token_subset=idx)
    slots = inp.slot_mapping.numpy()[idx]
    for name in ("k_data", "k_scale", "v_data", "v_scale"):
        got = getattr(cache, name).cpu().numpy()
        ref = getattr(pools, name)
        p, o = slots // 16, slots % 16
        assert np.array_equal(got[p, :, o], ref[p, :, o]), name


def test_append_extremes_and_padding():
    """Outlier-heavy and tiny-magnitude rows, zero rows, and skipped slots."""
    wl = W.Workload("edge", [1], [96], 2, 2, seed=13)
    inp = W.make_inputs(wl, with_q=False)
    k = inp.k.float()
    k[0] = 0.0                                   # an all-zero token
    k[1] *= 1e-30                                # scales in the E4M3 subnormal range or zero
    k[2, :, :16] = 3.0e4                          # a block far above the others
    k[3, 0, 5] = -1e-3                            # small negative entries
    inp.k = k.to(torch.bfloat16)
    slots = inp.slot_mapping.clone()
    slots[10:14] = -1                            # padding tokens are skipped
    inp.slot_mapping = slots
    cache = G.gpu_cache(inp)
    _assert_same(cache, G.oracle_pools(inp))


def test_append_scale_rounding_boundaries():
    """Block maxima at every E4M3 rounding midpoint of the scale quotient, and
    one bf16 step to either side.  With g = fl32(1/6), 6 g rounds to exactly
    1, so amax / (6 g) is the block maximum itself: at a midpoint the scale
    byte is decided by the tie rule (nearest even), next to one by the nearer
    code, and the codes follow from that byte.  Every byte must match."""
    wl = W.Workload("scale_ties", [1], [128], 2, 2, seed=17)
    inp = W.make_inputs(wl, with_q=False)
    e4 = torch.arange(0, 127, dtype=torch.uint8).view(torch.float8_e4m3fn).float()  # 0 .. 448
    mids = (e4[1:] + e4[:-1]) / 2
    assert torch.equal(mids.to(torch.bfloat16).float(), mids)  # at most 5 significant bits
    mb = mids.to(torch.bfloat16).view(torch.int16)
    targets = torch.cat([mids, (mb - 1).view(torch.bfloat16).float(), (mb + 1).view(torch.bfloat16).float()])
    gen = torch.Generator().manual_seed(5)
    k = inp.k.float().view(-1, 16)                       # one row per 16-value block
    t = targets[torch.arange(k.shape[0]) % targets.numel()]
    k = (torch.rand(k.shape, generator=gen) * 2 - 1) * t[:, None]
    pos = torch.arange(k.shape[0]) % 16                  # the element that carries the maximum
    sign = torch.where(torch.arange(k.shape[0]) % 3 == 0, -1.0, 1.0)
    k[torch.arange(k.shape[0]), pos] = sign * t
    inp.k = k.view_as(inp.k).to(torch.bfloat16)
    assert torch.equal(inp.k.float().view(-1, 16).abs().amax(1), t)
    inp.k_global = float(np.float32(1.0 / 6.0))
    assert np.float32(6.0) * np.float32(inp.k_global) == np.float32(1.0)
    cache = G.gpu_cache(inp)
    _assert_same(cache, G.oracle_pools(inp))
    assert G.nk().nvfp4kv_get_device_status() == 0


def test_append_bad_slot_flagged():
    inp = W.make_inputs(W.Workload("bad", [1], [20], 2, 2, seed=2), with_q=False)
    slots = inp.slot_mapping.clone()
    slots[4] = inp.num_pages * 16 + 5           # beyond the pool
    inp.slot_mapping = slots
    b = G.nk()
    G.gpu_cache(inp)
    torch.cuda.synchronize()
    assert b.nvfp4kv_get_device_status() == -6
    assert b.nvfp4kv_get_device_status() == 0  # cleared by the read


def test_quantize_rows_matches_oracle():
    import oracle
    b = G.nk()
    gen = torch.Generator().manual_seed(21)
    x = (torch.randn(777, 128, generator=gen) * torch.exp(torch.randn(777, 1, generator=gen) * 3)).to(torch.bfloat16)
    x[5] = 0
    xf = x.float().numpy()
    g = float(np.float32(np.abs(xf).max() / 2688.0))
    p, s, _ = b.nvfp4_quantize_rows(x.to(G.dev()), b.QUANT_GLOBAL, g)
    rp, rs, _ = oracle.quantize_rows(xf, oracle.GLOBAL, g)
    assert np.array_equal(p.cpu().numpy(), rp) and np.array_equal(s.cpu().numpy(), rs)
    p, s, rg = b.nvfp4_quantize_rows(x.to(G.dev()), b.QUANT_PER_ROW)
    rp, rs, rrg = oracle.quantize_rows(xf, oracle.PER_ROW)
    assert np.array_equal(p.cpu().numpy(), rp) and np.array_equal(s.cpu().numpy(), rs)
    assert np.array_equal(rg.cpu().numpy(), rrg)
    out = b.nvfp4_dequantize_rows(p, s, row_scales=rg).float().cpu().numpy()
    ref = oracle.dequantize_rows(rp, rs, row_g=rrg)
    assert np.allclose(out, ref, rtol=2 ** -8, atol=0)
