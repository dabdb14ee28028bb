"""Paged decode on the GPU against the oracle (BF16 query, decoded K/V):
max-abs <= 2e-2 and relative Frobenius <= 1e-2 ("NVFP4 KV cache prefill vs
decode performance", section "Decode can win on fewer bytes read")."""
import numpy as np
import pytest
import torch

from nvfp4_paged_kv_append_gb300 import workloads as W

from . import _gpu as G

pytestmark = pytest.mark.gpu


def _decode_case(wl, fill=0, sample=None, split_len=None):
    inp = W.make_inputs(wl)
    b = G.nk()
    cache = G.gpu_cache(inp, fill=fill)
    # the decode query of request b is its (single) query row
    q = inp.q.to(G.dev())
    pt = inp.page_table.to(G.dev())
    lse = torch.full((wl.batch, wl.num_q_heads), float("nan"), device=G.dev())
    ws = torch.empty(b.nvfp4_workspace_bytes(b.OP_DECODE, wl.batch, wl.num_q_heads, wl.num_kv_heads, 0,
                                             pt.shape[1] * 16), dtype=torch.uint8, device=G.dev())
    o = b.nvfp4_paged_decode(q, cache, pt, inp.kv_lens.to(G.dev()), sm_scale=inp.sm_scale, lse=lse, workspace=ws)
    torch.cuda.synchronize()
    assert b.nvfp4kv_get_device_status() == 0
    if split_len is not None:
        # the schedule header (item count, claim counter, split length) opens
        # the workspace: the schedule kernel chose the expected item length
        assert int(ws[:16].view(torch.int32)[2]) == split_len
    reqs = range(wl.batch) if sample is None else sample
    rows = [(r, 0) for r in reqs if wl.kv_lens[r] > 0]
    pools = G.oracle_pools(inp)
    ref = G.oracle_prefill(pools, inp, "bf16", causal=False, rows=rows)
    got = o.float().cpu().numpy()
    mx, fro, n = G.compare_rows(got, ref, inp.qo_indptr)
    lerr = G.compare_lse(lse.cpu().numpy(), ref, inp.qo_indptr)
    return mx, fro, lerr, got, inp


@pytest.mark.parametrize("group", [1, 2, 4, 8, 16])
def test_decode_groups(group):
    wl = W.Workload(f"dec_g{group}", [1] * 5, [1, 17, 256, 257, 700], 2 * group, 2, seed=group)
    mx, fro, lerr, _, _ = _decode_case(wl)
    assert mx <= G.MAX_ABS and fro <= G.REL_FRO, (mx, fro)
    assert lerr <= 1e-3, lerr


def test_decode_outliers_and_junk_pool():
    """Pool bytes outside the written slots are 0x7F (an E4M3 NaN): every
    unused slot of a partly filled page must be ignored."""
    wl = W.Workload("dec_out", [1] * 3, [33, 513, 1000], 8, 2, dist="outliers", seed=4)
    mx, fro, lerr, got, _ = _decode_case(wl, fill=0x7F)
    assert np.isfinite(got).all()
    assert mx <= G.MAX_ABS and fro <= G.REL_FRO, (mx, fro)


def test_decode_full_size_all_requests():
    """32 requests with kv_len ~ U[1K, 32K], 32/8 heads, at full size (the
    benchmark's decode batch); the oracle checks every request and head."""
    wl = W.decode_batch()
    mx, fro, lerr, _, _ = _decode_case(wl, split_len=4096)
    assert mx <= G.MAX_ABS and fro <= G.REL_FRO, (mx, fro)
    assert lerr <= 1e-3


def test_decode_split_length_2048():
    """Enough work for 2,048-token items but not for 4,096 ones (at least two
    items per attention CTA on 152 SMs): 20 requests of 14K-16K keys, 32/8
    heads, every request against the oracle."""
    rng = np.random.default_rng(33)
    kv = [int(x) for x in rng.integers(14000, 16001, size=20)]
    wl = W.Workload("dec_split2048", [1] * 20, kv, 32, 8, seed=33)
    mx, fro, lerr, _, _ = _decode_case(wl, split_len=2048)
    assert mx <= G.MAX_ABS and fro <= G.REL_FRO, (mx, fro)
    assert lerr <= 1e-3


def test_decode_empty_request():
    wl = W.Workload("dec_empty", [1, 1], [0, 40], 4, 2, seed=8)
    inp = W.make_inputs(wl)
    b = G.nk()
    cache = G.gpu_cache(inp)
    o = b.nvfp4_paged_decode(inp.q.to(G.dev()), cache, inp.page_table.to(G.dev()), inp.kv_lens.to(G.dev()),
                             sm_scale=inp.sm_scale)
    torch.cuda.synchronize()
    assert float(o[0].abs().max()) == 0.0


def test_decode_more_than_1024_requests():
    """1,100 requests (the schedule takes them 1,024 at a time), mostly short
    with some over two splits; sampled requests against the oracle."""
    rng = np.random.default_rng(21)
    kv = rng.integers(1, 200, size=1100)
    long_ = rng.choice(1100, size=60, replace=False)
    kv[long_] = rng.integers(1025, 2600, size=60)
    wl = W.Workload("dec_1100", [1] * 1100, [int(x) for x in kv], 8, 2, seed=21)
    sample = sorted({0, 1023, 1024, 1099, int(kv.argmax())} | {int(x) for x in long_[:6]})
    mx, fro, lerr, _, _ = _decode_case(wl, sample=sample)
    assert mx <= G.MAX_ABS and fro <= G.REL_FRO, (mx, fro)
    assert lerr <= 1e-3, lerr


def test_decode_kv_len_beyond_table_flagged():
    """A kv_len longer than the page table allows is flagged (shape error);
    that request's output is zero and the others are unaffected."""
    wl = W.Workload("dec_bad", [1] * 3, [300, 1500, 40], 8, 2, seed=9)
    inp = W.make_inputs(wl)
    b = G.nk()
    cache = G.gpu_cache(inp)
    kvl = inp.kv_lens.clone()
    kvl[1] = inp.page_table.shape[1] * 16 + 1
    o = b.nvfp4_paged_decode(inp.q.to(G.dev()), cache, inp.page_table.to(G.dev()), kvl.to(G.dev()),
                             sm_scale=inp.sm_scale)
    torch.cuda.synchronize()
    assert b.nvfp4kv_get_device_status() == -2
    got = o.float().cpu().numpy()
    assert float(np.abs(got[1]).max()) == 0.0
    pools = G.oracle_pools(inp)
    ref = G.oracle_prefill(pools, inp, "bf16", causal=False, rows=[(0, 0), (2, 0)])
    mx, fro, _ = G.compare_rows(got, ref, inp.qo_indptr)
    assert mx <= G.MAX_ABS and fro <= G.REL_FRO, (mx, fro)


@pytest.mark.parametrize("fmt", ["nvfp4", "fp8"])
def test_decode_repeatable(fmt):
    """The batch-32 decode gives the same bits on every call, whatever the
    workspace held before: items are claimed in a different order by
    different CTAs each time, the split merges run wherever the last split
    finishes, and no result may depend on that."""
    wl = W.decode_batch()
    inp = W.make_inputs(wl)
    b = G.nk()
    d = G.dev()
    if fmt == "fp8":
        cache = b.Fp8Cache(inp.num_pages, wl.num_kv_heads, W.fp8_scale(inp.k), W.fp8_scale(inp.v), device=d)
        b.fp8_kv_append(inp.k.to(d), inp.v.to(d), inp.slot_mapping.to(d), cache)
        dec, wsb = b.fp8_paged_decode, b.fp8_workspace_bytes
    else:
        cache = G.gpu_cache(inp)
        dec, wsb = b.nvfp4_paged_decode, b.nvfp4_workspace_bytes
    q, pt, kvl = inp.q.to(d), inp.page_table.to(d), inp.kv_lens.to(d)
    ws = torch.empty(wsb(b.OP_DECODE, wl.batch, wl.num_q_heads, wl.num_kv_heads, 0, pt.shape[1] * 16),
                     dtype=torch.uint8, device=d)
    outs = []
    for i in range(8):
        ws.fill_(i * 41 % 256)
        lse = torch.empty(wl.batch, wl.num_q_heads, device=d)
        o = dec(q, cache, pt, kvl, sm_scale=inp.sm_scale, lse=lse, workspace=ws)
        torch.cuda.synchronize()
        outs.append((o.view(torch.int16).cpu(), lse.view(torch.int32).cpu()))
    assert b.nvfp4kv_get_device_status() == 0
    for o, l in outs[1:]:
        assert torch.equal(o, outs[0][0]) and torch.equal(l, outs[0][1])
