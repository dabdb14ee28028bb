"""The Python binding checks dtypes, shapes and device placement before any
pointer reaches the library (every pointer of the ABI except the cache
descriptor is a device pointer).  On the CPU the checks run all the way to
the device-placement test, so valid shapes are seen to pass every other
check and invalid ones to be refused."""
import pytest
import torch

from nvfp4_paged_kv_append_gb300 import workloads as W

ON_DEVICE = "must live on a CUDA device"


@pytest.fixture(scope="module")
def b():
    import __graft_entry__ as g
    g.build()
    from nvfp4_paged_kv_append_gb300 import binding
    return binding


def _cache(b, inp):
    return b.Cache(inp.num_pages, inp.wl.num_kv_heads, inp.k_global, inp.v_global, device=torch.device("cpu"))


@pytest.fixture(scope="module")
def inp():
    return W.make_inputs(W.Workload("bind", [3, 5], [20, 40], 8, 2, seed=2))


def test_valid_calls_reach_only_the_device_check(b, inp):
    c = _cache(b, inp)
    with pytest.raises(ValueError, match=ON_DEVICE):
        b.nvfp4_kv_append(inp.k, inp.v, inp.slot_mapping, c)
    lse = torch.empty(inp.wl.total_q, inp.wl.num_q_heads)
    with pytest.raises(ValueError, match=ON_DEVICE):
        b.nvfp4_paged_prefill(inp.q, c, inp.page_table, inp.kv_lens, inp.qo_indptr, lse=lse)
    ws = torch.empty(1 << 16, dtype=torch.uint8)
    with pytest.raises(ValueError, match=ON_DEVICE):
        b.nvfp4_paged_prefill_plan(c, inp.wl.total_q, inp.wl.num_q_heads, inp.page_table, inp.kv_lens,
                                   inp.qo_indptr, ws)
    with pytest.raises(ValueError, match=ON_DEVICE):
        b.nvfp4_paged_prefill_run(inp.q, c, inp.page_table, inp.kv_lens, inp.qo_indptr, ws)
    with pytest.raises(ValueError, match=ON_DEVICE):
        b.nvfp4_paged_prefill_noalloc(inp.q, c, inp.page_table, inp.kv_lens, inp.qo_indptr)
    qd = inp.q[inp.qo_indptr[1:] - 1].contiguous()  # one query per request
    with pytest.raises(ValueError, match=ON_DEVICE):
        b.nvfp4_paged_decode(qd, c, inp.page_table, inp.kv_lens, lse=torch.empty(2, 8))
    x = torch.randn(6, 128).to(torch.bfloat16)
    with pytest.raises(ValueError, match=ON_DEVICE):
        b.nvfp4_quantize_rows(x, b.QUANT_PER_ROW)
    with pytest.raises(ValueError, match=ON_DEVICE):
        b.nvfp4_dequantize_rows(torch.zeros(6, 64, dtype=torch.uint8), torch.zeros(6, 8, dtype=torch.uint8),
                                row_scales=torch.ones(6))


def test_bad_dtypes_and_shapes_are_refused(b, inp):
    c = _cache(b, inp)
    with pytest.raises(ValueError, match="q must be"):
        b.nvfp4_paged_prefill(inp.q.float(), c, inp.page_table, inp.kv_lens, inp.qo_indptr)
    with pytest.raises(ValueError, match="kv_lens must be"):
        b.nvfp4_paged_prefill(inp.q, c, inp.page_table, inp.kv_lens.long(), inp.qo_indptr)
    with pytest.raises(ValueError, match="qo_indptr must be"):
        b.nvfp4_paged_prefill(inp.q, c, inp.page_table, inp.kv_lens, inp.qo_indptr[:-1])
    with pytest.raises(ValueError, match="page_table must be"):
        b.nvfp4_paged_prefill(inp.q, c, inp.page_table[:1], inp.kv_lens, inp.qo_indptr)
    with pytest.raises(ValueError, match="lse must be"):
        b.nvfp4_paged_prefill(inp.q, c, inp.page_table, inp.kv_lens, inp.qo_indptr,
                              lse=torch.empty(inp.wl.total_q, 3))
    with pytest.raises(ValueError, match="out must have"):
        b.nvfp4_paged_prefill(inp.q, c, inp.page_table, inp.kv_lens, inp.qo_indptr,
                              out=torch.empty(1, 8, 128, dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="one query token per request"):
        b.nvfp4_paged_decode(inp.q, c, inp.page_table, inp.kv_lens)
    with pytest.raises(ValueError, match="slot_mapping must be"):
        b.nvfp4_kv_append(inp.k, inp.v, inp.slot_mapping.int(), c)
    with pytest.raises(ValueError, match="k and v must be"):
        b.nvfp4_kv_append(inp.k, inp.v[:, :1].contiguous(), inp.slot_mapping, c)
    with pytest.raises(ValueError, match="workspace must be"):
        b.nvfp4_paged_prefill_run(inp.q, c, inp.page_table, inp.kv_lens, inp.qo_indptr, torch.empty(16))
    with pytest.raises(ValueError, match="packed must be"):
        b.nvfp4_dequantize_rows(torch.zeros(6, 32, dtype=torch.uint8), torch.zeros(6, 8, dtype=torch.uint8))


def test_host_cache_is_refused_first(b, inp):
    """The cache pools are checked before the other tensors: a cache in host
    memory is named in the error even when the other arguments are fine."""
    c = _cache(b, inp)
    with pytest.raises(ValueError, match="cache pools must live on a CUDA device"):
        b.nvfp4_paged_prefill(inp.q, c, inp.page_table, inp.kv_lens, inp.qo_indptr)
    with pytest.raises(ValueError, match="cache pools must live on a CUDA device"):
        b.nvfp4_kv_append(inp.k, inp.v, inp.slot_mapping, c)
    qd = inp.q[inp.qo_indptr[1:] - 1].contiguous()
    with pytest.raises(ValueError, match="cache pools must live on a CUDA device"):
        b.nvfp4_paged_decode(qd, c, inp.page_table, inp.kv_lens)


def test_device_helper_refuses_host_and_mixed_tensors(b):
    with pytest.raises(ValueError, match="must live on a CUDA device"):
        b._device(torch.zeros(2), None)
    with pytest.raises(ValueError, match="must live on a CUDA device"):
        b._device(None)
    # any non-CUDA device is refused, not only the host
    with pytest.raises(ValueError, match="must live on a CUDA device"):
        b._device(torch.zeros(2, device="meta"))
