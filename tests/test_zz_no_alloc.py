"""The allocation-free prefill entry point against the regular one.

Some callers cannot allocate device memory when they call the library (an
engine whose serving path allows no cudaMalloc, or a plugin host that passes
no scratch pointer); nvfp4_paged_prefill_noalloc keeps its work schedule in
the library's static device array instead of a caller workspace.  Its output
must match nvfp4_paged_prefill's within the parity tolerance, on two calls in
a row (the array keeps the previous call's contents).  This file is collected
last so that a first-failure run has already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

from nvfp4_paged_kv_append_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _nk():
    from nvfp4_paged_kv_append_gb300 import build
    build.build()
    from nvfp4_paged_kv_append_gb300 import binding
    return binding


def _excess(a, b):
    """max |a - b| beyond half a bf16 ulp of b (both outputs are bf16)."""
    a = a.float().cpu().numpy().astype(np.float64)
    b = b.float().cpu().numpy().astype(np.float64)
    half_ulp = np.ldexp(1.0, np.floor(np.log2(np.maximum(np.abs(b), 2.0 ** -126))).astype(np.int64) - 8)
    return float(np.maximum(np.abs(a - b) - half_ulp, 0.0).max())


@pytest.mark.parametrize("variant", [0, 1])
def test_noalloc_matches_workspace_entry_point(variant):
    nk = _nk()
    dev = torch.device("cuda:0")
    results = []
    for cfg in ("small_ragged", "shortq"):   # two different schedules, back to back
        inp = W.make_inputs(W.CONFIGS[cfg]())
        cache = nk.Cache(inp.num_pages, inp.wl.num_kv_heads, inp.k_global, inp.v_global, device=dev)
        nk.nvfp4_kv_append(inp.k.to(dev), inp.v.to(dev), inp.slot_mapping.to(dev), cache)
        args = (inp.q.to(dev), cache, inp.page_table.to(dev), inp.kv_lens.to(dev), inp.qo_indptr.to(dev))
        ref = nk.nvfp4_paged_prefill(*args, sm_scale=inp.sm_scale, variant=variant)
        for call in range(2):
            out = torch.full_like(ref, float("nan"))
            nk.nvfp4_paged_prefill_noalloc(*args, sm_scale=inp.sm_scale, variant=variant, out=out)
            torch.cuda.synchronize()
            assert nk.nvfp4kv_get_device_status() == 0
            err = _excess(out, ref)
            results.append((cfg, call, err))
            assert err <= 2e-2, (cfg, call, err)
            assert torch.isfinite(out.float()).all()


def test_noalloc_rejects_oversized_schedule():
    nk = _nk()
    cap = nk.nvfp4_paged_prefill_noalloc_max_bytes()
    assert cap == 1 << 20
    d = nk.CacheDesc(16, 16, 32, 48, 4, 16, 8, 128, 1.0, 1.0)
    # 4M query tokens x 64 q heads over 8 kv heads: far more work items than fit
    rc = nk.lib.nvfp4_paged_prefill_noalloc(16, 4_000_000, 64, ctypes.byref(d), 16, 1, 16, 16, 1, 1, 0.1, 0,
                                            16, None, None)
    assert rc == -3
