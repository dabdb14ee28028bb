"""The allocation-free prefill entry point.

Some callers cannot allocate device memory when they call the library (an
engine whose serving path allows no cudaMalloc, or a plugin host that passes
no scratch pointer); nvfp4_paged_prefill_noalloc keeps its work schedule in
the library's static device array instead of a caller workspace, and always
runs the in-kernel mode.  On two calls in a row (the array keeps the previous
call's contents) its output must match the oracle within the parity tolerance
and equal, bit for bit, nvfp4_paged_prefill given a schedule-only workspace.
This file is collected last so that a first-failure run has already run every
other test."""
import ctypes

import numpy as np
import pytest
import torch

from nvfp4_paged_kv_append_gb300 import workloads as W

from . import _gpu as G

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("variant,q_mode", [(0, "a4q"), (1, "bf16")])
def test_noalloc_matches_oracle_and_inkernel_mode(variant, q_mode):
    nk = G.nk()
    dev = G.dev()
    for cfg in ("small_ragged", "shortq"):   # two different schedules, back to back
        inp = G.inputs(cfg)
        cache = G.gpu_cache(inp)
        args = (inp.q.to(dev), cache, inp.page_table.to(dev), inp.kv_lens.to(dev), inp.qo_indptr.to(dev))
        ws_min = G.prefill_workspace(inp, "inkernel")
        same = nk.nvfp4_paged_prefill(*args, sm_scale=inp.sm_scale, variant=variant, workspace=ws_min)
        rows = None if cfg == "small_ragged" else W.tile_rows(inp.wl)
        ref = G.oracle_prefill_cached(cfg, q_mode, rows)
        for call in range(2):
            out = torch.full_like(same, float("nan"))
            nk.nvfp4_paged_prefill_noalloc(*args, sm_scale=inp.sm_scale, variant=variant, out=out)
            torch.cuda.synchronize()
            assert nk.nvfp4kv_get_device_status() == 0
            assert torch.equal(out.view(torch.int16), same.view(torch.int16)), (cfg, call)
            mx, fro, n = G.compare_rows(out.float().cpu().numpy(), ref, inp.qo_indptr)
            assert mx <= G.MAX_ABS and fro <= G.REL_FRO, (cfg, call, mx, fro, n)


def test_noalloc_rejects_oversized_schedule():
    """A call whose schedule would not fit the static array is refused on the
    host (nothing is launched); the buffers are real, small device tensors."""
    nk = G.nk()
    dev = G.dev()
    cap = nk.nvfp4_paged_prefill_noalloc_max_bytes()
    assert cap == 1 << 20
    cache = nk.Cache(4, 8, 1.0, 1.0, device=dev)
    q = torch.zeros(16, 64, 128, dtype=torch.bfloat16, device=dev)
    out = torch.empty_like(q)
    pt = torch.zeros(1, 4, dtype=torch.int32, device=dev)
    kvl = torch.full((1,), 16, dtype=torch.int32, device=dev)
    qo = torch.tensor([0, 16], dtype=torch.int32, device=dev)
    d = cache.desc()
    P = ctypes.c_void_p
    # total_q claims 4M query tokens x 64 q heads over 8 kv heads: far more
    # work items than the array holds, so the call returns before any launch
    rc = nk.lib.nvfp4_paged_prefill_noalloc(P(q.data_ptr()), 4_000_000, 64, ctypes.byref(d), P(pt.data_ptr()), 4,
                                            P(kvl.data_ptr()), P(qo.data_ptr()), 1, 1, 0.1, 0, 0.0,
                                            P(out.data_ptr()), None, None)
    assert rc == -3
    torch.cuda.synchronize()
    assert nk.nvfp4kv_get_device_status() == 0
    assert np.isfinite(q.float().cpu().numpy()).all()


def test_noalloc_refuses_the_fp4pv_variant():
    """The FP4 PV variant reads only repacked records, which the static array
    (a schedule only) does not hold: refused before any launch."""
    nk = G.nk()
    dev = G.dev()
    inp = G.inputs("tiny")
    cache = G.gpu_cache(inp)
    args = (inp.q.to(dev), cache, inp.page_table.to(dev), inp.kv_lens.to(dev), inp.qo_indptr.to(dev))
    with pytest.raises(nk.NvFp4Error) as e:
        nk.nvfp4_paged_prefill_noalloc(*args, variant=nk.VARIANT_A4Q_FP4PV)
    assert e.value.code == nk.NVFP4KV_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert nk.nvfp4kv_get_device_status() == 0
