"""The library's calls inside CUDA graphs: every call is asynchronous on the
caller's stream, with no host synchronisation and no allocation, so a
serving engine can capture it.  Decode (both formats) and prefill (plan and
run) captured once and replayed give, bit for bit, the outputs of eager
calls on the same inputs."""
import pytest
import torch

from nvfp4_paged_kv_append_gb300 import workloads as W

from . import _gpu as G

pytestmark = pytest.mark.gpu


def _replay_equals_eager(fn, out):
    """fn writes `out`; eager result, then a captured graph replayed twice."""
    fn()
    torch.cuda.synchronize()
    eager = out.clone()
    out.zero_()
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        fn()  # warm-up on the capture stream (first-use set-up happens outside the capture)
    torch.cuda.current_stream().wait_stream(stream)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    for _ in range(2):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), eager.view(torch.int16))


@pytest.mark.parametrize("fmt", ["nvfp4", "fp8"])
def test_decode_in_a_graph(fmt):
    wl = W.Workload("graph_dec", [1] * 6, [40, 1500, 3000, 17, 900, 5000], 16, 4, seed=3)
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
    out = torch.empty_like(q)
    _replay_equals_eager(lambda: dec(q, cache, pt, kvl, sm_scale=inp.sm_scale, out=out, workspace=ws,
                                     stream=torch.cuda.current_stream()), out)
    assert b.nvfp4kv_get_device_status() == 0


@pytest.mark.parametrize("variant", [0, 1, 2])
def test_prefill_plan_and_run_in_a_graph(variant):
    inp = G.inputs("small_ragged")
    wl = inp.wl
    b = G.nk()
    d = G.dev()
    cache = G.gpu_cache(inp)
    q, pt, kvl, qo = inp.q.to(d), inp.page_table.to(d), inp.kv_lens.to(d), inp.qo_indptr.to(d)
    ws = G.prefill_workspace(inp, "auto")
    out = torch.empty_like(q)

    def step():
        s = torch.cuda.current_stream()
        b.nvfp4_paged_prefill_plan(cache, wl.total_q, wl.num_q_heads, pt, kvl, qo, ws, variant=variant, stream=s)
        b.nvfp4_paged_prefill_run(q, cache, pt, kvl, qo, ws, sm_scale=inp.sm_scale, variant=variant, out=out,
                                  stream=s)

    _replay_equals_eager(step, out)
    assert b.nvfp4kv_get_device_status() == 0
