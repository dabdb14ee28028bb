"""Helpers shared by the GPU parity tests: run the CUDA path through the
binding, run the oracle on the same seeded inputs, compare."""
import numpy as np
import torch

import oracle
from nvfp4_paged_kv_append_gb300 import workloads as W

MAX_ABS = 2e-2   # attention output tolerance: max |gpu - oracle| beyond the output's bf16 rounding
REL_FRO = 1e-2   # ||gpu - oracle||_F / ||oracle||_F


def bf16_half_ulp(x):
    """Half a bf16 unit in the last place of |x| (8 significant bits): the
    rounding the stored bf16 output adds on top of the kernel's own error."""
    a = np.maximum(np.abs(x), np.float64(2.0 ** -126))
    return np.ldexp(1.0, np.floor(np.log2(a)).astype(np.int64) - 8)


def nk():
    from nvfp4_paged_kv_append_gb300 import build
    build.build()
    from nvfp4_paged_kv_append_gb300 import binding
    return binding


def dev():
    return torch.device("cuda:0")


_INPUTS = {}
_POOLS = {}


def inputs(cfg):
    """Seeded inputs of a named configuration, built once per session."""
    if cfg not in _INPUTS:
        _INPUTS[cfg] = W.make_inputs(W.CONFIGS[cfg]())
    return _INPUTS[cfg]


def pools_for(cfg):
    """Oracle cache of a named configuration, built once per session."""
    if cfg not in _POOLS:
        _POOLS[cfg] = oracle_pools(inputs(cfg))
    return _POOLS[cfg]


def gpu_cache(inp, fill=0, append_order=None):
    """Build the cache on the GPU with the CUDA append (optionally appending
    tokens in a shuffled order)."""
    b = nk()
    c = b.Cache(inp.num_pages, inp.wl.num_kv_heads, inp.k_global, inp.v_global, device=dev(), fill=fill)
    k, v, s = inp.k, inp.v, inp.slot_mapping
    if append_order is not None:
        k, v, s = k[append_order], v[append_order], s[append_order]
    b.nvfp4_kv_append(k.contiguous().to(dev()), v.contiguous().to(dev()), s.contiguous().to(dev()), c)
    return c


def oracle_pools(inp, token_subset=None):
    pools = oracle.Pools(inp.num_pages, inp.wl.num_kv_heads)
    k, v, s = inp.k.float().numpy(), inp.v.float().numpy(), inp.slot_mapping.numpy()
    if token_subset is not None:
        k, v, s = k[token_subset], v[token_subset], s[token_subset]
    oracle.kv_append(pools, k, v, s, inp.k_global, inp.v_global)
    return pools


def compare_rows(got, ref, qo_indptr):
    """got: [total_q, Hq, D] numpy; ref: oracle dict {(b, i): (o, lse)}.
    Returns (max_abs, rel_fro, n_rows) where max_abs is the largest
    |gpu - oracle| in excess of half a bf16 ulp of the oracle value (the
    output is stored as bf16)."""
    diffs, refs = [], []
    for (b, i), (o, _) in ref.items():
        g = got[int(qo_indptr[b]) + i]
        diffs.append(g - o)
        refs.append(o)
    d = np.stack(diffs)
    r = np.stack(refs)
    excess = np.maximum(np.abs(d) - bf16_half_ulp(r), 0.0)
    return float(excess.max()), float(np.linalg.norm(d) / max(np.linalg.norm(r), 1e-30)), len(diffs)


def compare_rows_slack(got, ref, qo_indptr):
    """As compare_rows, for oracle values (o, lse, slack) of the FP4 PV
    experiment: the excess is measured beyond half a bf16 ulp plus the slack
    (how far the output may move when P decisions that lie within the
    oracle's eps of a rounding boundary go the other way).  Also returns the
    largest raw |gpu - oracle| and the largest slack."""
    diffs, refs, slacks = [], [], []
    for (b, i), (o, _, sl) in ref.items():
        diffs.append(got[int(qo_indptr[b]) + i] - o)
        refs.append(o)
        slacks.append(sl)
    d, r, sl = np.stack(diffs), np.stack(refs), np.stack(slacks)
    excess = np.maximum(np.abs(d) - bf16_half_ulp(r) - sl, 0.0)
    return (float(excess.max()), float(np.linalg.norm(d) / max(np.linalg.norm(r), 1e-30)), len(diffs),
            float(np.abs(d).max()), float(sl.max()))


def compare_lse(got_lse, ref, qo_indptr):
    err = 0.0
    for (b, i), vals in ref.items():
        err = max(err, float(np.abs(got_lse[int(qo_indptr[b]) + i] - vals[1]).max()))
    return err


def prefill_workspace(inp, mode):
    """mode "auto": room for repack mode (used when the batch qualifies);
    "inkernel": the schedule only, so V is dequantized inside the kernel."""
    b = nk()
    wl = inp.wl
    max_kv = inp.page_table.shape[1] * 16 if mode == "auto" else 0
    n = b.nvfp4_workspace_bytes(b.OP_PREFILL, wl.batch, wl.num_q_heads, wl.num_kv_heads, wl.total_q, max_kv)
    return torch.empty(max(n, 16), dtype=torch.uint8, device=dev())


def run_prefill(inp, cache, variant, causal=True, with_lse=True, mode="auto"):
    b = nk()
    q = inp.q.to(dev())
    lse = torch.full((inp.wl.total_q, inp.wl.num_q_heads), float("nan"), device=dev()) if with_lse else None
    o = b.nvfp4_paged_prefill(q, cache, inp.page_table.to(dev()), inp.kv_lens.to(dev()), inp.qo_indptr.to(dev()),
                              causal=causal, sm_scale=inp.sm_scale, variant=variant, lse=lse,
                              workspace=prefill_workspace(inp, mode))
    torch.cuda.synchronize()
    status = b.nvfp4kv_get_device_status()
    return o.float().cpu().numpy(), (lse.cpu().numpy() if with_lse else None), status


def oracle_prefill(pools, inp, q_mode, causal=True, rows=None):
    return oracle.paged_attention(pools, inp.q.float().numpy(), inp.qo_indptr, inp.kv_lens, inp.page_table,
                                  inp.wl.num_q_heads, inp.k_global, inp.v_global, causal, inp.sm_scale,
                                  q_mode=q_mode, rows=rows)


_ORACLE_OUT = {}


def oracle_prefill_cached(cfg, q_mode, rows, causal=True):
    """oracle_prefill on a named configuration's session inputs, computed once
    per (configuration, query mode, row set) and shared by the tests that run
    the same rows in several kernel modes."""
    key = (cfg, q_mode, causal, None if rows is None else tuple(rows))
    if key not in _ORACLE_OUT:
        _ORACLE_OUT[key] = oracle_prefill(pools_for(cfg), inputs(cfg), q_mode, causal=causal, rows=rows)
    return _ORACLE_OUT[key]


def repack_mode_expected(wl, variant=0):
    """The library's rule for repack mode given a workspace with room for the
    records: requests average at least eight 128-row q tiles per kv head for
    A4Q (variant 0), two for dequant-ahead."""
    qtiles = (wl.total_q * wl.group + 127) // 128
    return qtiles >= (8 if variant == 0 else 2) * wl.batch
