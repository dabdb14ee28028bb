"""Pins of the oracle's attention against library routines, closed forms and
invariants.  Scores are computed before softmax and the query accuracy gate
covers lengths, head shapes, causal masks and scale outliers ("NVFP4 KV cache
A4Q prefill explained", section "Make query accuracy a release gate")."""
import math

import numpy as np
import pytest
import scipy.special as sps

from nvfp4_paged_kv_append_gb300 import workloads as W


def lib_attention(q, k, v, pos, q_len, causal, sm_scale):
    """scipy softmax + numpy matmul, one row at a time."""
    kv_len = k.shape[0]
    out, lse = [], []
    for r, i in enumerate(pos):
        last = kv_len - q_len + i if causal else kv_len - 1
        s = sm_scale * (k[: last + 1] @ q[r])
        out.append(sps.softmax(s) @ v[: last + 1])
        lse.append(sps.logsumexp(s))
    return np.array(out), np.array(lse)


@pytest.mark.parametrize("q_len,kv_len,causal", [(7, 7, True), (5, 19, True), (9, 33, False), (1, 40, True)])
def test_attention_vs_library(orc, q_len, kv_len, causal):
    rng = np.random.default_rng(q_len * 100 + kv_len)
    D = 16
    q = rng.standard_normal((q_len, D))
    k = rng.standard_normal((kv_len, D)) * 2
    v = rng.standard_normal((kv_len, D))
    pos = np.arange(q_len)
    o, lse = orc.attention_rows(q, pos, q_len, k, v, causal, 0.3)
    o_ref, lse_ref = lib_attention(q, k, v, pos, q_len, causal, 0.3)
    np.testing.assert_allclose(o, o_ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref, rtol=1e-12, atol=1e-12)


def test_attention_closed_forms(orc):
    rng = np.random.default_rng(2)
    D, n = 8, 12
    q = rng.standard_normal((n, D))
    v = rng.standard_normal((n, D))
    # equal keys: uniform weights, O = mean of the visible V rows
    k = np.tile(rng.standard_normal(D), (n, 1))
    o, lse = orc.attention_rows(q, np.arange(n), n, k, v, True, 1.0)
    for i in range(n):
        np.testing.assert_allclose(o[i], v[: i + 1].mean(axis=0), rtol=1e-13, atol=1e-13)
        assert abs(lse[i] - (q[i] @ k[0] + math.log(i + 1))) < 1e-12
    # one visible key: the first causal row with q_len == kv_len returns V[0]
    k = rng.standard_normal((n, D)) * 10
    o, _ = orc.attention_rows(q[:1], np.array([0]), n, k, v, True, 1.0)
    np.testing.assert_array_equal(o[0], v[0])
    # bottom-right alignment: with q_len < kv_len the last query sees every key
    o_last, _ = orc.attention_rows(q[:1], np.array([3]), 4, k, v, True, 0.5)
    o_full, _ = orc.attention_rows(q[:1], np.array([0]), 1, k, v, False, 0.5)
    np.testing.assert_array_equal(o_last, o_full)


def test_paged_gather_invariant_under_page_permutation(orc):
    """Moving pages to other pool positions (and the page table with them)
    leaves the decoded K/V and the attention output unchanged."""
    wl = W.Workload("t", [20], [37], 4, 2, seed=3)
    inp = W.make_inputs(wl)
    k = inp.k.float().numpy()
    v = inp.v.float().numpy()
    outs = []
    for seed in (0, 1):
        perm = np.random.default_rng(seed).permutation(inp.num_pages).astype(np.int32)
        pt = perm[: (37 + 15) // 16][None, :]
        j = np.arange(37)
        slots = pt[0, j // 16].astype(np.int64) * 16 + j % 16
        pools = orc.Pools(inp.num_pages, 2)
        orc.kv_append(pools, k, v, slots, inp.k_global, inp.v_global)
        res = orc.paged_attention(pools, inp.q.float().numpy(), inp.qo_indptr, inp.kv_lens, pt, 4,
                                  inp.k_global, inp.v_global, True, inp.sm_scale)
        outs.append(np.stack([res[(0, i)][0] for i in range(20)]))
        kd = orc.gather_decode(pools, "k", pt[0], 37, 1, inp.k_global)
        p_, s_, _ = orc.quantize_rows(k[:, 1], orc.GLOBAL, inp.k_global)
        np.testing.assert_array_equal(kd, orc.dequantize_rows(p_, s_, g=inp.k_global))
    np.testing.assert_array_equal(outs[0], outs[1])


def test_paged_attention_matches_dense_library(orc):
    """The paged, quantized path equals library attention on the decoded
    dense K/V (GQA head mapping h_kv = h_q // G, ragged batch)."""
    wl = W.Workload("t", [13, 5], [13, 30], 6, 2, seed=4)
    inp = W.make_inputs(wl)
    pools = orc.Pools(inp.num_pages, 2)
    orc.kv_append(pools, inp.k.float().numpy(), inp.v.float().numpy(), inp.slot_mapping.numpy(),
                  inp.k_global, inp.v_global)
    res = orc.paged_attention(pools, inp.q.float().numpy(), inp.qo_indptr, inp.kv_lens,
                              inp.page_table, 6, inp.k_global, inp.v_global, True, inp.sm_scale)
    kvi = inp.kv_indptr.numpy()
    for b in range(2):
        ql, kl = wl.q_lens[b], wl.kv_lens[b]
        for hq in range(6):
            h = hq // 3
            kr = inp.k[kvi[b]:kvi[b] + kl, h].float().numpy()
            vr = inp.v[kvi[b]:kvi[b] + kl, h].float().numpy()
            p_, s_, _ = orc.quantize_rows(kr, orc.GLOBAL, inp.k_global)
            kd = orc.dequantize_rows(p_, s_, g=inp.k_global)
            p_, s_, _ = orc.quantize_rows(vr, orc.GLOBAL, inp.v_global)
            vd = orc.dequantize_rows(p_, s_, g=inp.v_global)
            qr = inp.q[inp.qo_indptr[b]:inp.qo_indptr[b + 1], hq].float().numpy().astype(np.float64)
            o_ref, lse_ref = lib_attention(qr, kd, vd, np.arange(ql), ql, True, inp.sm_scale)
            for i in range(ql):
                np.testing.assert_allclose(res[(b, i)][0][hq], o_ref[i], rtol=1e-11, atol=1e-12)
                np.testing.assert_allclose(res[(b, i)][1][hq], lse_ref[i], rtol=1e-12)


def test_a4q_error_grows_with_outliers(orc):
    """The A4Q query changes the scores before softmax: its output differs
    from the BF16-query output, and scale outliers make the gap larger."""
    errs = {}
    for dist in ("normal", "outliers"):
        wl = W.Workload("t", [64], [64], 2, 1, dist=dist, seed=9)
        inp = W.make_inputs(wl)
        pools = orc.Pools(inp.num_pages, 1)
        orc.kv_append(pools, inp.k.float().numpy(), inp.v.float().numpy(), inp.slot_mapping.numpy(),
                      inp.k_global, inp.v_global)
        args = (pools, inp.q.float().numpy(), inp.qo_indptr, inp.kv_lens, inp.page_table, 2,
                inp.k_global, inp.v_global, True, inp.sm_scale)
        a = orc.paged_attention(*args, q_mode="a4q")
        b = orc.paged_attention(*args, q_mode="bf16")
        diff = max(np.abs(a[key][0] - b[key][0]).max() for key in a)
        scale = max(np.abs(b[key][0]).max() for key in b)
        errs[dist] = diff / scale
        assert diff > 0
    assert errs["outliers"] > errs["normal"]


def test_dense_attention_ragged_batch_vs_library(orc):
    """The unquantized reference used for the accuracy report: a ragged batch
    with grouped heads, every row against scipy softmax on the raw values."""
    rng = np.random.default_rng(31)
    q_lens, kv_lens, Hq, Hkv, D = [3, 5], [9, 5], 4, 2, 16
    q = rng.standard_normal((sum(q_lens), Hq, D)).astype(np.float32)
    k = rng.standard_normal((sum(kv_lens), Hkv, D)).astype(np.float32)
    v = rng.standard_normal((sum(kv_lens), Hkv, D)).astype(np.float32)
    qo = np.array([0, 3, 8])
    kvi = np.array([0, 9, 14])
    rows = [(b, i) for b in range(2) for i in range(q_lens[b])]
    got = orc.dense_attention(q, qo, k, v, kvi, Hq, True, 0.25, rows)
    for b, i in rows:
        for hq in range(Hq):
            h = hq // (Hq // Hkv)
            kb = k[kvi[b]:kvi[b + 1], h].astype(np.float64)
            vb = v[kvi[b]:kvi[b + 1], h].astype(np.float64)
            o_ref, lse_ref = lib_attention(q[qo[b] + i, hq][None].astype(np.float64), kb, vb, [i], q_lens[b],
                                           True, 0.25)
            np.testing.assert_allclose(got[(b, i)][0][hq], o_ref[0], rtol=1e-12, atol=1e-12)
            assert abs(got[(b, i)][1][hq] - lse_ref[0]) < 1e-12
