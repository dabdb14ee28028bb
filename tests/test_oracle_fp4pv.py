"""Pins of the oracle's FP4 PV experiment (readings X1..X5 in
oracle/nvfp4_oracle.h).  The pages keep PV wide because the cache's V block
scales run along the head dimension while PV reduces over tokens ("NVFP4 KV
cache A4Q prefill explained", sections "Why NVFP4 KV cache A4Q prefill exists"
and "Compare A4Q with dequantize-ahead repacking"); the experiment re-codes V
along tokens and codes P with the cache's block codec.  What pins it here:
the re-layout's axis against numpy reductions and torch's E4M3 cast, exact
round trips of on-grid values, closed forms (uniform and one-hot attention),
its distance to the exact attention, and the independence from the tiling
and threshold that X3's whole-number reference gives."""
import math

import numpy as np
import pytest
import torch

E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def torch_e4m3(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_token_major_scales_follow_tokens(orc):
    """One scale per head dimension, from the amax over the page's 16 slots
    (numpy's reduction along axis 0, torch's E4M3 cast); each decoded value is
    a nearest point of its dimension's grid."""
    rng = np.random.default_rng(21)
    D = 128
    mag = np.exp2(rng.uniform(-8, 8, D)).astype(np.float32)       # per-dimension magnitude
    x = (rng.standard_normal((16, D)) * mag).astype(np.float32)
    codes, scales = orc.v_token_major_page(x)
    amax = np.abs(x).max(axis=0)                                   # over the 16 tokens
    want = torch_e4m3(amax / np.float32(6.0))
    np.testing.assert_array_equal(scales, want)
    dec = orc.decode_token_major(codes, scales, 1.0)               # [16, D]
    sdec = np.array([orc.e4m3_value(int(b)) for b in scales])
    grid = np.concatenate([-np.array(E2M1[::-1]), np.array(E2M1)])
    dist = np.abs(x[:, :, None] - grid[None, None, :] * sdec[None, :, None]).min(axis=2)
    assert np.all(np.abs(dec - x) <= dist * (1 + 1e-6) + 1e-30)


def test_token_major_round_trip_on_grid(orc):
    """Values that are E2M1 codes times a per-dimension E4M3 scale, with a
    magnitude 6 in every dimension's 16 slots, come back exactly: this fixes
    the axis, the slot order and the nibble order."""
    rng = np.random.default_rng(5)
    D = 128
    c = rng.integers(0, 16, (16, D))
    c[rng.integers(0, 16, D), np.arange(D)] = 7                    # a magnitude 6 in every column
    s_bytes = rng.integers(0x08, 0x7E, D)                          # normal E4M3 scales
    s = np.array([orc.e4m3_value(int(b)) for b in s_bytes])
    vals = np.array([orc.e2m1_value(int(v)) for v in c.ravel()]).reshape(16, D)
    x = (vals * s[None, :]).astype(np.float32)
    codes, scales = orc.v_token_major_page(x)
    np.testing.assert_array_equal(scales, s_bytes)
    np.testing.assert_array_equal(orc.decode_token_major(codes, scales, 1.0), x)
    lo = np.array([[codes[d, t // 2] >> (4 * (t % 2)) & 15 for t in range(16)] for d in range(D)])
    neg0 = (c == 8)                                                # -0 is coded as +0's magnitude
    np.testing.assert_array_equal(np.where(neg0.T, lo & 7, lo), np.where(neg0.T, 0, c.T))


def test_token_major_gather_ignores_slots_past_kv_len(orc):
    """Slots of the last page past kv_len count as zero, whatever they hold."""
    rng = np.random.default_rng(8)
    H, D, kv = 2, 128, 37
    k = rng.standard_normal((48, H, D)).astype(np.float32)
    v = rng.standard_normal((48, H, D)).astype(np.float32)
    row = np.array([2, 0, 3], np.int32)
    slots = row[np.arange(48) // 16].astype(np.int64) * 16 + np.arange(48) % 16
    full = orc.Pools(4, H)
    orc.kv_append(full, k, v, slots, 0.01, 0.02)                   # slots 37..47 written too
    part = orc.Pools(4, H)
    orc.kv_append(part, k[:kv], v[:kv], slots[:kv], 0.01, 0.02)    # ... or left zero
    for h in range(H):
        a = orc.gather_v_token_major(full, row, kv, h, 0.02)
        b = orc.gather_v_token_major(part, row, kv, h, 0.02)
        np.testing.assert_array_equal(a, b)
        # the first two pages: the page-level re-layout of the decoded slots
        raw = orc.gather_decode(full, "v", row, 32, h, 1.0).astype(np.float32)
        for p in range(2):
            cds, scs = orc.v_token_major_page(raw[16 * p:16 * p + 16])
            np.testing.assert_array_equal(a[16 * p:16 * p + 16], orc.decode_token_major(cds, scs, 0.02))


def test_fp4pv_uniform_scores_give_prefix_means(orc):
    """q = 0: every score is 0, every p is 1, coded as 6 x E4M3(28) x g_p with
    g_p = fl32(16/2688); so causal row i returns 168 g_p times the mean of
    the first i+1 values, and lse = ln(i+1)."""
    rng = np.random.default_rng(3)
    n, D = 40, 32
    v = rng.standard_normal((n, D))
    k = rng.standard_normal((n, D))
    q = np.zeros((n, D))
    o, lse = orc.fp4pv_attention_rows(q, np.arange(n), n, k, v, True, 0.125)
    g_p = float(np.float32(16.0) / np.float32(2688.0))
    want = 168.0 * g_p * np.cumsum(v, axis=0) / np.arange(1, n + 1)[:, None]
    np.testing.assert_allclose(o, want, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(lse, np.log(np.arange(1, n + 1)), rtol=1e-12, atol=1e-14)


def test_fp4pv_one_hot(orc):
    """One key 40 log2 units above the rest: its p is a power of two and
    exact in FP4; every other p codes to 0.  The row returns that key's value
    times 168 g_p and lse = 40 ln 2."""
    rng = np.random.default_rng(4)
    kv, D, star = 300, 16, 137
    score = rng.uniform(-5.0, 0.0, kv)
    score[star] = 40.0
    k = np.zeros((kv, D))
    k[:, 0] = score
    q = np.zeros((1, D))
    q[0, 0] = 1.0
    v = rng.standard_normal((kv, D))
    o, lse = orc.fp4pv_attention_rows(q, np.array([0]), 1, k, v, False, math.log(2.0))
    g_p = float(np.float32(16.0) / np.float32(2688.0))
    np.testing.assert_allclose(o[0], 168.0 * g_p * v[star], rtol=1e-9)
    assert abs(lse[0] - 40.0 * math.log(2.0)) < 1e-9


def _random_case(seed, kv=300, D=128):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((kv, D))
    k = rng.standard_normal((kv, D))
    v = rng.standard_normal((kv, D))
    return q, k, v


def test_fp4pv_close_to_exact_but_quantized(orc):
    """Against the exact attention on the same values.  Each coded p is off by
    at most half the widest E2M1 gap (2) times its block scale, and the block
    scale is amax/6 within E4M3's 2^-4, so |o4 - o|_d <= sum over blocks of
    (17/96) amax_b sum_(j in b) |v_jd| / l, computed here from numpy's exact
    p.  FP4 P is coarse (one mantissa bit): on these normal scores the rows
    move by several per cent, and visibly (above 1e-3), so P is really coded.
    lse is untouched (it uses the unquantized p)."""
    q, k, v = _random_case(11)
    n, sm = q.shape[0], 1 / math.sqrt(128)
    pos = np.arange(0, n, 7)
    o4, l4 = orc.fp4pv_attention_rows(q[pos], pos, n, k, v, True, sm)
    oe, le = orc.attention_rows(q[pos], pos, n, k, v, True, sm)
    for r, i in enumerate(pos):
        s2 = sm * (k[: i + 1] @ q[pos[r]]) / math.log(2.0)
        p = np.exp2(s2 - s2.max())
        nb = -(-(i + 1) // 16)
        pb = np.zeros(nb * 16)
        pb[: i + 1] = p
        vb = np.zeros((nb * 16, v.shape[1]))
        vb[: i + 1] = np.abs(v[: i + 1])
        amax = pb.reshape(nb, 16).max(axis=1)
        bound = (17.0 / 96.0) * (amax[:, None] * vb.reshape(nb, 16, -1).sum(axis=1)).sum(axis=0) / p.sum()
        assert np.all(np.abs(o4[r] - oe[r]) <= bound * (1 + 1e-9) + 1e-12), r
    rel = np.linalg.norm(o4 - oe) / np.linalg.norm(oe)
    assert 1e-3 < rel < 0.2, rel
    np.testing.assert_allclose(l4, le, rtol=1e-12, atol=1e-12)


def _trend_case(kv=600, D=16, seed=2):
    """Scores rising by 12 log2 units across the keys with a little noise, so
    the running reference moves several times."""
    rng = np.random.default_rng(seed)
    k = np.zeros((kv, D))
    k[:, 0] = 0.02 * np.arange(kv) + rng.uniform(-0.5, 0.5, kv)
    k[:, 1:] = rng.standard_normal((kv, D - 1)) * 0.05
    q = np.zeros((4, D))
    q[:, 0] = 1.0
    q[:, 1:] = rng.standard_normal((4, D - 1)) * 0.05
    v = rng.standard_normal((kv, D))
    return q, k, v


def test_fp4pv_independent_of_tiling_and_threshold(orc):
    """X3: references are whole numbers, so changing the tile size or the
    threshold only multiplies each block by a power of two, which the block
    codec carries exactly: the outputs agree to rounding."""
    q, k, v = _trend_case()
    kv = k.shape[0]
    pos = np.array([kv - 1, 450, 300, 130])
    base, lb = orc.fp4pv_attention_rows(q, pos, kv, k, v, True, math.log(2.0), tile=128, tau=4)
    for tile, tau in [(16, 4), (128, 0), (64, 2), (256, 8), (32, 1)]:
        o, lse = orc.fp4pv_attention_rows(q, pos, kv, k, v, True, math.log(2.0), tile=tile, tau=tau)
        np.testing.assert_allclose(o, base, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(lse, lb, rtol=1e-12)


def _one_block_row(orc, s, eps, D=4, seed=6):
    """One non-causal row over len(s) keys whose log2 scores are exactly s."""
    rng = np.random.default_rng(seed)
    kv = len(s)
    k = np.zeros((kv, D))
    k[:, 0] = s
    q = np.zeros((1, D))
    q[0, 0] = 1.0
    v = rng.standard_normal((kv, D))
    return orc.fp4pv_attention_rows(q, np.array([0]), 1, k, v, False, math.log(2.0), eps=eps)


@pytest.mark.parametrize("kind", ["code", "scale"])
def test_fp4pv_slack_covers_a_real_flip(orc, kind):
    """A P value placed just below and just above an E2M1 boundary (2.5, in
    units of its block scale), or a block maximum just below and above an
    E4M3 midpoint (27 between 26 and 28), codes differently on the two sides;
    the slack reported on either side covers the change, and is zero with
    eps = 0 when nothing lies exactly on a boundary."""
    rng = np.random.default_rng(12)
    base = rng.uniform(-3.9, -1.1, 16)
    outs = []
    for sign in (-1.0, 1.0):
        s = base.copy()
        if kind == "code":
            s[0] = 0.0                                              # p = 1: the block scale is 28
            s[5] = math.log2(2.5 / 6.0) + sign * 1e-6               # p * inv = 2.5 (1 +- 7e-7)
        else:
            s[0] = math.log2(27.0 / 28.0) + sign * 1e-6             # amax * 28 = 27 (1 +- 7e-7)
        o, _, sl = _one_block_row(orc, s, eps=1e-5)
        _, _, sl0 = _one_block_row(orc, s, eps=0.0)
        assert not sl0.any()
        outs.append((o[0], sl[0]))
    (o_lo, sl_lo), (o_hi, sl_hi) = outs
    moved = np.abs(o_hi - o_lo)
    assert moved.max() > 1e-3                                       # the decision really flipped
    # (moving the score by 1e-6 also moves that p and l, hence o,
    # continuously by about 1e-6 relative: hence the small allowance on |o|)
    cont = 1e-5 * (np.abs(o_lo) + np.abs(o_hi))
    assert np.all(moved <= sl_lo + cont) and np.all(moved <= sl_hi + cont)


def test_fp4pv_slack_zero_away_from_boundaries(orc):
    """Uniform scores code p = 1 as 6 x E4M3(28), far from every boundary."""
    rng = np.random.default_rng(3)
    n, D = 40, 32
    v = rng.standard_normal((n, D))
    k = rng.standard_normal((n, D))
    _, _, sl = orc.fp4pv_attention_rows(np.zeros((n, D)), np.arange(n), n, k, v, True, 0.125, eps=1e-3)
    assert not sl.any()
