"""Pins of the oracle's block codec, cache write and Q scheme.

Round trips, hand-worked blocks (tests/golden/codec_examples.json), the
amax-induced scale property and the rounding error bound.  The cache write
follows "NVFP4 KV cache prefill vs decode performance", section "NVFP4 stores
4.5 bits per value before padding" (quantize, choose block scales, pack FP4,
write scales, map into paged slots)."""
import json
import os

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

E4M3_NONZERO = np.arange(1, 0x7F, dtype=np.uint8)


def test_hand_worked_blocks(orc):
    d = json.load(open(os.path.join(GOLDEN, "codec_examples.json")))
    for blk in d["blocks"]:
        packed, scale = orc.quantize_block16(blk["x"], blk["g"])
        assert scale == blk["scale"], blk["why"]
        assert list(map(int, packed)) == blk["packed"], blk["why"]


@pytest.mark.parametrize("g", [1.0, 0.75, 2.0 ** -12, 3 * 2.0 ** -7, 64.0])
def test_round_trip_codes_and_scales(orc, g):
    """decode(codes, s, g) with one |code| = 6 re-encodes to (codes, s): the
    scale is amax-induced, and with g of few significant bits every product and
    quotient is exact, so any error in the scale formula, the divisor or the
    rounding shows up as a changed byte."""
    rng = np.random.default_rng(int(g * 1000) % 97)
    scales = [int(s) for s in E4M3_NONZERO[::5]] + [0x01, 0x08, 0x38, 0x7E]
    for s in scales:
        sdec = orc.e4m3_value(s)
        for trial in range(6):
            codes = rng.integers(0, 16, 16).astype(np.uint8)
            codes[rng.integers(0, 16)] = 7 if trial % 2 == 0 else 15  # |x| = 6*s*g
            x = np.array([orc.e2m1_value(c) * sdec * g for c in codes], np.float64)
            x32 = x.astype(np.float32)
            assert np.all(x32.astype(np.float64) == x)  # exact in fp32
            packed, scale = orc.quantize_block16(x32, g)
            assert scale == s, (s, g)
            got = np.empty(16, np.uint8)
            got[0::2] = packed & 15
            got[1::2] = packed >> 4
            # -0.0 inputs re-encode as code 8, +0 as code 0: compare exactly
            assert np.array_equal(got, codes), (s, g, codes, got)


def test_block_max_gets_code_six(orc):
    """With a normal E4M3 scale (s >= 2^-6) the largest element of a block is
    encoded as +-6: the scale is amax/6 relative to g (a scale rule based on
    another divisor would move it)."""
    rng = np.random.default_rng(5)
    for _ in range(3000):
        g = float(np.float32(np.exp(rng.uniform(np.log(1e-3), np.log(10)))))
        x = (rng.standard_normal(16) * np.exp(rng.uniform(-3, 3))).astype(np.float32)
        packed, scale = orc.quantize_block16(x, g)
        if orc.e4m3_value(scale) < 2.0 ** -6:
            continue
        codes = np.empty(16, np.uint8)
        codes[0::2] = packed & 15
        codes[1::2] = packed >> 4
        i = int(np.argmax(np.abs(x)))
        assert codes[i] & 7 == 7, (x, g, scale, codes)


def test_rounding_error_bound(orc):
    """|x - decode| is at most half the E2M1 grid step at q = x/(g*s), scaled
    by g*s, except where q saturates at 6."""
    rng = np.random.default_rng(7)
    x = (rng.standard_normal((400, 128)) * np.exp(rng.uniform(-4, 4, (400, 1)))).astype(np.float32)
    g = float(np.float32(np.abs(x).max() / 2688.0))
    packed, scales, _ = orc.quantize_rows(x, orc.GLOBAL, g)
    xd = orc.dequantize_rows(packed, scales, g=g)
    s = np.repeat(np.array([[orc.e4m3_value(b) for b in row] for row in scales]), 16, axis=1)
    unit = g * s
    q = np.abs(x.astype(np.float64)) / np.where(unit > 0, unit, 1)
    step = np.where(q < 2, 0.5, np.where(q < 4, 1.0, 2.0))
    bound = np.where(q > 6, (q - 6) * unit, 0.5 * step * unit) * (1 + 1e-6) + 1e-30
    err = np.abs(x - xd)
    zero_blocks = np.repeat(s == 0, 1, axis=1)
    ok = (err <= bound) | zero_blocks
    assert ok.all()


def test_zero_and_tiny_blocks(orc):
    packed, scale = orc.quantize_block16(np.zeros(16), 1.0)
    assert scale == 0 and not packed.any()
    # amax/6 far below the smallest E4M3 subnormal (2^-9): scale 0, codes 0 (R3)
    x = np.full(16, -1e-6, np.float32)
    packed, scale = orc.quantize_block16(x, 1.0)
    assert scale == 0 and not packed.any()


def test_per_row_q_scheme(orc):
    """R6 (the A4Q Q scheme is left open by the pages): per-row scale
    amax/2688, then the block codec.  Pinned to its reading only: the row's
    largest block gets scale 448 and the row decodes within the bound."""
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((64, 128)) * 3).astype(np.float32)
    x[5] = 0
    packed, scales, row_g = orc.quantize_rows(x, orc.PER_ROW)
    assert row_g[5] == 0 and not packed[5].any() and not scales[5].any()
    for r in range(64):
        if r == 5:
            continue
        assert row_g[r] == np.float32(np.abs(x[r]).max() / np.float32(2688.0))
        blk = int(np.argmax(np.abs(x[r]))) // 16
        assert scales[r, blk] == 0x7E
    xd = orc.dequantize_rows(packed, scales, row_g=row_g)
    rel = np.abs(xd - x).max(axis=1) / np.maximum(np.abs(x).max(axis=1), 1e-30)
    assert rel.max() < 0.25


def test_append_layout_and_skip(orc):
    """A token written at slot s lands at page s//16, offset s%16 of the
    [page][head][16][64] data and [page][head][16][8] scale pools; slot -1 is
    skipped; the bytes equal the direct row quantization."""
    rng = np.random.default_rng(11)
    T, Hkv, D = 40, 2, 128
    pools = orc.Pools(num_pages=6, Hkv=Hkv, D=D)
    k = rng.standard_normal((T, Hkv, D)).astype(np.float32)
    v = rng.standard_normal((T, Hkv, D)).astype(np.float32)
    slots = rng.permutation(6 * 16)[:T].astype(np.int64)
    slots[3] = -1
    kg, vg = 0.01, 0.02
    orc.kv_append(pools, k, v, slots, kg, vg)
    for t in range(T):
        s = slots[t]
        for h in range(Hkv):
            if s < 0:
                continue
            p_, s_, _ = orc.quantize_rows(k[t, h][None], orc.GLOBAL, kg)
            assert np.array_equal(pools.k_data[s // 16, h, s % 16], p_[0])
            assert np.array_equal(pools.k_scale[s // 16, h, s % 16], s_[0])
            p_, s_, _ = orc.quantize_rows(v[t, h][None], orc.GLOBAL, vg)
            assert np.array_equal(pools.v_data[s // 16, h, s % 16], p_[0])
    # nothing was written for the skipped token: untouched slots stay zero
    written = np.zeros(6 * 16, bool)
    written[slots[slots >= 0]] = True
    flat = pools.k_data.transpose(0, 2, 1, 3).reshape(6 * 16, -1)
    assert not flat[~written].any()
    with pytest.raises(ValueError):
        orc.kv_append(pools, k[:1], v[:1], np.array([6 * 16], np.int64), kg, vg)


@pytest.mark.parametrize("q_scale", [1.0, 0.375])
def test_single_scale_query_round_trip(orc, q_scale):
    """The A4Q query with one caller-given scale for every row (per-tensor or
    single-level scheme): values that are exactly code x E4M3 scale x q_scale,
    with one |code| = 6 per 16-value block, come back unchanged."""
    rng = np.random.default_rng(int(q_scale * 64))
    rows = []
    for _ in range(12):
        row = []
        for blk in range(8):
            s = orc.e4m3_value(int(rng.integers(0x20, 0x60)))
            codes = rng.integers(0, 16, 16)
            codes[rng.integers(0, 16)] = 7
            row += [orc.e2m1_value(int(c)) * s * q_scale for c in codes]
        rows.append(row)
    x = np.array(rows, np.float64)
    assert np.all(x.astype(np.float32).astype(np.float64) == x)
    got = orc.decode_q_a4q(x.astype(np.float32), q_scale)
    np.testing.assert_array_equal(got, x)
    # the per-row scheme on the same rows differs (its scale is amax/2688)
    assert not np.array_equal(orc.decode_q_a4q(x.astype(np.float32)), x)
