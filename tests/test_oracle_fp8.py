"""Pins of the oracle's FP8 (E4M3) comparison cache.

The pages compare NVFP4 with an 8-bit FP8 cache: one byte per value, scale
metadata kept apart ("NVFP4 KV cache prefill vs decode performance", sections
"NVFP4 stores 4.5 bits per value before padding" and "A worked per-token
cache estimate": FP8 bytes per token = 2 * L * H * D, 131,072 B for L = 64,
H = 8, D = 128).  The element codec is pinned against torch's float8_e4m3fn
cast, an independent library, and by the definition at the edges that torch
does not cover (saturation above 448)."""
import json
import os

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def torch_e4m3(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_fp8_encode_matches_torch_cast(orc):
    """Nearest-even E4M3 of signed values inside the finite range, including
    every tie between neighbouring codes and values around the subnormals."""
    rng = np.random.default_rng(8)
    x = np.concatenate([
        rng.standard_normal(20000) * np.exp(rng.uniform(-8, 5, 20000)),
        rng.uniform(-448, 448, 5000),
    ]).astype(np.float32)
    x = x[np.abs(x) <= 448]
    # every midpoint between consecutive non-negative codes, both signs
    vals = np.array([orc.e4m3_value(b) for b in range(0x7F)])
    mids = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)
    x = np.concatenate([x, mids, -mids, np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(1e9))])
    np.testing.assert_array_equal(orc.fp8_encode_array(x), torch_e4m3(x))


def test_fp8_saturation_and_signed_zero(orc):
    """Above 448 the code saturates at +-448 (0x7E / 0xFE), never NaN; a tiny
    negative value keeps its sign (0x80, which decodes to -0 == 0)."""
    codes = orc.fp8_encode_array([448.0, 465.0, 1e6, -3e38, -1e-6, 1e-6])
    assert list(codes) == [0x7E, 0x7E, 0x7E, 0xFE, 0x80, 0x00]
    assert orc.e4m3_value(0x80) == 0.0


def test_fp8_quantize_uses_the_reciprocal_of_the_scale(orc):
    """code = E4M3(fl32(x * fl32(1/g))) (reading F2), not E4M3(fl32(x / g)):
    near the ties of the code grid the two readings differ, and the oracle
    must give torch's cast of the product every time."""
    g = np.float32(0.7)
    inv = np.float32(np.float32(1.0) / g)
    vals = np.array([orc.e4m3_value(b) for b in range(0x7F)])
    mids = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)
    xs = []
    for m in mids[1:]:
        x = np.float32(m * g)
        for _ in range(3):
            xs += [x, np.nextafter(x, np.float32(0)), np.nextafter(x, np.float32(1e9))]
            x = np.nextafter(x, np.float32(1e9))
    xs = np.array(xs, np.float32)
    by_mul = torch_e4m3((xs * inv).astype(np.float32))
    by_div = torch_e4m3((xs / g).astype(np.float32))
    assert np.count_nonzero(by_mul != by_div) >= 5          # the readings are distinguishable here
    np.testing.assert_array_equal(orc.fp8_quantize(xs, float(g)), by_mul)


def test_fp8_round_trip_and_error_bound(orc):
    """Values that are exactly e4m3 x g come back unchanged; others land
    within half a unit in the last place (3 mantissa bits: 2^-4 relative for
    normal values)."""
    g = 0.03125
    codes = np.array([b for b in range(256) if (b & 0x7F) != 0x7F], np.uint8)
    x = np.array([orc.e4m3_value(int(b)) * g for b in codes], np.float32)
    np.testing.assert_array_equal(orc.fp8_quantize(x, g) & 0x7F, codes & 0x7F)
    rng = np.random.default_rng(3)
    y = (rng.standard_normal(4000) * 3).astype(np.float32)
    gy = float(np.float32(np.abs(y).max() / 448))
    dec = np.array([orc.e4m3_value(int(b)) for b in orc.fp8_quantize(y, gy)]) * gy
    normal = np.abs(y) >= gy * 2.0 ** -6
    assert np.all(np.abs(dec - y)[normal] <= np.abs(y)[normal] * 2.0 ** -4 * (1 + 1e-6))


def test_fp8_cache_bytes_worked_example(orc):
    """The pages' per-token FP8 figure: 2 * 64 layers * 8 heads * 128 dims =
    131,072 bytes."""
    g = json.load(open(os.path.join(GOLDEN, "accounting.json")))
    w = g["worked_per_token_L64"]
    assert w["layers"] * orc.fp8_cache_bytes(1, 1, w["kv_heads"], w["head_dim"]) == w["fp8_bytes_per_token"]
    assert orc.fp8_cache_bytes(10, 16, 8, 128) == 10 * 16 * 8 * 256


def test_fp8_append_layout_and_skips(orc):
    """Token t's codes land in its slot's row (page, head, offset); negative
    slots are skipped; an out-of-range slot is refused."""
    rng = np.random.default_rng(4)
    T, H, D = 40, 2, 128
    k = rng.standard_normal((T, H, D)).astype(np.float32)
    v = rng.standard_normal((T, H, D)).astype(np.float32)
    slots = rng.permutation(4 * 16)[:T].astype(np.int64)
    slots[5] = -1
    pools = orc.FP8Pools(4, H, fill=0xAB)
    orc.fp8_kv_append(pools, k, v, slots, 0.01, 0.02)
    for t in (0, 5, 17, 39):
        p, o = divmod(int(slots[t]), 16)
        for h in range(H):
            if slots[t] < 0:
                continue
            np.testing.assert_array_equal(pools.k_data[p, h, o], orc.fp8_quantize(k[t, h], 0.01))
            np.testing.assert_array_equal(pools.v_data[p, h, o], orc.fp8_quantize(v[t, h], 0.02))
    written = {int(s) for s in slots if s >= 0}
    untouched = [s for s in range(64) if s not in written]
    assert all(np.all(pools.k_data[s // 16, :, s % 16] == 0xAB) for s in untouched)
    bad = slots.copy()
    bad[0] = 64
    with pytest.raises(ValueError):
        orc.fp8_kv_append(orc.FP8Pools(4, H), k, v, bad, 0.01, 0.02)


def test_fp8_paged_attention_equals_dense_on_decoded_values(orc):
    """Attention over the paged FP8 cache equals attention over the decoded
    values laid out densely (the paging changes nothing)."""
    rng = np.random.default_rng(9)
    H, Hq, D, kv = 2, 4, 128, 37
    k = rng.standard_normal((kv, H, D)).astype(np.float32)
    v = rng.standard_normal((kv, H, D)).astype(np.float32)
    q = rng.standard_normal((5, Hq, D)).astype(np.float32)
    pt = rng.permutation(4).astype(np.int32)[None, :3]
    slots = (pt[0][np.arange(kv) // 16].astype(np.int64) * 16 + np.arange(kv) % 16)
    pools = orc.FP8Pools(4, H)
    orc.fp8_kv_append(pools, k, v, slots, 0.01, 0.02)
    ref = orc.paged_attention(pools, q, [0, 5], [kv], pt, Hq, 0.01, 0.02, True, 0.09)
    for h in range(H):
        kd = np.array([[orc.e4m3_value(int(b)) for b in orc.fp8_quantize(k[j, h], 0.01)] for j in range(kv)]) * np.float32(0.01)
        vd = np.array([[orc.e4m3_value(int(b)) for b in orc.fp8_quantize(v[j, h], 0.02)] for j in range(kv)]) * np.float32(0.02)
        for gq in range(2):
            o, lse = orc.attention_rows(q[:, 2 * h + gq].astype(np.float64), np.arange(5), 5, kd, vd, True, 0.09)
            for i in range(5):
                np.testing.assert_allclose(ref[(0, i)][0][2 * h + gq], o[i], rtol=1e-12, atol=1e-12)
