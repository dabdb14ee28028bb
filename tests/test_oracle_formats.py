"""Pins of the oracle's number formats against the format definitions and an
independent library cast (not against the oracle itself).

Formats: 4-bit E2M1 values and one E4M3 scale per 16 values ("NVFP4 KV cache
vs NVFP4 weights", section "NVFP4 KV cache vs NVFP4 weights"; "NVFP4 KV cache
prefill vs decode performance", section "NVFP4 stores 4.5 bits per value
before padding")."""
import numpy as np
import pytest
import torch


def e2m1_from_bits(code):
    """E2M1 from its bit fields: sign | 2-bit exponent (bias 1) | 1-bit mantissa."""
    s, e, m = (code >> 3) & 1, (code >> 1) & 3, code & 1
    mag = 0.5 * m if e == 0 else 2.0 ** (e - 1) * (1 + 0.5 * m)
    return -mag if s else mag


def test_e2m1_decode_all_codes(orc):
    for c in range(16):
        assert orc.e2m1_value(c) == e2m1_from_bits(c)
    mags = sorted({abs(e2m1_from_bits(c)) for c in range(16)})
    assert mags == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e4m3_decode_all_bytes_vs_torch(orc):
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    for b in range(256):
        v = orc.e4m3_value(b)
        if np.isnan(ref[b]):
            assert np.isnan(v), b
        else:
            assert v == ref[b], (b, v, ref[b])
    assert orc.e4m3_value(0x7E) == 448.0  # the max finite value


def _e4m3_sample():
    vals = torch.arange(0, 127, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    mids = (vals[1:] + vals[:-1]) / 2
    pts = [vals, mids]
    for m in mids:
        f = np.float32(m)
        pts.append(np.array([np.nextafter(f, np.float32(0)), np.nextafter(f, np.float32(1e9))], np.float64))
    rng = np.random.default_rng(0)
    pts.append(np.exp(rng.uniform(np.log(1e-4), np.log(448), 20000)))
    pts.append(rng.uniform(0, 2.0 ** -6, 5000))
    x = np.concatenate(pts).astype(np.float32)
    return x[(x >= 0) & (x <= 448)]


def test_e4m3_encode_rne_vs_torch_cast(orc):
    x = _e4m3_sample()
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = orc.e4m3_encode_array(x)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(float(x[i]), int(got[i]), int(ref[i])) for i in bad[:10]]


def test_e4m3_encode_saturates(orc):
    # Reading R1: saturating conversion -- anything above 448 stores 448.
    for x in [448.0, 449.0, 464.0, 500.0, 1e6, 3.0e38]:
        assert orc.e4m3_encode(x) == 0x7E


def e2m1_rne_grid(q):
    """E2M1 round-to-nearest-even on each binade's uniform grid via np.rint
    (half to even): spacing 0.5 below 2, 1 in [2,4), 2 from 4; saturate at 6.
    Returns codes (sign bit kept)."""
    a = np.abs(q.astype(np.float64))
    r = np.where(a < 2, np.rint(a * 2) / 2, np.where(a < 4, np.rint(a), 2 * np.rint(a / 2)))
    r = np.minimum(r, 6.0)
    table = {0.0: 0, 0.5: 1, 1.0: 2, 1.5: 3, 2.0: 4, 3.0: 5, 4.0: 6, 6.0: 7}
    mag = np.array([table[v] for v in r], np.uint8)
    return mag | (np.signbit(q).astype(np.uint8) << 3)


def test_e2m1_encode_vs_grid_rounding(orc):
    rng = np.random.default_rng(1)
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0, 7.0], np.float32)
    pts = [mids, -mids]
    for m in mids:
        pts.append(np.array([np.nextafter(m, np.float32(0)), np.nextafter(m, np.float32(9))], np.float32))
    pts.append(rng.uniform(-8, 8, 50000).astype(np.float32))
    pts.append(np.array([0.0, -0.0, 1e-30, -1e-30, 100.0, -100.0, 1e30, -3e38], np.float32))
    q = np.concatenate(pts).astype(np.float32)
    got = orc.e2m1_encode_array(q)
    ref = e2m1_rne_grid(q)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(float(q[i]), int(got[i]), int(ref[i])) for i in bad[:10]]


_E2M1_GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], np.float32)


def e2m1_rne_grid_fast(q):
    """The same grid rounding as e2m1_rne_grid, vectorized: every step is exact
    in fp32 for |q| < 8 (doubling, rint, halving), and the rounded magnitude
    is one of the eight grid values, whose index is its code."""
    a = np.abs(q)
    r = np.where(a < 2, np.rint(a * 2) / 2, np.where(a < 4, np.rint(a), 2 * np.rint(a / 2)))
    r = np.minimum(r, np.float32(6.0)).astype(np.float32)
    code = np.searchsorted(_E2M1_GRID, r).astype(np.uint8)
    assert np.array_equal(_E2M1_GRID[code], r)
    return code | (np.signbit(q).astype(np.uint8) << 3)


def test_e2m1_encode_every_fp32_in_decision_range(orc):
    """Every fp32 value in [0.125, 8), both signs (about 10^8 inputs), against
    the grid rounding.  These binades hold every rounding threshold (0.25 ...
    5) and the saturation point 6; below 0.125 every value is nearer to 0 than
    to 0.5, and from 8 up every value saturates, which the sampled checks
    below and the tie test cover."""
    lo = int(np.float32(0.125).view(np.uint32))
    hi = int(np.float32(8.0).view(np.uint32))
    step = 1 << 23
    for sign in (0, 1 << 31):
        for start in range(lo, hi, step):
            bits = np.arange(start, min(start + step, hi), dtype=np.uint32) | np.uint32(sign)
            q = bits.view(np.float32)
            got = orc.e2m1_encode_array(q)
            ref = e2m1_rne_grid_fast(q)
            bad = np.nonzero(got != ref)[0]
            assert bad.size == 0, [(float(q[i]), int(got[i]), int(ref[i])) for i in bad[:10]]


def test_e2m1_encode_outside_decision_range(orc):
    """Below 0.125 (down to the smallest subnormal) the code is +-0; from 8 up
    (through the largest finite value and infinity) it is +-6."""
    rng = np.random.default_rng(2)
    tiny = np.concatenate([np.exp2(rng.uniform(-149, -3, 200000)).astype(np.float32),
                           np.array([0.0, np.nextafter(np.float32(0.125), np.float32(0)), 1.4e-45], np.float32)])
    big = np.concatenate([np.exp2(rng.uniform(3, 127.9, 200000)).astype(np.float32),
                          np.array([8.0, np.finfo(np.float32).max, np.inf], np.float32)])
    for q, code in ((tiny, 0), (big, 7)):
        assert np.all(orc.e2m1_encode_array(q) == code)
        assert np.all(orc.e2m1_encode_array(-q) == (code | 8))


def test_e2m1_tie_rules(orc):
    # ties go to the even code: .25->0, .75->1.0, 1.25->1.0, 1.75->2, 2.5->2, 3.5->4, 5->4
    expect = {0.25: 0, 0.75: 2, 1.25: 2, 1.75: 4, 2.5: 4, 3.5: 6, 5.0: 6, 6.0: 7, 9.0: 7}
    for x, c in expect.items():
        assert orc.e2m1_encode(x) == c, x
        assert orc.e2m1_encode(-x) == (c | 8), -x


def test_e2m1_sign_of_zero_reading(orc):
    # Reading R2: the sign of q is kept, so small negatives give code 0x8 (-0).
    assert orc.e2m1_encode(-0.1) == 0x8
    assert orc.e2m1_encode(0.1) == 0x0
    assert orc.e2m1_value(0x8) == 0.0
