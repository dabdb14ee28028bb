"""The pins catch plausible mistakes.  Each test plants one mistake in the
oracle -- on the CPU, through a proxy that replaces a single oracle function
with a wrong variant -- and checks that the pin written for that part of the
oracle fails on it.  (The formats and rules are those of "NVFP4 KV cache vs
NVFP4 weights", section "NVFP4 KV cache vs NVFP4 weights", and "NVFP4 KV
cache A4Q prefill explained", section "Quantize Q instead of expanding K".)"""
import math

import numpy as np
import pytest

from . import test_oracle_attention as A
from . import test_oracle_codec as C
from . import test_oracle_formats as F

E2M1_MAGS = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


class Mutant:
    """The oracle with some functions replaced."""

    def __init__(self, base, **replaced):
        self._base = base
        self.__dict__.update(replaced)

    def __getattr__(self, name):
        return getattr(self._base, name)


def _fails(pin, *args):
    with pytest.raises(AssertionError):
        pin(*args)


def test_e2m1_ties_away_from_zero_is_caught(orc):
    def ties_away(x):
        sign = 8 if math.copysign(1.0, x) < 0 else 0
        a = min(abs(x), 6.0)
        code = min(range(8), key=lambda c: (abs(E2M1_MAGS[c] - a), -E2M1_MAGS[c]))
        return code | sign

    _fails(F.test_e2m1_tie_rules, Mutant(orc, e2m1_encode=ties_away))


def test_e4m3_truncation_is_caught(orc):
    vals = np.array([orc.e4m3_value(b) for b in range(127)])

    def truncate(x):
        x = np.minimum(np.asarray(x, np.float64), 448.0)
        return np.array([int(np.nonzero(vals <= xi)[0].max()) for xi in x], np.uint8)

    _fails(F.test_e4m3_encode_rne_vs_torch_cast, Mutant(orc, e4m3_encode_array=truncate))


def test_e2m1_exponent_bias_is_caught(orc):
    def bias0(code):
        s, e, m = (code >> 3) & 1, (code >> 1) & 3, code & 1
        mag = float(m) if e == 0 else 2.0 ** e * (1 + 0.5 * m)
        return -mag if s else mag

    _fails(F.test_e2m1_decode_all_codes, Mutant(orc, e2m1_value=bias0))


def test_swapped_nibble_order_is_caught(orc):
    def swapped(x, g):
        packed, scale = orc.quantize_block16(x, g)
        packed = np.asarray(packed, np.uint8)
        return ((packed >> 4) | (packed << 4)).astype(np.uint8), scale

    _fails(C.test_hand_worked_blocks, Mutant(orc, quantize_block16=swapped))


def test_dropped_factor_six_in_the_scale_is_caught(orc):
    def no_six(x, g):
        return orc.quantize_block16(x, g / 6.0)

    _fails(C.test_round_trip_codes_and_scales, Mutant(orc, quantize_block16=no_six), 1.0)


def test_top_left_causal_alignment_is_caught(orc):
    def top_left(q, pos, q_len, k, v, causal, sm_scale):
        return orc.attention_rows(q, pos, len(k), k, v, causal, sm_scale)

    _fails(A.test_attention_vs_library, Mutant(orc, attention_rows=top_left), 5, 19, True)


def test_dropped_softmax_scale_is_caught(orc):
    def unscaled(q, pos, q_len, k, v, causal, sm_scale):
        return orc.attention_rows(q, pos, q_len, k, v, causal, 1.0)

    _fails(A.test_attention_vs_library, Mutant(orc, attention_rows=unscaled), 9, 33, False)


def test_division_instead_of_reciprocal_is_caught(orc):
    """Codes taken from fl32(x / fl32(g * s)) instead of x times the rounded
    reciprocal: the hand-worked block with a non-power-of-two scale differs."""
    def divided(x, g):
        x = np.asarray(x, np.float32)
        g = np.float32(g)
        amax = np.float32(np.abs(x).max())
        s_real = np.float32(amax / np.float32(np.float32(6.0) * g)) if amax > 0 else np.float32(0.0)
        scale = orc.e4m3_encode(s_real)
        d = np.float32(g * np.float32(orc.e4m3_value(scale)))
        codes = [0] * 16 if d == 0 else [orc.e2m1_encode(np.float32(xi / d)) for xi in x]
        packed = np.array([codes[2 * i] | (codes[2 * i + 1] << 4) for i in range(8)], np.uint8)
        return packed, scale

    _fails(C.test_hand_worked_blocks, Mutant(orc, quantize_block16=divided))


def test_fp8_truncation_and_dropped_sign_are_caught(orc):
    """An FP8 element encoder that truncates toward zero, or one that drops
    the sign, fails the pin against torch's float8_e4m3fn cast."""
    from . import test_oracle_fp8 as P8
    vals = np.array([orc.e4m3_value(b) for b in range(0x7F)])

    def truncate(x):
        x = np.asarray(x, np.float32).ravel()
        mag = np.array([int(np.nonzero(vals <= min(abs(float(xi)), 448.0))[0].max()) for xi in x], np.uint8)
        return mag | np.where(np.signbit(x), 0x80, 0).astype(np.uint8)

    def unsigned(x):
        return orc.fp8_encode_array(np.abs(np.asarray(x, np.float32)))

    _fails(P8.test_fp8_encode_matches_torch_cast, Mutant(orc, fp8_encode_array=truncate))
    _fails(P8.test_fp8_encode_matches_torch_cast, Mutant(orc, fp8_encode_array=unsigned))


def _fp4pv_rows(orc, ceil_ref=True, weight=True):
    """X2..X5 written out in numpy on the oracle's block codec, with one step
    that can be planted wrong: a fractional reference (no ceil), or the
    2^(m_t - m_end) weight of earlier tiles dropped."""
    def rows(q, pos, q_len, k, vhat, causal, sm_scale, tile=128, tau=4):
        g_p = orc.fp4pv_p_scale(tau)
        e2m1 = np.array([orc.e2m1_value(c) for c in range(16)])
        out, lse = np.zeros((len(pos), k.shape[1])), np.zeros(len(pos))
        for r, i in enumerate(pos):
            last = k.shape[0] - q_len + int(i) if causal else k.shape[0] - 1
            s = sm_scale * (k[: last + 1] @ q[r]) / math.log(2.0)
            m, refs = -math.inf, []
            for t in range(last // tile + 1):
                mt = s[t * tile:(t + 1) * tile].max()
                if mt > m + tau:
                    m = math.ceil(mt) if ceil_ref else mt
                refs.append(m)
            l = np.exp2(s - m).sum()
            o = np.zeros(k.shape[1])
            for b0 in range(0, last + 1, 16):
                n = min(16, last + 1 - b0)
                p = np.zeros(16, np.float32)
                p[:n] = np.exp2(s[b0:b0 + n] - refs[b0 // tile])
                packed, sc = orc.quantize_block16(p, g_p)
                codes = np.stack([packed & 15, packed >> 4], axis=1).ravel()[:n]
                w = (2.0 ** (refs[b0 // tile] - m) if weight else 1.0) * orc.e4m3_value(sc) * g_p
                o += (w * e2m1[codes]) @ vhat[b0:b0 + n]
            out[r], lse[r] = o / l, (m + math.log2(l)) * math.log(2.0)
        return out, lse
    return rows


def test_fp4pv_planted_mistakes_are_caught(orc):
    """FP4 PV (readings X1..X5): an unquantized P, a fractional reference, a
    dropped weight of earlier tiles, and a V re-layout that keeps the cache's
    own axis each fail their pin."""
    from . import test_oracle_fp4pv as P4
    # the numpy restatement passes the pins it is planted into
    P4.test_fp4pv_independent_of_tiling_and_threshold(Mutant(orc, fp4pv_attention_rows=_fp4pv_rows(orc)))

    def unquantized(q, pos, q_len, k, vhat, causal, sm_scale, tile=128, tau=4):
        return orc.attention_rows(q, pos, q_len, k, vhat, causal, sm_scale)

    _fails(P4.test_fp4pv_close_to_exact_but_quantized, Mutant(orc, fp4pv_attention_rows=unquantized))
    _fails(P4.test_fp4pv_independent_of_tiling_and_threshold,
           Mutant(orc, fp4pv_attention_rows=_fp4pv_rows(orc, ceil_ref=False)))
    _fails(P4.test_fp4pv_independent_of_tiling_and_threshold,
           Mutant(orc, fp4pv_attention_rows=_fp4pv_rows(orc, weight=False)))

    def cache_axis(x16):
        """Blocks along the head dimension of each slot (the cache's axis),
        codes then read out per dimension: the scale of dimension d is that of
        slot 0's block holding d."""
        x = np.asarray(x16, np.float32)
        packed, scales, _ = orc.quantize_rows(x, orc.GLOBAL, 1.0)     # [16, D/2], [16, D/16]
        D = x.shape[1]
        nib = np.stack([packed & 15, packed >> 4], axis=2).reshape(16, D)  # [slot, d]
        codes = (nib[0::2].T | (nib[1::2].T << 4)).astype(np.uint8)       # [D, 8]
        return codes, scales[0][np.arange(D) // 16].astype(np.uint8)

    _fails(P4.test_token_major_scales_follow_tokens, Mutant(orc, v_token_major_page=cache_axis))
    _fails(P4.test_token_major_round_trip_on_grid, Mutant(orc, v_token_major_page=cache_axis))
