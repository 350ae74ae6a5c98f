"""Pins for the oracle's q8_0 quantiser and f16 rounding (no GPU).

None of these re-runs the oracle's own formula: the codes are checked against
a brute-force search over all 255 int8 codes in exact arithmetic, the scales
against hand-computed fp16 bit patterns, ties against hand-built blocks.
"""

import numpy as np
import pytest

from oracle import q8_0


def f16_bits(a):
    return np.asarray(a, dtype=np.float16).view(np.uint16)


def brute_force_codes(x, d):
    """argmin_k |x - d*k| over k in [-127, 127], ties to the code farther from zero.

    Exact: x and d are float32, so d*k and x - d*k are exact in float64.
    """
    ks = np.arange(-127, 128, dtype=np.float64)
    err = np.abs(x.astype(np.float64)[..., None] - d.astype(np.float64)[..., None, None] * ks)
    tie = err == err.min(axis=-1, keepdims=True)
    return ks[np.argmax(np.where(tie, np.abs(ks), -1.0), axis=-1)]


def test_codes_match_brute_force_search():
    rng = np.random.default_rng(7)
    x = (rng.standard_normal((1500, 32)) * rng.choice([1e-3, 1.0, 4.0, 300.0], size=(1500, 1))).astype(np.float32)
    d_h, q = q8_0.quantize_blocks(x)
    amax = np.abs(x).max(axis=1)
    d = (amax / np.float32(127)).astype(np.float32)
    bf = brute_force_codes(x, d)
    # the method divides in float32; where the exact ratio lies within one float32 ulp of a
    # half-integer that rounding may pick the neighbour, so only those elements may differ
    ratio = x.astype(np.float64) / d.astype(np.float64)[:, None]
    frac = np.abs(np.abs(ratio) - np.floor(np.abs(ratio)) - 0.5)
    near_tie = frac <= np.spacing(np.abs(ratio).astype(np.float32)).astype(np.float64)
    mismatch = (q.astype(np.float64) != bf) & ~near_tie
    assert not mismatch.any()
    assert (np.abs(q.astype(np.int64) - bf) <= 1).all()


def test_scale_hand_values():
    # amax 127 -> d = 1 -> fp16 0x3C00;  amax 1 -> d = 1/127 = 1.00787...*2^-7 -> mantissa 1032/1024 -> 0x2008
    # amax 63.5 -> d = 0.5 -> 0x3800;  amax 15.875 -> d = 0.125 -> 0x3000
    for amax, bits in [(127.0, 0x3C00), (1.0, 0x2008), (63.5, 0x3800), (15.875, 0x3000)]:
        x = np.zeros(32, np.float32)
        x[5] = -amax
        d_h, q = q8_0.quantize_blocks(x)
        assert int(f16_bits(d_h)[0]) == bits
        assert int(q[5]) == -127


def test_subnormal_scales_round_to_nearest_even():
    # d = 2^-20 = 16 * 2^-24 -> subnormal 0x0010
    # d = 2^-25 = half the smallest subnormal -> tie -> even -> +0
    # d = 3 * 2^-25 = 1.5 smallest subnormals -> tie between 1 and 2 -> even -> 0x0002
    for d, bits in [(2.0 ** -20, 0x0010), (2.0 ** -25, 0x0000), (3 * 2.0 ** -25, 0x0002)]:
        x = np.zeros(32, np.float32)
        x[0] = np.float32(127 * d)
        assert float(np.float32(127 * d)) == 127 * d
        d_h, q = q8_0.quantize_blocks(x)
        assert int(f16_bits(d_h)[0]) == bits
        assert int(q[0]) == 127


def test_ties_round_away_from_zero():
    # amax 15.875 -> d = 0.125 exactly; x = (k + 1/2) * d gives exact half-integer ratios
    x = np.zeros(32, np.float32)
    x[0] = 15.875
    x[1:9] = np.array([0.0625, -0.0625, 0.1875, -0.1875, 0.3125, -0.3125, 15.8125, -15.8125], np.float32)
    _, q = q8_0.quantize_blocks(x)
    assert q[:9].tolist() == [127, 1, -1, 2, -2, 3, -3, 127, -127]


def test_zero_block_and_exact_multiples():
    x = np.zeros((2, 32), np.float32)
    x[1] = np.arange(-16, 16, dtype=np.float32)
    x[1, 0] = -127.0                       # amax 127 -> d = 1 -> the codes are the values
    d_h, q = q8_0.quantize_blocks(x)
    assert (q[0] == 0).all() and int(f16_bits(d_h[0, 0])) == 0
    assert q[1].tolist() == x[1].astype(np.int64).tolist()
    assert int(f16_bits(d_h[1, 0])) == 0x3C00


def test_reconstruction_bound_and_exact_dequantisation():
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((2000, 128)) * 3).astype(np.float32)
    d_h, q = q8_0.quantize_blocks(x)
    xh = q8_0.dequantize_blocks(d_h, q)
    # dequantisation is exact in float32: equals the float64 product
    exact = d_h.astype(np.float64)[..., None] * q.reshape(2000, 4, 32).astype(np.float64)
    assert (xh.reshape(2000, 4, 32).astype(np.float64) == exact).all()
    xb = x.reshape(2000, 4, 32).astype(np.float64)
    d = (np.abs(x.reshape(2000, 4, 32)).max(-1) / np.float32(127)).astype(np.float64)
    bound = d / 2 * (1 + 1e-6) + 127 * np.abs(d - d_h.astype(np.float64))
    assert (np.abs(xb - exact) <= bound[..., None]).all()
    # the element holding amax is coded +-127
    i = np.abs(x.reshape(2000, 4, 32)).argmax(-1)
    assert (np.abs(np.take_along_axis(q.reshape(2000, 4, 32), i[..., None], -1)) == 127).all()


def test_f16_rounding_hand_values():
    vals = np.array([1.0, -2.0, 0.5, 65504.0, 2.0 ** -24, 1.0 / 3.0, -0.0, 0.1,
                     1 + 2.0 ** -11, 1 + 3 * 2.0 ** -11], np.float32)
    bits = [0x3C00, 0xC000, 0x3800, 0x7BFF, 0x0001, 0x3555, 0x8000, 0x2E66, 0x3C00, 0x3C02]
    assert f16_bits(q8_0.to_f16(vals)).tolist() == bits


def test_underflowing_scale_codes_zero():
    # amax = 2^-144 = 32 * 2^-149: amax/127 rounds to float32 zero, x/d is undefined, the block codes to zeros
    x = np.zeros(32, np.float32)
    x[0] = np.float32(2.0 ** -144)
    x[1] = -np.float32(2.0 ** -145)
    assert float(np.float32(2.0 ** -144) / np.float32(127)) == 0.0
    d_h, q = q8_0.quantize_blocks(x)
    assert (q == 0).all() and int(f16_bits(d_h)[0]) == 0


def test_rejects_non_finite():
    x = np.zeros(32, np.float32)
    x[3] = np.inf
    with pytest.raises(ValueError):
        q8_0.quantize_blocks(x)
