"""Pins of the oracle's KIVI quantiser and packing to what the pages and the
arithmetic fix (no GPU)."""
from fractions import Fraction

import numpy as np
import pytest

from oracle import kivi

BITS = (2, 3, 4, 8)


def _fp16_values(rng, shape, scale=1.0):
    return (rng.standard_normal(shape) * scale).astype(np.float16).astype(np.float32)


@pytest.mark.parametrize("bits", BITS)
def test_error_bound_half_scale(bits):
    """|x - deq(q(x))| <= scale/2 per element (up to float32 rounding)."""
    rng = np.random.default_rng(bits)
    x = _fp16_values(rng, (64, 8, 32))
    x[:, 3, :] *= 40.0                                        # outlier slices
    q, s, z = kivi.quantize_slices(x, bits)
    deq = kivi.dequantize_slices(q, s, z)
    s32 = s.astype(np.float32)[..., None]
    err = np.abs(x - deq)
    slack = 4 * np.spacing(np.abs(x) + np.abs(z.astype(np.float32)[..., None]))
    assert np.all(err <= 0.5 * s32 * (1 + 2.0 ** -9) + slack)


@pytest.mark.parametrize("bits", BITS)
def test_code_is_nearest_level_brute_force(bits):
    """Each code minimises |x - (z + q s)| over all 2^b codes in exact
    arithmetic (half-way cases go to the even code); fp32 may only differ on
    quotients within 1e-5 of a half-integer."""
    rng = np.random.default_rng(100 + bits)
    x = _fp16_values(rng, (200, 32))
    q, s, z = kivi.quantize_slices(x, bits)
    lb = (1 << bits) - 1
    checked = 0
    for i in range(x.shape[0]):
        S = Fraction(float(s[i]))
        Z = Fraction(float(z[i]))
        for j in range(32):
            t = (Fraction(float(x[i, j])) - Z) / S
            best = min(range(lb + 1), key=lambda c: (abs(t - c), c % 2))
            frac = t - int(t)
            if abs(frac - Fraction(1, 2)) < Fraction(1, 100000):
                continue
            assert q[i, j] == best, (i, j, float(t))
            checked += 1
    assert checked > 0.99 * x.size


def test_exact_half_way_goes_to_even():
    """x - z = (k + 1/2) s exactly: the code is the even neighbour."""
    s = 0.25
    x = np.zeros((1, 32), np.float32)
    x[0, 0] = 0.0                 # min -> zero = 0
    x[0, 1] = 0.75                # max -> range 0.75 over 3 levels: s = 0.25
    x[0, 2] = 0.125               # t = 0.5 -> 0
    x[0, 3] = 0.375               # t = 1.5 -> 2
    x[0, 4] = 0.625               # t = 2.5 -> 2
    q, sh, zh = kivi.quantize_slices(x, 2)
    assert float(sh[0]) == s and float(zh[0]) == 0.0
    assert list(q[0, :5]) == [0, 3, 0, 2, 2]


@pytest.mark.parametrize("bits", BITS)
def test_constant_slice_eps(bits):
    """A constant slice (P1 bug class 1) keeps a nonzero scale and round-trips."""
    x = np.full((3, 32), 0.7109375, np.float32)     # fp16-exact
    q, s, z = kivi.quantize_slices(x, bits)
    assert np.all(q == 0)
    assert np.all(s.astype(np.float32) > 0)
    assert float(s[0]) == float(np.float16(np.float32(1e-5)))
    assert np.array_equal(kivi.dequantize_slices(q, s, z), x)


def test_tiny_range_no_nan():
    """A slice whose range is below eps (P1 bug class 2): finite, within s/2."""
    x = (np.float32(1.0) + np.arange(32, dtype=np.float32) * np.float32(2.0 ** -10)).astype(np.float32)
    x = x.astype(np.float16).astype(np.float32)[None]
    q, s, z = kivi.quantize_slices(x, 2)
    d = kivi.dequantize_slices(q, s, z)
    assert np.all(np.isfinite(d))
    assert np.all(np.abs(d - x) <= 0.5 * s.astype(np.float32)[..., None] + 1e-6)


@pytest.mark.parametrize("bits", BITS)
def test_grid_values_round_trip_and_end_codes(bits):
    """Values on the grid z + k s (both ends present) give codes k exactly and
    dequantise exactly; the clamp reaches 0 and 2^b - 1 (P1 bug class 3)."""
    lb = (1 << bits) - 1
    rng = np.random.default_rng(7)
    k = rng.integers(0, lb + 1, size=(16, 32))
    k[:, 0] = 0
    k[:, 1] = lb
    s, z = 2.0 ** -3, -1.0
    x = (z + k * s).astype(np.float32)
    q, sh, zh = kivi.quantize_slices(x, bits)
    assert np.array_equal(q, k.astype(np.uint8))
    assert np.array_equal(kivi.dequantize_slices(q, sh, zh), x)
    assert q.min() == 0 and q.max() == lb


def test_nan_rejected():
    x = np.zeros((1, 32), np.float32)
    x[0, 5] = np.nan
    with pytest.raises(ValueError):
        kivi.quantize_slices(x, 4)


def test_k_groups_per_channel_v_per_token_axes():
    """K: one scale per channel over the 32 tokens; V: one per token per 32
    channels (the KIVI placement)."""
    rng = np.random.default_rng(3)
    k = _fp16_values(rng, (32, 64))
    k[:, 5] *= 100.0                          # channel outlier -> only channel 5's scale
    q, s, z = kivi.quantize_k_group(k, 2)
    assert s.shape == (64,) and q.shape == (32, 64)
    big = float(s[5])
    assert all(float(s[c]) < big / 10 for c in range(64) if c != 5)
    v = _fp16_values(rng, (32, 64))
    v[7, :32] *= 100.0                        # token outlier in channel group 0
    qv, sv, zv = kivi.quantize_v_rows(v, 4)
    assert sv.shape == (32, 2)
    assert float(sv[7, 0]) > 10 * max(float(sv[t, 0]) for t in range(32) if t != 7)
    assert float(sv[7, 1]) < 10 * float(np.median(sv[:, 1].astype(np.float32)))


@pytest.mark.parametrize("bits", BITS)
def test_pack_unpack_every_level(bits):
    lb = (1 << bits) - 1
    codes = np.array([(i * 7 + 3) % (lb + 1) for i in range(4 * 256)], np.uint8).reshape(4, 256)
    codes[0, : lb + 1] = np.arange(lb + 1)
    packed = kivi.pack_codes(codes, bits)
    assert packed.shape == (4, codes.shape[1] * bits // 8)
    assert np.array_equal(kivi.unpack_codes(packed, bits), codes)


def test_pack_layout_v0_in_low_bits():
    """Foundry spec, "Step 3: Packing": [v0:2][v1:2][v2:2][v3:2] and
    [v0:4][v1:4], read with v0 in the least-significant bits; 3-bit codes
    eight to three bytes. Worked by hand: codes 1..7, 0 are the bit string
    001 010 011 100 101 110 111 000 from bit 0 up, i.e. the 24-bit value
    0x1F58D1, stored D1 58 1F."""
    assert kivi.pack_codes(np.array([[1, 2, 3, 0]], np.uint8), 2)[0, 0] == 0b00111001
    assert kivi.pack_codes(np.array([[1, 2, 3, 4, 5, 6, 7, 0]], np.uint8), 3).tolist() == [[0xD1, 0x58, 0x1F]]
    assert kivi.pack_codes(np.array([[0, 0, 0, 0, 0, 0, 0, 7]], np.uint8), 3).tolist() == [[0x00, 0x00, 0xE0]]
    assert kivi.pack_codes(np.array([[0, 0, 7, 0, 0, 7, 0, 0]], np.uint8), 3).tolist() == [[0xC0, 0x81, 0x03]]
    assert kivi.pack_codes(np.array([[0xA, 0x5]], np.uint8), 4)[0, 0] == 0x5A
    assert list(kivi.pack_codes(np.array([[7, 200]], np.uint8), 8)[0]) == [7, 200]


def test_pack_3bit_is_three_quarters_of_4bit():
    """The 3-bit form stores no unused bits: a row takes 3/4 of the 4-bit
    row's bytes (the page's memory table counts K3 this way)."""
    for D in (64, 128):
        c = np.zeros((1, D), np.uint8)
        assert kivi.pack_codes(c, 3).shape[-1] * 4 == kivi.pack_codes(c, 4).shape[-1] * 3


# ------------------------------------------------------------------ q4_0 V form

def _slice(vals):
    x = np.zeros(32, np.float32)
    x[:len(vals)] = vals
    return x


def test_q4_0_worked_slices():
    """d = m / -8 with m the first value of largest magnitude; code
    floor(x / d + 8.5) clamped to [0, 15]; value (code - 8) d."""
    q, s, z = kivi.quantize_slices_q4_0(_slice([1.0, -2.0, 0.5, 0.75]))
    assert float(s) == 0.25 and float(z) == -2.0
    assert q[:5].tolist() == [12, 0, 10, 11, 8]
    # a positive extreme gives a negative d; -1 lands between levels
    q, s, z = kivi.quantize_slices_q4_0(_slice([3.0, -1.0]))
    assert float(s) == -0.375 and float(z) == 3.0
    assert q[:3].tolist() == [0, 11, 8]
    # equal magnitudes: the first decides the sign; the other one clamps at 15
    q, s, z = kivi.quantize_slices_q4_0(_slice([-4.0, 4.0]))
    assert float(s) == 0.5 and q[:2].tolist() == [0, 15]
    # all zeros: d = 0 and every code 8
    q, s, z = kivi.quantize_slices_q4_0(np.zeros(32, np.float32))
    assert float(s) == 0.0 and float(z) == 0.0 and np.all(q == 8)


def test_q4_0_nearest_level_brute_force_and_affine_readback():
    """Away from the clamp each code is the nearest level (code - 8) d, ties
    upwards, within |d| / 2; the affine read-back code * s + z equals
    (code - 8) d exactly."""
    rng = np.random.default_rng(11)
    x = _fp16_values(rng, (400, 32), 3.0)
    q, s, z = kivi.quantize_slices_q4_0(x)
    d = s.astype(np.float64)[:, None]
    lv = (np.arange(16)[None, None, :] - 8) * d[..., None]          # [400, 1, 16]
    deq = kivi.dequantize_slices(q, s, z).astype(np.float64)
    assert np.array_equal(deq, (q.astype(np.float64) - 8) * d)
    x64 = x.astype(np.float64)
    free = (x64 / d) < 7.5 - 1e-6                                   # not clamped at 15
    err = np.abs(x64[..., None] - lv)                               # [400, 32, 16]
    best = err.min(axis=-1)
    assert np.all(np.abs(x64 - deq)[free] <= np.abs(d).repeat(32, 1)[free] / 2 + 1e-6)
    assert np.all(np.abs(np.abs(x64 - deq) - best)[free] <= 1e-6)
