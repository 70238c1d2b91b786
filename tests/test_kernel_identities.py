"""Arithmetic identities the CUDA quantizers rely on, checked on the CPU
against their definitions (no GPU, no CUDA code imported).

* The ue8m0 exponent of the V41 scale: the kernels fold the mantissa test
  `(bits & 0x7FFFFF) > 0x600000` into one add, `(bits + 0x1FFFFF) >> 23`;
  checked for every non-negative fp32 bit pattern.
* The FP4 reciprocal: one Newton-Raphson step from an approximation within
  one ulp lands within 2^-21 ulp of 1/s before its last rounding, so it
  rounds to RN(1/s) whenever 1/s is farther than that from a rounding
  midpoint; checked with exact rationals for all 126 positive e4m3 scales.
* The negative-zero clean-up on packed codes: clearing the sign of every
  e4m3 byte (e2m1 nibble) whose magnitude is zero, by one masked add, equals
  the per-element definition and never carries into a neighbour.
* The ratio-2 row count of a request slot in 32 bits: the decode kernel
  takes floor((p0 + n) / 2) - floor(p0 / 2) as (n + (p0 & 1)) >> 1 on
  unsigned words, for n > 0 and any int32 start p0."""
from fractions import Fraction

import numpy as np


def test_ue8m0_carry_form_equals_the_mantissa_test_for_every_nonnegative_float():
    # bits < 2^31, so bits + 0x1FFFFF fits in 32 bits; buffers reused in place
    step = 1 << 24
    base = np.arange(step, dtype=np.uint32)
    b, plain, carry = np.empty_like(base), np.empty_like(base), np.empty_like(base)
    above = np.empty(step, dtype=bool)
    for start in range(0, 1 << 31, step):
        np.add(base, np.uint32(start), out=b)
        np.right_shift(b, 23, out=plain)
        np.bitwise_and(b, np.uint32(0x7FFFFF), out=carry)
        np.greater(carry, np.uint32(0x600000), out=above)
        plain += above
        np.add(b, np.uint32(0x1FFFFF), out=carry)
        carry >>= 23
        assert np.array_equal(plain, carry), hex(start)


def _e4m3_value(code):
    e, m = (code >> 3) & 15, code & 7
    return Fraction(m, 8) * Fraction(1, 64) if e == 0 else (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)


def _ulps_to_nearest_fp32_midpoint(v):
    """Distance of the positive rational v from the nearest midpoint between
    adjacent fp32 values, in ulps of v's binade (v is a normal fp32 value's
    neighbourhood: all reciprocals here lie in [2^-9, 2^9])."""
    k = 0
    while Fraction(2) ** (k + 1) <= v:
        k += 1
    while Fraction(2) ** k > v:
        k -= 1
    ulp = Fraction(2) ** (k - 23)
    frac = (v / ulp) - int(v / ulp)          # position inside its ulp, in [0, 1)
    return abs(frac - Fraction(1, 2))


def test_newton_reciprocal_margin_for_every_e4m3_scale():
    margins = [_ulps_to_nearest_fp32_midpoint(1 / _e4m3_value(c)) for c in range(1, 127)]
    worst = min(margins)
    assert worst == Fraction(1, 30)           # at 0x0F: s = 15 / 512
    assert worst > Fraction(1, 1 << 21)       # the Newton step's error bound
    # the powers of two are exact: 1/s is itself an fp32 value (margin 1/2)
    assert all(margins[c - 1] == Fraction(1, 2) for c in (0x08, 0x10, 0x38, 0x40, 0x70))


def _clear_negative_zero_e4m3x4(w):
    nonzero = ((w & 0x7F7F7F7F) + 0x7F7F7F7F) & 0x80808080
    return w & (nonzero | 0x7F7F7F7F)


def _clear_negative_zero_e2m1x8(w):
    nonzero = ((w & 0x77777777) + 0x77777777) & 0x88888888
    return w & (nonzero | 0x77777777)


def test_negative_zero_cleanup_matches_its_definition():
    rng = np.random.default_rng(5)
    # every byte value in every position, with random neighbours
    for pos in range(4):
        for byte in range(256):
            others = rng.integers(0, 1 << 32, 64, dtype=np.uint64)
            w = (others & ~np.uint64(0xFF << (8 * pos))) | np.uint64(byte << (8 * pos))
            got = _clear_negative_zero_e4m3x4(w)
            for x, y in zip(w.tolist(), got.tolist()):
                want = 0
                for i in range(4):
                    b = (x >> (8 * i)) & 0xFF
                    want |= (0 if b == 0x80 else b) << (8 * i)
                assert y == want
    # every nibble value in every position, with random neighbours
    for pos in range(8):
        for nib in range(16):
            others = rng.integers(0, 1 << 32, 64, dtype=np.uint64)
            w = (others & ~np.uint64(0xF << (4 * pos))) | np.uint64(nib << (4 * pos))
            got = _clear_negative_zero_e2m1x8(w)
            for x, y in zip(w.tolist(), got.tolist()):
                want = 0
                for i in range(8):
                    q = (x >> (4 * i)) & 0xF
                    want |= (0 if q == 0x8 else q) << (4 * i)
                assert y == want


def test_ratio2_row_count_in_32_bits_equals_the_difference_of_halves():
    rng = np.random.default_rng(3)
    lim = np.iinfo(np.int32)
    p0 = np.concatenate([rng.integers(lim.min, lim.max, 1 << 20, endpoint=True),
                         np.arange(-64, 65), [lim.min, lim.min + 1, lim.max - 1, lim.max]])
    n = np.concatenate([rng.integers(1, lim.max, 1 << 20, endpoint=True),
                        rng.integers(1, 9, 129), [1, lim.max, 2, lim.max]])
    p0, n = p0.astype(np.int64), n.astype(np.int64)
    want = np.floor_divide(p0 + n, 2) - np.floor_divide(p0, 2)      # exact in int64
    got = (n.astype(np.uint32) + (p0.astype(np.int32).view(np.uint32) & np.uint32(1))) >> np.uint32(1)
    assert np.array_equal(got.astype(np.int64), want)
