"""Pins for the oracle's number formats: each is checked against something
other than itself -- torch's fp8/bf16 casts (library routines), an
independent round-to-nearest-even by binade scaling (np.rint), the
ue8m0 bit formula quoted in the sglang PR #39652 review, and hand-worked
values of its closed form."""
import json
import os

import numpy as np
import pytest
import torch

import oracle


def _e4m3_mags():
    return np.array([oracle.e4m3_value(c) for c in range(127)])


def _rint_round(x, min_q, mant_bits, max_val):
    """Round-half-even of |x| to `mant_bits` fraction bits in its binade
    (binades below 2^min_q share that binade's step), saturating at max_val.
    Independent of the oracle's enumeration."""
    a = np.abs(np.asarray(x, np.float64))
    _, p = np.frexp(a)
    q = np.maximum(p - 1, min_q)
    step = np.ldexp(1.0, q - mant_bits)
    v = np.minimum(np.rint(a / step) * step, max_val)
    return np.where(np.signbit(x) & (v != 0), -v, v)


def test_e4m3_decode_matches_torch():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    mine = np.array([oracle.e4m3_value(c) for c in range(256)])
    assert np.array_equal(np.isnan(mine), np.isnan(ref))
    assert np.isnan(mine[0x7F]) and np.isnan(mine[0xFF])
    ok = ~np.isnan(ref)
    assert np.array_equal(mine[ok], ref[ok])
    assert mine[0x7E] == 448.0 and mine[0x08] == 2.0 ** -6 and mine[0x01] == 2.0 ** -9


def _e4m3_probe_points():
    mags = _e4m3_mags()
    mids = (mags[:-1] + mags[1:]) / 2
    pts = np.concatenate([mags, mids]).astype(np.float32)
    up = np.nextafter(pts, np.float32(np.inf))
    dn = np.nextafter(pts, np.float32(0))
    rng = np.random.default_rng(11)
    rnd = (rng.uniform(0, 464, 200000)).astype(np.float32)
    tiny = (rng.uniform(0, 2.0 ** -5, 50000)).astype(np.float32)
    allp = np.concatenate([pts, up, dn, rnd, tiny])
    return np.concatenate([allp, -allp])


def test_e4m3_encode_matches_torch_rne():
    x = _e4m3_probe_points()
    x = x[np.abs(x) <= 464]                      # torch does not saturate above
    mine = oracle.e4m3_encode(x.astype(np.float64))
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy().copy()
    ref[ref == 0x80] = 0                          # clear_negative_zero
    assert np.array_equal(mine, ref)


def test_e4m3_encode_matches_binade_rint():
    x = _e4m3_probe_points().astype(np.float64)
    x = np.concatenate([x, [480.0, 1e6, -1e30, 465.0]])
    codes = oracle.e4m3_encode(x)
    got = np.array([oracle.e4m3_value(int(c)) for c in codes])
    ref = _rint_round(x, -6, 3, 448.0)
    assert np.array_equal(got, ref)
    assert not np.any(codes == 0x80)
    assert np.all(codes[np.abs(x) >= 448] & 0x7F == 0x7E)   # satfinite


def test_e2m1_values_and_encode_matches_binade_rint():
    mags = [oracle.e2m1_value(c) for c in range(8)]
    assert mags == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    assert [oracle.e2m1_value(8 + c) for c in range(8)] == [-m for m in mags]
    m = np.array(mags)
    mids = (m[:-1] + m[1:]) / 2
    pts = np.concatenate([m, mids, np.nextafter(mids, 0), np.nextafter(mids, 10), [6.5, 7.0, 100.0]])
    rng = np.random.default_rng(5)
    pts = np.concatenate([pts, rng.uniform(0, 8, 100000)]).astype(np.float32).astype(np.float64)
    x = np.concatenate([pts, -pts])
    codes = oracle.e2m1_encode(x)
    got = np.array([oracle.e2m1_value(int(c)) for c in codes])
    ref = _rint_round(x, 0, 1, 6.0)
    assert np.array_equal(got, ref)
    assert not np.any(codes == 0x8)


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(3)
    bits = rng.integers(0, 0x7F800000, 400000, dtype=np.uint32)
    # plus exact ties: low 16 bits == 0x8000 with both parities
    ties = (rng.integers(0, 0x7F7F, 20000, dtype=np.uint32) << 16) | 0x8000
    f = np.concatenate([bits, ties]).view(np.float32)
    f = np.concatenate([f, -f])
    mine = oracle.bf16_bits(f.astype(np.float64))
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(mine, ref)


def _bit_formula(a):
    """The formula as the sglang #39652 review quotes it."""
    bits = np.asarray(a, np.float32).view(np.uint32).astype(np.int64)
    e = (bits >> 23) - 8 + ((bits & 0x7FFFFF) > 0x600000)
    return np.maximum(e, 114)


def test_ue8m0_hand_worked_points(golden_dir):
    with open(os.path.join(golden_dir, "ue8m0_points.json")) as f:
        pts = json.load(f)["points"]
    a = np.array([p["amax"] for p in pts], np.float32)
    want = np.array([p["byte"] for p in pts])
    assert np.array_equal(oracle.ue8m0(a), want)


def _check_ue8m0(a):
    a = np.asarray(a, np.float32)
    got = oracle.ue8m0(a).astype(np.int64)
    bad = np.nonzero(got != _bit_formula(a))[0]
    assert bad.size == 0, f"{bad.size} mismatches, first amax={a[bad[0]]!r}"
    # minimality: 448 * 2^(e-128) < amax <= 448 * 2^(e-127) unless clamped
    ad = a.astype(np.float64)
    hi = np.ldexp(448.0, got - 127)
    lo = np.ldexp(448.0, got - 128)
    assert np.all(ad <= hi)
    assert np.all((got == 114) | (ad > lo))


def test_ue8m0_every_positive_bf16_zero_and_denormals():
    bf = (np.arange(1, 0x7F80, dtype=np.uint32) << 16).view(np.float32)
    _check_ue8m0(np.concatenate([[0.0], bf]).astype(np.float32))
    den = np.arange(1, 1 << 23, dtype=np.uint32).view(np.float32)
    _check_ue8m0(den)


def test_ue8m0_around_every_448_power_of_two():
    pts = []
    for k in range(-160, 121):
        with np.errstate(over="ignore"):
            base = np.float32(np.ldexp(448.0, k))
        if not np.isfinite(base) or base == 0:
            continue
        b = np.array([base], np.float32).view(np.uint32).astype(np.int64)[0]
        lo, hi = max(b - 64, 1), min(b + 64, 0x7F7FFFFF)
        pts.append(np.arange(lo, hi + 1, dtype=np.int64).astype(np.uint32))
    _check_ue8m0(np.concatenate(pts).view(np.float32))


@pytest.mark.slow
def test_ue8m0_134m_random_fp32():
    """2^27 (~134M) random positive finite fp32 values, as in the review."""
    rng = np.random.default_rng(134)
    for _ in range(8):
        bits = rng.integers(1, 0x7F800000, 1 << 24, dtype=np.uint32)
        _check_ue8m0(bits.view(np.float32))
