"""Helpers for the GPU-vs-oracle parity tests.

Tolerances (the contract's rules):
  * gather-dequant output and scale bytes: bit-exact;
  * codes: bit-exact when the oracle quantizes the GPU's own fp32 pre-quant
    rows ("identical-input" mode);
  * end to end: pre-quant rows within 1e-5 of the fp64 oracle, relative to the
    row's max magnitude; at most 1e-4 of the codes may differ, each by one
    code step -- every differing code counts, including those whose fp64
    value sits on a rounding tie (reported separately as tie flips); a scale
    byte may differ only where the fp64 group amax sits within 1e-5
    (relative) of the boundary that decides it, and the codes of such a group
    are then not counted.
"""
import numpy as np
import torch

import oracle

PREQUANT_RTOL = 1e-5
CODE_FRACTION = 1e-4
BOUNDARY_RTOL = 1e-5


def dev_bf16(a_u16, device="cuda"):
    return torch.from_numpy(np.ascontiguousarray(a_u16).view(np.int16)).view(torch.bfloat16).to(device)


def dev(a, device="cuda"):
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def host_u16(t):
    return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)


def assert_prequant_close(g, r, rtol=PREQUANT_RTOL):
    g = np.asarray(g, np.float64)
    r = np.asarray(r, np.float64)
    scale = np.abs(r).max(axis=1)
    err = np.abs(g - r).max(axis=1)
    bad = err > rtol * scale
    assert not bad.any(), (f"{bad.sum()} rows outside {rtol} relative; worst "
                           f"{(err / np.maximum(scale, 1e-300)).max():.3g}")
    return float((err / np.maximum(scale, 1e-300)).max()) if len(err) else 0.0


def _signed_index(codes, bits):
    mag_mask = (1 << (bits - 1)) - 1
    m = (codes & mag_mask).astype(np.int64)
    s = (codes >> (bits - 1)).astype(np.int64)
    return np.where(s == 1, -m, m)


def _near_pow2(v):
    with np.errstate(divide="ignore"):
        e = np.round(np.log2(np.maximum(v, 1e-300)))
    return np.abs(v / np.exp2(e) - 1.0) <= BOUNDARY_RTOL


TIE_RTOL = 2.0 ** -20

_E4M3 = None
_E2M1 = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], np.float64)


def _e4m3_mags():
    global _E4M3
    if _E4M3 is None:
        _E4M3 = np.array([oracle.e4m3_value(c) for c in range(127)])
    return _E4M3


def _at_tie(y, mags):
    """|y| within TIE_RTOL (relative) of a rounding midpoint of `mags`."""
    mids = (mags[:-1] + mags[1:]) / 2
    a = np.abs(y)
    i = np.clip(np.searchsorted(mids, a), 1, len(mids) - 1)
    d = np.minimum(np.abs(a - mids[i - 1]), np.abs(a - mids[i]))
    return d <= TIE_RTOL * a


def _code_ties(layout, ref_rows, ref_prequant_f64):
    """Codes whose oracle value sits on a rounding tie: an fp32 pipeline that
    differs from fp64 by one ulp may round them either way."""
    x = np.asarray(ref_prequant_f64, np.float64)
    n = x.shape[0]
    if layout == oracle.V41:
        e = ref_rows[:, 512:528].astype(np.int64)
        return _at_tie(x * np.repeat(np.ldexp(1.0, 127 - e), 32, axis=1), _e4m3_mags())
    if layout == oracle.V4:
        e = ref_rows[:, 576:583].astype(np.int64)
        return _at_tie(x[:, :448] * np.repeat(np.ldexp(1.0, 127 - e), 64, axis=1), _e4m3_mags())
    sv = np.array([oracle.e4m3_value(int(c)) for c in ref_rows[:, 256:288].reshape(-1)]).reshape(n, 32)
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.where(np.repeat(sv, 16, axis=1) > 0, x / np.repeat(sv, 16, axis=1), 0.0)
    return _at_tie(q, _E2M1)


def compare_rows_end_to_end(layout, got_rows, ref_rows, ref_prequant_f64, min_allowed=0):
    """got_rows / ref_rows: uint8 [n, row_bytes]; ref_prequant_f64 [n, 512].
    Every code that differs from the oracle's counts against CODE_FRACTION of
    the compared codes; `min_allowed` is an absolute floor of that budget for
    cases too small for the fraction to allow a single code.  Returns a dict:
    differing codes, of them at rounding ties, codes compared, flipped scale
    groups, group size."""
    n = got_rows.shape[0]
    if layout == oracle.V4:
        # nope: 7 ue8m0 groups of 64 dims; rope: bf16 values within one bf16
        # step of the oracle's (its fp32 value differs from the GPU's by
        # at most the pre-quant tolerance)
        gs, rs = got_rows[:, 576:583], ref_rows[:, 576:583]
        amax = np.abs(ref_prequant_f64[:, :448]).reshape(n, 7, 64).max(axis=2)
        flip = gs != rs
        if flip.any():
            assert np.all(np.abs(gs[flip].astype(int) - rs[flip].astype(int)) == 1)
            assert np.all(_near_pow2(amax[flip] / 448.0)), "scale flip away from a 2^k boundary"
        assert not got_rows[:, 583].any()
        gr = oracle.bf16_to_f64(np.ascontiguousarray(got_rows[:, 448:576]).view(np.uint16))
        rr = oracle.bf16_to_f64(np.ascontiguousarray(ref_rows[:, 448:576]).view(np.uint16))
        row_tol = PREQUANT_RTOL * np.abs(ref_prequant_f64).max(axis=1, keepdims=True)
        assert np.all(np.abs(gr - rr) <= np.abs(rr) * 2.0 ** -7 + row_tol)
        gc = _signed_index(got_rows[:, :448], 8)
        rc = _signed_index(ref_rows[:, :448], 8)
        keep = ~np.repeat(flip, 64, axis=1)
        group = 64
    elif layout == oracle.V41:
        gs, rs = got_rows[:, 512:], ref_rows[:, 512:]
        amax = np.abs(ref_prequant_f64).reshape(n, 16, 32).max(axis=2)
        flip = gs != rs
        if flip.any():
            assert np.all(np.abs(gs[flip].astype(int) - rs[flip].astype(int)) == 1)
            assert np.all(_near_pow2(amax[flip] / 448.0)), "scale flip away from a 2^k boundary"
        gc = _signed_index(got_rows[:, :512], 8)
        rc = _signed_index(ref_rows[:, :512], 8)
        keep = ~np.repeat(flip, 32, axis=1)
        group = 32
    else:
        gs, rs = got_rows[:, 256:], ref_rows[:, 256:]
        amax = np.abs(ref_prequant_f64).reshape(n, 32, 16).max(axis=2)
        flip = gs != rs
        if flip.any():
            gv = np.array([oracle.e4m3_value(int(c)) for c in gs[flip]])
            rv = np.array([oracle.e4m3_value(int(c)) for c in rs[flip]])
            mid = (gv + rv) / 2
            assert np.all(np.abs(gs[flip].astype(int) - rs[flip].astype(int)) == 1)
            assert np.all(np.abs(amax[flip] / 6.0 / mid - 1.0) <= BOUNDARY_RTOL), \
                "FP4 scale flip away from a rounding boundary"
        def nibbles(rows):
            b = rows[:, :256]
            return np.stack([b & 0xF, b >> 4], -1).reshape(n, 512)
        gc = _signed_index(nibbles(got_rows), 4)
        rc = _signed_index(nibbles(ref_rows), 4)
        keep = ~np.repeat(flip, 16, axis=1)
        group = 16
    diff = (gc != rc) & keep
    assert np.all(np.abs(gc - rc)[diff] <= 1), "a code differs by more than one step"
    n_diff = int(diff.sum())
    n_tie = int((diff & _code_ties(layout, ref_rows, ref_prequant_f64)).sum())
    total = int(keep.sum())
    allowed = max(CODE_FRACTION * total, min_allowed)
    assert n_diff <= allowed, (f"{n_diff} of {total} codes differ (> {allowed:.1f}); "
                               f"{n_tie} of them at rounding ties")
    return dict(diff=n_diff, tie_flips=n_tie, total=total, scale_flips=int(flip.sum()),
                group=group)


def assert_bf16_equal_nan_aware(got_u16, ref_u16):
    g = oracle.bf16_to_f64(got_u16)
    r = oracle.bf16_to_f64(ref_u16)
    gn, rn = np.isnan(g), np.isnan(r)
    assert np.array_equal(gn, rn)
    assert np.array_equal(np.asarray(got_u16)[~gn], np.asarray(ref_u16)[~rn])
