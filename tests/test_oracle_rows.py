"""Pins for the oracle's row quantizer, dequantizer and paged addressing.

store_row is checked against an independent numpy composition: the ue8m0
byte from the bit formula quoted in the sglang PR #39652 review, the e4m3 /
e2m1 codes from round-half-even by binade scaling (np.rint), the FP4 scale
from an fp32 division by numpy.  Dequant is checked against torch's fp8
decode and bf16 cast.  Row sizes are the page's numbers."""
import json
import os

import numpy as np
import torch

import oracle
from deepseek_v4_compressed_c2_gb300 import workloads as W

from test_oracle_formats import _bit_formula, _rint_round


def test_row_sizes_are_the_pages_numbers(golden_dir):
    with open(os.path.join(golden_dir, "kvlayout_row_bytes.json")) as f:
        g = json.load(f)
    rb = g["row_bytes"]
    assert oracle.row_bytes(oracle.V4) == rb["V4"] == 448 + 2 * 64 + 8
    assert oracle.row_bytes(oracle.V41) == rb["V41"] == 512 + 512 // 32
    assert oracle.row_bytes(oracle.V41_FP4) == rb["V41_FP4"] == 512 // 2 + 512 // 16


def _tiny_rows(seed=0):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((48, 512)).astype(np.float32)
    idx = rng.choice(x.size, x.size // 100, replace=False)
    x.reshape(-1)[idx] *= 50                                  # outliers
    special = np.zeros((8, 512), np.float32)
    special[1, 7] = -3.0                                      # a lone value
    special[2] = np.ldexp(1.0, rng.integers(-20, 20, 512)).astype(np.float32)
    special[3] = (rng.standard_normal(512) * 1e-7).astype(np.float32)   # below the clamp
    special[4, ::32] = 448.0                                  # amax = 448 * 2^0 exactly
    special[5] = -0.0
    special[6] = rng.uniform(-1e30, 1e30, 512).astype(np.float32)
    special[7, :] = np.float32(2.0 ** -140)                    # fp32 denormals
    return np.concatenate([x, special])


def test_v41_store_row_matches_independent_composition():
    x = _tiny_rows()
    rows = oracle.quantize_rows(oracle.V41, x)
    assert rows.shape == (x.shape[0], 528)
    xg = x.reshape(-1, 16, 32).astype(np.float64)
    amax = np.abs(x.reshape(-1, 16, 32)).max(axis=2)
    e = _bit_formula(amax)
    assert np.array_equal(rows[:, 512:], e.astype(np.uint8))
    y = xg * np.ldexp(1.0, 127 - e)[:, :, None]
    want = _rint_round(y, -6, 3, 448.0).reshape(-1, 512)
    codes = rows[:, :512]
    got = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(got, want)
    assert not np.any(codes == 0x80)                           # -0 stored as +0


def test_v41_round_trip_error_bound():
    x = _tiny_rows(1)
    rows = oracle.quantize_rows(oracle.V41, x)
    deq = oracle.dequant_rows(oracle.V41, rows)
    e = rows[:, 512:].astype(np.int64)
    scale = np.repeat(np.ldexp(1.0, e - 127), 32, axis=1)
    y = np.abs(x.astype(np.float64)) / scale
    _, p = np.frexp(y)
    half_ulp = np.ldexp(1.0, np.maximum(p - 1, -6) - 4) * scale
    assert np.all(np.abs(deq - x.astype(np.float64)) <= half_ulp)


def test_fp4_store_row_matches_independent_composition():
    x = _tiny_rows(2)
    x[0, :16] = [6, -6, 0.5, 1.5, 3, 4, 2, 1, 0, -0.25, 0.75, 5, -5, 2.5, 3.5, 1.75]
    rows = oracle.quantize_rows(oracle.V41_FP4, x)
    assert rows.shape == (x.shape[0], 288)
    amax = np.abs(x.reshape(-1, 32, 16)).max(axis=2).astype(np.float32)
    sdiv = (amax / np.float32(6.0)).astype(np.float32)          # IEEE fp32 division
    sval = _rint_round(sdiv.astype(np.float64), -6, 3, 448.0)
    sbytes = rows[:, 256:]
    got_s = torch.from_numpy(sbytes.copy()).view(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(got_s, sval)
    s32 = sval.astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        q = (x.reshape(-1, 32, 16) / s32[:, :, None]).astype(np.float32)
    want = np.where(s32[:, :, None] == 0, 0.0, _rint_round(q.astype(np.float64), 0, 1, 6.0))
    lo = rows[:, :256] & 0xF
    hi = rows[:, :256] >> 4
    nib = np.stack([lo, hi], axis=-1).reshape(-1, 512)         # dim 2i = low nibble
    table = np.array([oracle.e2m1_value(c) for c in range(16)])
    assert np.array_equal(table[nib], want.reshape(-1, 512))
    assert not np.any(nib == 0x8)


def test_fp4_round_trip_error_bound():
    x = _tiny_rows(3)
    rows = oracle.quantize_rows(oracle.V41_FP4, x)
    deq = oracle.dequant_rows(oracle.V41_FP4, rows)
    s = torch.from_numpy(rows[:, 256:].copy()).view(torch.float8_e4m3fn).double().numpy()
    s = np.repeat(s, 16, axis=1)
    a = np.abs(x.astype(np.float64))
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.where(s > 0, a / s, 0.0)
    _, p = np.frexp(q)
    half_ulp = np.ldexp(1.0, np.maximum(p - 1, 0) - 2)
    bound = s * (half_ulp * (1 + 2.0 ** -20) + np.maximum(q - 6.0, 0.0))
    bound = np.where(s > 0, bound, a)                          # s == 0: codes 0
    assert np.all(np.abs(deq - x.astype(np.float64)) <= bound + 1e-300)


def test_dequant_gather_is_exact_bf16_and_handles_bad_ids():
    x = _tiny_rows(4)[:40]
    for layout in (oracle.V41, oracle.V41_FP4):
        rows = oracle.quantize_rows(layout, x)
        pool = rows.reshape(-1)
        ids = np.array([3, -1, 0, 39, 40, 1000, 7], np.int32)
        out, faults = oracle.dequant_gather(layout, pool, 40, ids)
        assert faults == 2                                     # ids 40 and 1000
        ref = oracle.dequant_rows(layout, rows)
        for i, rid in enumerate(ids):
            if 0 <= rid < 40:
                exp = torch.from_numpy(ref[rid]).float().to(torch.bfloat16)
                assert np.array_equal(out[i], exp.view(torch.int16).numpy().view(np.uint16))
                # the products are exact: bf16 value == fp64 value
                assert np.array_equal(oracle.bf16_to_f64(out[i]), ref[rid])
            else:
                assert not out[i].any()


def test_dequant_of_arbitrary_bytes_matches_torch_decode():
    """Every code byte under a spread of scale bytes (not only what the store
    writes) against torch's fp8 decode times the scale."""
    rng = np.random.default_rng(9)
    n = 64
    v41 = rng.integers(0, 256, (n, 528), dtype=np.uint8)
    v41[:, :256] = np.arange(256, dtype=np.uint8)
    v41[:, 512:] = rng.integers(1, 255, (n, 16), dtype=np.uint8)
    out, _ = oracle.dequant_gather(oracle.V41, v41.reshape(-1), n, np.arange(n, dtype=np.int32))
    code = torch.from_numpy(v41[:, :512].copy()).view(torch.float8_e4m3fn).double()
    sc = torch.from_numpy(np.ldexp(1.0, v41[:, 512:].astype(np.int64) - 127)).repeat_interleave(32, 1)
    ref = (code * sc).float().to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(oracle.bf16_to_f64(ref))
    assert np.array_equal(np.isnan(oracle.bf16_to_f64(out)), nan)
    assert np.array_equal(out[~nan], ref[~nan])

    fp4 = rng.integers(0, 256, (n, 288), dtype=np.uint8)
    out, _ = oracle.dequant_gather(oracle.V41_FP4, fp4.reshape(-1), n, np.arange(n, dtype=np.int32))
    nib = np.stack([fp4[:, :256] & 0xF, fp4[:, :256] >> 4], -1).reshape(n, 512)
    e2 = np.array([0, .5, 1, 1.5, 2, 3, 4, 6, -0., -.5, -1, -1.5, -2, -3, -4, -6])[nib]
    s = torch.from_numpy(fp4[:, 256:].copy()).view(torch.float8_e4m3fn).double().numpy()
    ref = torch.from_numpy(e2 * np.repeat(s, 16, 1)).float().to(torch.bfloat16)
    ref = ref.view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(oracle.bf16_to_f64(ref))
    assert np.array_equal(np.isnan(oracle.bf16_to_f64(out)), nan)
    assert np.array_equal(out[~nan], ref[~nan])


def test_paged_addressing_brute_force():
    """Random permuted page tables: every written row lands inside the page the
    table assigns, written byte ranges are disjoint, page 0 and every other
    byte keep their sentinel."""
    rng = np.random.default_rng(21)
    for layout, ratio, page_bits in [(oracle.V41, 1, 3), (oracle.V41, 2, 2),
                                     (oracle.V41_FP4, 2, 4), (oracle.V41_FP4, 1, 0)]:
        lens = [int(v) for v in rng.integers(0, 90, 6)]
        rb = oracle.row_bytes(layout)
        per = [n // ratio for n in lens]
        pages = [-(-p // (1 << page_bits)) for p in per]
        phys = rng.permutation(sum(pages)) + 1
        pt = np.zeros((6, max(1, max(pages))), np.int32)
        o = 0
        for r, p in enumerate(pages):
            pt[r, :p] = phys[o:o + p]
            o += p
        pool_rows = (sum(pages) + 1) << page_bits
        pool = np.full(pool_rows * rb, 0xA5, np.uint8)
        rows = W.bf16_from_f32(rng.standard_normal((sum(lens), 1024)).astype(np.float32))
        ext = np.zeros((2, 6), np.int32)
        ext[0] = np.concatenate([[0], np.cumsum(lens)[:-1]])
        ext[1] = lens
        res = oracle.compress_store(layout, ratio, rows, ext, page_table=pt,
                                    page_bits=page_bits, pool=pool, pool_rows=pool_rows)
        assert res["total"] == sum(per) and res["faults"] == 0
        written = np.zeros(pool.size, bool)
        k = 0
        page_bytes = rb << page_bits
        for r in range(6):
            for j in range(per[r]):
                off = int(pt[r, j >> page_bits]) * page_bytes + (j & ((1 << page_bits) - 1)) * rb
                assert off >= page_bytes                          # never page 0
                assert not written[off:off + rb].any()            # disjoint
                written[off:off + rb] = True
                want = oracle.quantize_rows(layout, res["prequant_f32"][k:k + 1])[0]
                assert np.array_equal(pool[off:off + rb], want)
                k += 1
        assert np.all(pool[~written] == 0xA5)
        for slot in range(0, pool_rows, 7):
            assert oracle.row_offset(layout, page_bits, slot) == slot * rb


def test_v4_store_row_matches_independent_composition():
    """V4 reading: 448 e4m3 nope codes (ue8m0 per 64 dims, the same closed
    form), 64 bf16 rope values, 7 scale bytes and a zero pad byte."""
    x = _tiny_rows(7)
    rows = oracle.quantize_rows(oracle.V4, x)
    assert rows.shape == (x.shape[0], 584)
    amax = np.abs(x[:, :448].reshape(-1, 7, 64)).max(axis=2)
    e = _bit_formula(amax)
    assert np.array_equal(rows[:, 576:583], e.astype(np.uint8))
    assert not rows[:, 583].any()
    y = x[:, :448].reshape(-1, 7, 64).astype(np.float64) * np.ldexp(1.0, 127 - e)[:, :, None]
    want = _rint_round(y, -6, 3, 448.0).reshape(-1, 448)
    got = torch.from_numpy(rows[:, :448].copy()).view(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(got, want)
    rope = torch.from_numpy(x[:, 448:].copy()).to(torch.bfloat16).view(torch.int16).numpy()
    assert np.array_equal(rows[:, 448:576].copy().view(np.int16), rope)
    deq = oracle.dequant_rows(oracle.V4, rows)
    assert np.array_equal(deq[:, 448:], oracle.bf16_to_f64(rope.view(np.uint16)))
