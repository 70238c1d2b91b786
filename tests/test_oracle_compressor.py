"""Pins for the oracle's fused compressor (pool -> RMSNorm -> RoPE -> store).

The oracle's fp64 rows are checked against a composition of torch library
routines in fp64 (torch.softmax over the pair, F.rms_norm, complex
multiplication through torch.view_as_complex), and against closed-form
special cases: equal scores give the pair's mean, a score gap of 80 gives
the dominant kv, unit weights give RMS = sqrt(ms / (ms + eps)), a (1, 0)
table is the identity and a (0, 1) table is a quarter turn.  The plan's row
counts are the config's numbers (golden fixture)."""
import json
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from deepseek_v4_compressed_c2_gb300 import workloads as W


def _bf(b):
    return torch.from_numpy(oracle.bf16_to_f64(b))


def torch_reference(ratio, rows, ext, norm_w, eps, freqs):
    """fp64 torch composition of the compressor for every planned row."""
    n_slots = ext.shape[1]
    kv = _bf(rows[:, :512])
    sc = _bf(rows[:, 512:1024]) if ratio == 2 else None
    out, pos = [], []
    for r in range(n_slots):
        first, cnt = int(ext[0, r]), max(int(ext[1, r]), 0)
        for j in range(cnt // ratio):
            s = first + ratio * j
            if ratio == 1:
                x = kv[s]
            else:
                w = torch.softmax(sc[s:s + 2], dim=0)
                x = (w * kv[s:s + 2]).sum(0)
            out.append(x)
            pos.append(ratio * j)
    x = torch.stack(out) if out else torch.zeros(0, 512, dtype=torch.float64)
    if norm_w is not None:
        x = F.rms_norm(x, (512,), weight=_bf(norm_w), eps=float(np.float32(eps)))
    latent = x.clone()
    if freqs is not None:
        f = torch.from_numpy(freqs.astype(np.float64))[torch.tensor(pos, dtype=torch.long)]
        rot = torch.view_as_complex(f.reshape(-1, 32, 2).contiguous())
        xr = torch.view_as_complex(x[:, 448:].reshape(-1, 32, 2).contiguous())
        x = x.clone()
        x[:, 448:] = torch.view_as_real(xr * rot).reshape(-1, 64)
    return latent.numpy(), x.numpy()


def _small_case(seed, ratio, lens, norm=True, rope=True):
    rng = np.random.default_rng(seed)
    rows = W.bf16_from_f32(rng.standard_normal((sum(lens) + 5, 1024)).astype(np.float32) * 2)
    ext = np.zeros((2, len(lens) + 1), np.int32)
    ext[0, :len(lens)] = np.concatenate([[0], np.cumsum(lens)[:-1]])
    ext[1, :len(lens)] = lens
    w = W.bf16_from_f32(rng.uniform(0.5, 1.5, 512).astype(np.float32)) if norm else None
    freqs = W.rope_table(4096) if rope else None
    return rows, ext, w, freqs


@pytest.mark.parametrize("ratio", [1, 2])
@pytest.mark.parametrize("norm,rope", [(True, True), (False, True), (True, False), (False, False)])
def test_compressor_matches_torch_composition(ratio, norm, rope):
    rows, ext, w, freqs = _small_case(ratio * 10 + norm * 2 + rope, ratio, [7, 0, 64, 33], norm, rope)
    res = oracle.compress_store(oracle.V41, ratio, rows, ext, norm_w=w, eps=1e-6,
                                freqs=freqs, out_loc=np.zeros(200, np.int32), n_out=200)
    lat, pre = torch_reference(ratio, rows, ext, w, 1e-6, freqs)
    n = lat.shape[0]
    assert res["total"] == n
    got = res["prequant_f64"][:n]
    assert np.allclose(got, pre, rtol=1e-12, atol=1e-12)
    assert np.array_equal(res["prequant_f32"][:n], got.astype(np.float32))
    assert np.array_equal(res["latent"][:n], oracle.bf16_bits(lat))
    assert not res["prequant_f64"][n:].any() and not res["latent"][n:].any()


def test_pool_special_cases():
    rng = np.random.default_rng(4)
    kv = rng.uniform(0.5, 2.0, (4, 512)).astype(np.float32) * rng.choice([-1, 1], (4, 512))
    score = np.zeros((4, 512), np.float32)
    score[2] = 40.0
    score[3] = -40.0                       # pair (2, 3): gap of 80 for row 2
    rows = W.bf16_from_f32(np.concatenate([kv, score], axis=1))
    ext = np.array([[0], [4]], np.int32)
    res = oracle.compress_store(oracle.V41, 2, rows, ext, out_loc=np.zeros(2, np.int32), n_out=2)
    kvd = oracle.bf16_to_f64(rows[:, :512])
    assert np.array_equal(res["prequant_f64"][0], (kvd[0] + kvd[1]) / 2)   # equal scores: mean
    assert np.array_equal(res["prequant_f32"][1], kvd[2].astype(np.float32))  # dominant kv


def test_rmsnorm_unit_weight_closed_form():
    rng = np.random.default_rng(5)
    x = (rng.standard_normal((6, 512)) * np.array([1e-4, 1e-2, 1, 10, 100, 3])[:, None]).astype(np.float32)
    rows = W.bf16_from_f32(x)
    ones = W.bf16_from_f32(np.ones(512, np.float32))
    eps = 1e-6
    res = oracle.compress_store(oracle.V41, 1, rows, np.array([[0], [6]], np.int32),
                                norm_w=ones, eps=eps, out_loc=np.zeros(6, np.int32), n_out=6)
    xd = oracle.bf16_to_f64(rows)
    ms = (xd ** 2).mean(1)
    rms = np.sqrt((res["prequant_f64"] ** 2).mean(1))
    assert np.allclose(rms, np.sqrt(ms / (ms + np.float64(np.float32(eps)))), rtol=1e-13)


def test_rope_identity_and_quarter_turn():
    rng = np.random.default_rng(6)
    rows = W.bf16_from_f32(rng.standard_normal((8, 512)).astype(np.float32))
    ext = np.array([[0], [8]], np.int32)
    ident = np.zeros((8, 64), np.float32)
    ident[:, 0::2] = 1.0
    res = oracle.compress_store(oracle.V41, 1, rows, ext, freqs=ident,
                                out_loc=np.zeros(8, np.int32), n_out=8)
    assert np.array_equal(res["prequant_f64"], oracle.bf16_to_f64(rows))
    quarter = np.zeros((8, 64), np.float32)
    quarter[:, 1::2] = 1.0                                    # cos 0, sin 1
    res = oracle.compress_store(oracle.V41, 1, rows, ext, freqs=quarter,
                                out_loc=np.zeros(8, np.int32), n_out=8)
    x = oracle.bf16_to_f64(rows)
    y = res["prequant_f64"]
    assert np.array_equal(y[:, :448], x[:, :448])
    assert np.array_equal(y[:, 448::2], -x[:, 449::2])        # a' = -b
    assert np.array_equal(y[:, 449::2], x[:, 448::2])         # b' = a
    # the real table preserves each pair's norm and is the identity at pos 0
    res = oracle.compress_store(oracle.V41, 1, rows, ext, freqs=W.rope_table(64),
                                out_loc=np.zeros(8, np.int32), n_out=8)
    y = res["prequant_f64"]
    assert np.array_equal(y[0], x[0])
    n0 = x[:, 448::2] ** 2 + x[:, 449::2] ** 2
    n1 = y[:, 448::2] ** 2 + y[:, 449::2] ** 2
    assert np.allclose(n0, n1, rtol=1e-6)


def test_rope_table_against_closed_form():
    t = W.rope_table(4096)
    pos = np.arange(4096, dtype=np.float64)[:, None]
    ang = pos * 10000.0 ** (-np.arange(32, dtype=np.float64) / 32.0)
    for ref, got in ((np.cos(ang), t[:, 0::2]), (np.sin(ang), t[:, 1::2])):
        ulp = np.spacing(np.abs(ref).astype(np.float32)).astype(np.float64)
        assert np.all(np.abs(got.astype(np.float64) - ref) <= ulp)


def test_plan_counts_of_the_ratio2_config(golden_dir):
    with open(os.path.join(golden_dir, "ratio2_plan_cfg2.json")) as f:
        g = json.load(f)
    cfg = W.cfg2_ratio2_small()
    p = oracle.plan(2, cfg["ext"], cfg["page_table"], cfg["page_bits"])
    assert p["total"] == g["total_rows"]
    assert np.bincount(p["req"], minlength=4)[:4].tolist() == g["rows_per_request"]
    assert cfg["n_out"] == g["padded_rows"]
    assert cfg["lengths"] == g["extend_lengths"]
    # positions are ratio * j, sources the pair's first row
    for r in range(4):
        sel = p["req"] == r
        j = p["j"][sel]
        assert np.array_equal(j, np.arange(sel.sum()))
        assert np.array_equal(p["pos"][sel], 2 * j)
        assert np.array_equal(p["src"][sel], cfg["ext"][0, r] + 2 * j)


def test_out_loc_zero_rows_are_computed_not_stored_and_faults():
    rows, ext, w, freqs = _small_case(8, 2, [10, 9])
    pool = np.full(64 * 528, 0x5A, np.uint8)
    out_loc = np.array([3, 0, 5, 6, 0, 9, 10, -2, 64, 11, 0, 0], np.int32)  # 9.. pad
    res = oracle.compress_store(oracle.V41, 2, rows, ext, norm_w=w, freqs=freqs,
                                out_loc=out_loc, pool=pool, pool_rows=64)
    assert res["total"] == 9
    assert res["faults"] == 2                                  # slots -2 and 64
    assert res["prequant_f64"][1].any() and res["prequant_f64"][4].any()
    assert res["prequant_f64"][7].any()                        # computed, not stored
    assert not res["prequant_f64"][9:].any()                   # past the total
    stored = {3, 5, 6, 9, 10}
    for s in range(64):
        blk = pool[s * 528:(s + 1) * 528]
        assert (blk == 0x5A).all() == (s not in stored)
    # source rows past the input and positions past the table are faults
    bad_ext = ext.copy()
    bad_ext[1, 1] = 40                                         # runs past n_rows
    res = oracle.compress_store(oracle.V41, 2, rows, bad_ext, out_loc=np.zeros(30, np.int32))
    assert res["faults"] > 0
    short = W.rope_table(4)
    res = oracle.compress_store(oracle.V41, 2, rows, ext, freqs=short,
                                out_loc=np.zeros(9, np.int32))
    assert res["faults"] == 9 - 2 - 2                          # j >= 2 in each request


def test_identical_input_mode_quantizes_the_given_rows():
    rows, ext, w, freqs = _small_case(12, 1, [20])
    given = np.random.default_rng(1).standard_normal((20, 512)).astype(np.float32)
    pool = np.zeros(32 * 528, np.uint8)
    oracle.compress_store(oracle.V41, 1, rows, ext, norm_w=w, freqs=freqs,
                          out_loc=np.arange(1, 21, dtype=np.int32), pool=pool,
                          pool_rows=32, prequant_in=given)
    want = oracle.quantize_rows(oracle.V41, given)
    assert np.array_equal(pool.reshape(32, 528)[1:21], want)


def test_topk_to_slots_oracle():
    pt = np.array([[5, 2, 9], [7, 1, 0]], np.int32)
    topk = np.array([[0, 3, 4, 11, -1, 12], [1, 4, 8, 5, 2, -1]], np.int32)
    slots, lens, faults = oracle.topk_to_slots(topk, np.array([0, 1], np.int32), pt, 2)
    assert slots[0].tolist() == [20, 23, 8, 39, -1, -1]        # id 12 -> page 3 >= max_pages
    assert slots[1].tolist() == [29, 4, 0, 5, 30, -1]
    assert lens.tolist() == [4, 5] and faults == 1
    slots, lens, _ = oracle.topk_to_slots(topk, np.array([0, 1], np.int32), pt, 2,
                                          is_valid=np.array([1, 0], np.uint8))
    assert lens.tolist() == [4, 0] and (slots[1] == -1).all()


def test_topk_to_slots_oracle_page_entries_past_int32():
    """Page entries are non-negative page numbers whose slots fit int32: a
    negative entry, or one whose slot is 2^31 or more, maps to -1 with one
    fault (no 32-bit wrap to a small, in-range slot); the largest entry that
    still fits maps exactly.  Worked by hand with 64 rows per page."""
    big = 1 << 25                                  # slot 2^31 + id offset: past int32
    pt = np.array([[3, -3, big, big - 1]], np.int32)
    topk = np.array([[5, 64 + 5, 128 + 5, 192 + 5, 192 + 63]], np.int32)
    slots, lens, faults = oracle.topk_to_slots(topk, np.array([0], np.int32), pt, 6)
    assert slots[0].tolist() == [197, -1, -1, 2147483589, 2147483647]
    assert lens.tolist() == [3] and faults == 2


def test_fill_all_indices_oracle():
    """Short-context ids, worked by hand: each row counts up to its token's
    visible length and pads with -1; through topk_to_slots they select every
    visible compressed row of the request exactly once."""
    ids = oracle.fill_all_indices(np.array([0, 1, 4, 6, -3], np.int32), 5)
    assert ids.tolist() == [[-1, -1, -1, -1, -1], [0, -1, -1, -1, -1], [0, 1, 2, 3, -1],
                            [0, 1, 2, 3, 4], [-1, -1, -1, -1, -1]]
    pt = np.array([[5, 2, 9], [7, 1, 0]], np.int32)
    lens_in = np.array([6, 3], np.int32)
    slots, lens, faults = oracle.topk_to_slots(oracle.fill_all_indices(lens_in, 8),
                                               np.array([0, 1], np.int32), pt, 2)
    assert slots[0].tolist() == [20, 21, 22, 23, 8, 9, -1, -1]      # pages 5, 2 of request 0
    assert slots[1].tolist() == [28, 29, 30, -1, -1, -1, -1, -1]    # page 7 of request 1
    assert lens.tolist() == [6, 3] and faults == 0


def test_row_subset_mode_equals_the_full_run():
    rows, ext, w, freqs = _small_case(13, 2, [40, 17, 0, 66])
    full = oracle.compress_store(oracle.V41, 2, rows, ext, norm_w=w, freqs=freqs,
                                 out_loc=np.zeros(70, np.int32))
    which = np.array([69, 0, 5, 33, 60, 61], np.int64)        # 60.. are padding
    sub = oracle.compress_store(oracle.V41, 2, rows, ext, norm_w=w, freqs=freqs,
                                out_loc=np.zeros(70, np.int32), which=which)
    for key in ("prequant_f64", "prequant_f32", "latent"):
        assert np.array_equal(sub[key], full[key][which])
    with pytest.raises(ValueError):
        oracle.compress_store(oracle.V41, 2, rows, ext, out_loc=np.zeros(70, np.int32),
                              which=np.array([70]))
