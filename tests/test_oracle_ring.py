"""Pins for the pair-state ring and start positions (the ratio-2 decode /
verify path of sglang PR #39652's c2 compressor): compressing a request's
tokens in one step must equal compressing them in several steps -- chunks
with odd split points, one token per step (decode), or speculative verify
steps that are partly rolled back -- with the ring carrying the unpaired
token between steps.  A wrong ring index, position, slot or ordering breaks
these equalities."""
import numpy as np
import pytest

import oracle
from deepseek_v4_compressed_c2_gb300 import workloads as W

R = 6          # ring entries per request


def _setup(seed, n_tok, ratio=2, page_bits=3):
    rng = np.random.default_rng(seed)
    rows = W.bf16_from_f32(rng.standard_normal((n_tok, 1024)).astype(np.float32))
    w = W.bf16_from_f32(rng.uniform(0.5, 1.5, 512).astype(np.float32))
    n_c = n_tok // ratio + 1
    pages = -(-n_c // (1 << page_bits))
    pt = (rng.permutation(pages) + 1).astype(np.int32).reshape(1, -1)
    pool_rows = (pages + 1) << page_bits
    return rows, w, W.rope_table(1024), pt, pool_rows


def _run(rows, w, freqs, pt, pool_rows, steps, ratio=2, layout=oracle.V41, ring=None):
    """steps: list of (p0, n) over the same token sequence; returns the pool
    and the per-row fp64 pre-quant values keyed by compressed index."""
    rb = oracle.row_bytes(layout)
    pool = np.zeros(pool_rows * rb, np.uint8)
    if ring is None and ratio == 2:
        ring = np.zeros((1, R, 1024), np.uint16)
    got = {}
    for p0, n in steps:
        ext = np.array([[0], [n]], np.int32)
        sub = np.ascontiguousarray(rows[p0:p0 + n])
        sp = np.array([p0], np.int32)
        res = oracle.compress_store(layout, ratio, sub, ext, page_table=pt, page_bits=3,
                                    norm_w=w, freqs=freqs, pool=pool, pool_rows=pool_rows,
                                    start_pos=sp, ring=ring if ratio == 2 else None)
        assert res["faults"] == 0
        p = oracle.plan(ratio, ext, pt, 3, start_pos=sp)
        for k in range(res["total"]):
            got[int(p["c"][k])] = res["prequant_f64"][k]
    return pool, got


@pytest.mark.parametrize("layout", [oracle.V41, oracle.V41_FP4])
def test_chunked_prefill_equals_whole(layout):
    rows, w, fr, pt, pr = _setup(1, 101)
    whole_pool, whole = _run(rows, w, fr, pt, pr, [(0, 101)], layout=layout)
    for cuts in ([0, 37, 101], [0, 1, 2, 3, 50, 101], [0, 63, 64, 100, 101], [0, 11, 12, 99, 101]):
        steps = [(a, b - a) for a, b in zip(cuts[:-1], cuts[1:])]
        pool, got = _run(rows, w, fr, pt, pr, steps, layout=layout)
        assert np.array_equal(pool, whole_pool)
        assert sorted(got) == sorted(whole) == list(range(50))
        for c in whole:
            assert np.array_equal(got[c], whole[c])


def test_decode_one_token_per_step_equals_prefill():
    rows, w, fr, pt, pr = _setup(2, 40)
    whole_pool, whole = _run(rows, w, fr, pt, pr, [(0, 40)])
    pool, got = _run(rows, w, fr, pt, pr, [(q, 1) for q in range(40)])
    assert np.array_equal(pool, whole_pool)
    for c in whole:
        assert np.array_equal(got[c], whole[c])


def test_speculative_verify_with_rollback_equals_prefill():
    """Steps of 1 + 3 draft tokens; after each step only some drafts are
    accepted, and the next step restarts after the last accepted token."""
    rows, w, fr, pt, pr = _setup(3, 64)
    rng = np.random.default_rng(9)
    p0, steps = 0, []
    while p0 < 60:
        steps.append((p0, 4))
        p0 += int(rng.integers(1, 5))            # accepted 1..4 of the 4
    final = p0
    whole_pool, whole = _run(rows, w, fr, pt, pr, [(0, final)])
    pool, got = _run(rows, w, fr, pt, pr, steps)
    # every row the straight prefill of the accepted tokens writes is written
    # identically by the last step that produced it
    rb = 528
    for c in whole:
        assert np.array_equal(got[c], whole[c])
        slot = (int(pt[0, c >> 3]) << 3) | (c & 7)
        assert np.array_equal(pool[slot * rb:(slot + 1) * rb], whole_pool[slot * rb:(slot + 1) * rb])


def test_ratio1_start_positions_equal_whole():
    rows, w, fr, pt, pr = _setup(4, 30, ratio=1)
    whole_pool, whole = _run(rows, w, fr, pt, pr, [(0, 30)], ratio=1)
    pool, got = _run(rows, w, fr, pt, pr, [(0, 7), (7, 1), (8, 22)], ratio=1)
    assert np.array_equal(pool, whole_pool)
    for c in whole:
        assert np.array_equal(got[c], whole[c])


def test_ring_row_without_a_ring_is_a_fault_and_ring_keeps_last_even_tokens():
    rows, w, fr, pt, pr = _setup(5, 20)
    ext = np.array([[0], [4]], np.int32)
    pool = np.zeros(pr * 528, np.uint8)
    res = oracle.compress_store(oracle.V41, 2, rows[5:9].copy(), ext, page_table=pt, page_bits=3,
                                start_pos=np.array([5], np.int32), n_out=3, pool=pool,
                                pool_rows=pr)
    assert res["faults"] == 1                     # pair (4, 5) needs token 4
    ring = np.zeros((1, 3, 1024), np.uint16)
    oracle.compress_store(oracle.V41, 2, rows[0:15].copy(), np.array([[0], [15]], np.int32),
                          page_table=pt, page_bits=3, start_pos=np.array([0], np.int32),
                          ring=ring)
    # positions 8, 10, 12, 14 are the even tokens in the last 2R = 6 positions
    # (9..14): 10, 12, 14 land at entries 5 % 3, 6 % 3, 7 % 3
    assert np.array_equal(ring[0, 5 % 3], rows[10])
    assert np.array_equal(ring[0, 6 % 3], rows[12])
    assert np.array_equal(ring[0, 7 % 3], rows[14])


def test_negative_positions_are_faults_and_the_rest_matches_a_fresh_start():
    """A start position before 0 (out of contract) must not index the ring
    or the pool out of range: rows and ring tokens at negative positions
    count one fault each, the rest equals the same tokens started at 0."""
    rows, w, fr, pt, pr = _setup(9, 20)
    for freqs in (None, fr):
        pool = np.zeros(pr * 528, np.uint8)
        ring = np.full((1, 3, 1024), 0x3F80, np.uint16)
        res = oracle.compress_store(oracle.V41, 2, rows[0:9].copy(), np.array([[0], [9]], np.int32),
                                    page_table=pt, page_bits=3, norm_w=w, freqs=freqs,
                                    start_pos=np.array([-5], np.int32), pool=pool, pool_rows=pr,
                                    ring=ring)
        # positions -5..3: rows c = -3, -2, -1 (pos < 0) and ring token -2 are faults
        assert res["faults"] == 4 and res["total"] == 5
        assert np.array_equal(ring[0, 0], rows[5]) and np.array_equal(ring[0, 1], rows[7])
        assert (ring[0, 2] == 0x3F80).all()
        fresh = np.zeros(pr * 528, np.uint8)
        oracle.compress_store(oracle.V41, 2, rows[5:9].copy(), np.array([[0], [4]], np.int32),
                              page_table=pt, page_bits=3, norm_w=w, freqs=freqs,
                              start_pos=np.array([0], np.int32), pool=fresh, pool_rows=pr,
                              ring=np.zeros((1, 3, 1024), np.uint16))
        assert np.array_equal(pool, fresh)
