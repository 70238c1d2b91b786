"""GPU parity of the start-position / pair-state-ring form of the compressor
(decode, speculative verify, chunked prefill) against the CPU oracle, and
chunking invariance on the GPU itself."""
import numpy as np
import pytest
import torch

import oracle
from deepseek_v4_compressed_c2_gb300 import workloads as W
from parity import assert_prequant_close, compare_rows_end_to_end, dev, dev_bf16, host_u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from deepseek_v4_compressed_c2_gb300 import build as b
    b.build()
    from deepseek_v4_compressed_c2_gb300 import binding
    binding.lib()
    return binding


def gpu_step(B, cfg, pool, ring, *, want_pre=True):
    pre = torch.zeros((max(cfg["n_out"], 1), 512), dtype=torch.float32, device="cuda") if want_pre else None
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.dsv4kv_compress_store(cfg["layout"], 2, dev_bf16(cfg["rows"]), dev(cfg["ext"]), pool,
                            page_table=dev(cfg["page_table"]), page_bits=cfg["page_bits"],
                            rmsnorm_w=dev_bf16(cfg["norm_w"]), eps=cfg["eps"],
                            freqs_cis=dev(cfg["freqs"]), n_out=cfg["n_out"], prequant_out=pre,
                            err_word=err, start_pos=dev(cfg["start_pos"]), ring=ring)
    torch.cuda.synchronize()
    return None if pre is None else pre.cpu().numpy(), int(err.item())


# The ring form's launch follows the rows per SM: at most 16 (512 x 1 .. 7,
# 4096 x 1, 320 x 9: up to ~2000 rows) take the decode kernel (one chunk of
# request slots per CTA; 4096 slots is its largest step), more (2048 x 5,
# 1024 x 9: ~5000, ~4600 rows) the streaming kernel; the x 9 steps have
# n >= 2R, so the ring update rewrites the entry the step's first pair
# reads, and 512 x 7 makes chunks of more than 16 rows (overflow rows).
@pytest.mark.parametrize("n_new,layout,n_req", [(1, oracle.V41, 512), (4, oracle.V41, 512),
                                                (4, oracle.V41_FP4, 512), (7, oracle.V41, 512),
                                                (7, oracle.V41_FP4, 512), (7, oracle.V4, 512),
                                                (5, oracle.V41, 2048), (1, oracle.V41, 4096),
                                                (9, oracle.V41, 320), (9, oracle.V4, 1024)])
def test_decode_verify_step_matches_oracle(B, n_new, layout, n_req):
    cfg = dict(W.decode_verify(seed=11 + n_new, n_req=n_req, n_new=n_new, ring_size=4,
                               max_prefix=1024), layout=layout)
    rb = oracle.row_bytes(layout)
    pool = torch.full((cfg["pool_rows"] * rb,), 0xA5, dtype=torch.uint8, device="cuda")
    ring = dev_bf16(cfg["ring"])
    pre, err = gpu_step(B, cfg, pool, ring)
    ref_pool = np.full(cfg["pool_rows"] * rb, 0xA5, np.uint8)
    ref_ring = cfg["ring"].copy()
    kw = dict(page_table=cfg["page_table"], page_bits=cfg["page_bits"], norm_w=cfg["norm_w"],
              eps=cfg["eps"], freqs=cfg["freqs"], n_out=cfg["n_out"], start_pos=cfg["start_pos"])
    ref = oracle.compress_store(layout, 2, cfg["rows"], cfg["ext"], pool=ref_pool,
                                pool_rows=cfg["pool_rows"], ring=ref_ring, **kw)
    assert err == ref["faults"] == 0
    assert ref["total"] == cfg["n_out"]
    # the ring after the step: an exact copy of the right tokens
    assert np.array_equal(host_u16(ring).reshape(ref_ring.shape), ref_ring)
    # pre-quant within tolerance; bytes exact given the GPU's fp32 rows
    assert_prequant_close(pre[:ref["total"]], ref["prequant_f64"][:ref["total"]])
    same_pool = np.full(cfg["pool_rows"] * rb, 0xA5, np.uint8)
    oracle.compress_store(layout, 2, cfg["rows"], cfg["ext"], pool=same_pool,
                          pool_rows=cfg["pool_rows"], ring=cfg["ring"].copy(), prequant_in=pre, **kw)
    got = pool.cpu().numpy()
    assert np.array_equal(got, same_pool)
    p = oracle.plan(2, cfg["ext"], cfg["page_table"], cfg["page_bits"], start_pos=cfg["start_pos"])
    gp = got.reshape(-1, rb)[p["slot"]]
    rp = ref_pool.reshape(-1, rb)[p["slot"]]
    compare_rows_end_to_end(layout, gp, rp, ref["prequant_f64"], min_allowed=2)
    assert (p["src"] < 0).sum() > 0                 # ring-sourced rows were exercised


def test_gpu_chunked_prefill_with_ring_equals_whole(B):
    rng = np.random.default_rng(5)
    n = 301
    rows = W.bf16_from_f32(rng.standard_normal((n, 1024)).astype(np.float32))
    w = W.bf16_from_f32(rng.uniform(0.5, 1.5, 512).astype(np.float32))
    pt = (rng.permutation(3) + 1).astype(np.int32).reshape(1, -1)
    base = dict(layout=oracle.V41, norm_w=w, freqs=W.rope_table(512), eps=1e-6,
                page_table=pt, page_bits=6, pool_rows=4 << 6)

    def run(cuts):
        pool = torch.zeros(base["pool_rows"] * 528, dtype=torch.uint8, device="cuda")
        ring = torch.zeros((1, 3, 1024), dtype=torch.bfloat16, device="cuda")
        for a, b in zip(cuts[:-1], cuts[1:]):
            cfg = dict(base, rows=np.ascontiguousarray(rows[a:b]),
                       ext=np.array([[0], [b - a]], np.int32), start_pos=np.array([a], np.int32),
                       n_out=((b >> 1) - (a >> 1)))
            if cfg["n_out"] == 0:
                cfg["n_out"] = 1
            _, err = gpu_step(B, cfg, pool, ring, want_pre=False)
            assert err == 0
        return pool.cpu().numpy()

    whole = run([0, n])
    for cuts in ([0, 1, n], [0, 77, 78, 79, n], [0, 150, 151, 300, n], list(range(0, 40)) + [n]):
        assert np.array_equal(run(cuts), whole)


def test_ring_row_without_ring_is_a_counted_fault(B):
    cfg = W.decode_verify(seed=3, n_req=64, n_new=1, max_prefix=1024)
    pool = torch.zeros(cfg["pool_rows"] * 528, dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.dsv4kv_compress_store(1, 2, dev_bf16(cfg["rows"]), dev(cfg["ext"]), pool,
                            page_table=dev(cfg["page_table"]), page_bits=cfg["page_bits"],
                            n_out=cfg["n_out"], err_word=err, start_pos=dev(cfg["start_pos"]))
    torch.cuda.synchronize()
    assert int(err.item()) == int((cfg["start_pos"] % 2 == 1).sum()) == cfg["n_out"]


@pytest.mark.parametrize("rope", [False, True])
def test_negative_start_positions_fault_like_the_oracle(B, rope):
    rng = np.random.default_rng(21)
    n_req, R = 6, 3
    p0 = np.array([-5, -1, -2, 3, -7, 0], np.int32)
    n = np.array([9, 4, 1, 5, 2, 6], np.int32)
    first = np.concatenate([[0], np.cumsum(n)[:-1]]).astype(np.int32)
    rows = W.bf16_from_f32(rng.standard_normal((int(n.sum()), 1024)).astype(np.float32))
    ring0 = W.bf16_from_f32(rng.standard_normal((n_req, R, 1024)).astype(np.float32))
    w = W.bf16_from_f32(rng.uniform(0.5, 1.5, 512).astype(np.float32))
    pt = (rng.permutation(n_req) + 1).astype(np.int32).reshape(n_req, 1)
    ext = np.stack([first, n]).astype(np.int32)
    fr = W.rope_table(64) if rope else None
    n_out = int(sum(((a + b) >> 1) - (a >> 1) for a, b in zip(p0.tolist(), n.tolist())))
    pool_rows = (n_req + 1) << 6
    pool = torch.full((pool_rows * 528,), 0xA5, dtype=torch.uint8, device="cuda")
    ring = dev_bf16(ring0)
    pre = torch.zeros((n_out, 512), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.dsv4kv_compress_store(oracle.V41, 2, dev_bf16(rows), dev(ext), pool, page_table=dev(pt),
                            page_bits=6, rmsnorm_w=dev_bf16(w), eps=1e-6,
                            freqs_cis=None if fr is None else dev(fr), n_out=n_out,
                            prequant_out=pre, err_word=err, start_pos=dev(p0), ring=ring)
    torch.cuda.synchronize()
    ref_ring = ring0.copy()
    ref_pool = np.full(pool_rows * 528, 0xA5, np.uint8)
    pre_h = pre.cpu().numpy()
    ref = oracle.compress_store(oracle.V41, 2, rows, ext, page_table=pt, page_bits=6, norm_w=w,
                                eps=1e-6, freqs=fr, n_out=n_out, start_pos=p0, pool=ref_pool,
                                pool_rows=pool_rows, ring=ref_ring, prequant_in=pre_h)
    assert ref["faults"] > 0 and int(err.item()) == ref["faults"]
    assert np.array_equal(host_u16(ring).reshape(ref_ring.shape), ref_ring)
    assert np.array_equal(pool.cpu().numpy(), ref_pool)


@pytest.mark.parametrize("n_new,n_req", [(1, 300), (4, 300), (9, 300), (1, 2800), (9, 320),
                                         (9, 640)])
def test_ring_form_with_separate_score_or_padded_stride_equals_fused(B, n_new, n_req):
    """The ring form reading kv and score from separate buffers, or from rows
    padded to 1536 elements, writes the same pool and ring bytes as the fused
    | kv | score | rows (the decode kernel's loads and ring copies, ring-sourced
    pairs included, and the streaming kernel's per-half copies for 640 x 9)."""
    cfg = W.decode_verify(seed=30 + n_new, n_req=n_req, n_new=n_new, ring_size=4, max_prefix=512)
    rows = dev_bf16(cfg["rows"])
    common = dict(page_table=dev(cfg["page_table"]), page_bits=cfg["page_bits"],
                  rmsnorm_w=dev_bf16(cfg["norm_w"]), eps=cfg["eps"], freqs_cis=dev(cfg["freqs"]),
                  n_out=cfg["n_out"], start_pos=dev(cfg["start_pos"]))

    def run(r, score=None):
        pool = torch.zeros(cfg["pool_rows"] * 528, dtype=torch.uint8, device="cuda")
        ring = dev_bf16(cfg["ring"])
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        B.dsv4kv_compress_store(1, 2, r, dev(cfg["ext"]), pool, score=score, ring=ring,
                                err_word=err, **common)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        return pool.cpu().numpy(), host_u16(ring)

    fused = run(rows)
    kv = rows[:, :512].contiguous()
    sc = rows[:, 512:].contiguous()
    split = run(kv, score=sc)
    padded = torch.zeros((rows.shape[0], 1536), dtype=torch.bfloat16, device="cuda")
    padded[:, :1024] = rows
    wide = run(padded[:, :1024].as_strided((rows.shape[0], 1024), (1536, 1)))
    for got in (split, wide):
        assert np.array_equal(got[0], fused[0]) and np.array_equal(got[1], fused[1])


@pytest.mark.parametrize("n_new,n_req", [(3, 200), (9, 200), (9, 640), (9, 1280)])
def test_ring_form_with_fewer_output_rows_than_the_step_makes(B, n_new, n_req):
    """n_out below the step's row count: rows k >= n_out are neither computed
    nor stored, in the tiles and in the ring phase (n >= 2R rows), while the
    ring is still updated for every request, as in the oracle (the decode
    kernel, whose chunk prefix then saturates at n_out, up to 640 x 9; the
    streaming kernel for 1280 x 9 with n_out = half its ~5760 rows)."""
    cfg = W.decode_verify(seed=50 + n_new, n_req=n_req, n_new=n_new, ring_size=4, max_prefix=512)
    n_out = cfg["n_out"] // 2
    cfg = dict(cfg, n_out=n_out, layout=oracle.V41)
    pool = torch.full((cfg["pool_rows"] * 528,), 0xA5, dtype=torch.uint8, device="cuda")
    ring = dev_bf16(cfg["ring"])
    pre, err = gpu_step(B, cfg, pool, ring)
    ref_ring = cfg["ring"].copy()
    same_pool = np.full(cfg["pool_rows"] * 528, 0xA5, np.uint8)
    ref = oracle.compress_store(oracle.V41, 2, cfg["rows"], cfg["ext"], page_table=cfg["page_table"],
                                page_bits=cfg["page_bits"], norm_w=cfg["norm_w"], eps=cfg["eps"],
                                freqs=cfg["freqs"], n_out=n_out, start_pos=cfg["start_pos"],
                                pool=same_pool, pool_rows=cfg["pool_rows"], ring=ref_ring,
                                prequant_in=pre)
    assert err == ref["faults"] == 0
    assert np.array_equal(pool.cpu().numpy(), same_pool)
    assert np.array_equal(host_u16(ring).reshape(ref_ring.shape), ref_ring)


@pytest.mark.parametrize("form", ["odd_slots", "no_start", "no_ring", "out_loc", "latent",
                                  "padded"])
def test_decode_kernel_launch_forms_match_oracle(B, form):
    """The decode kernel (steps of at most 16 rows per SM) in its other launch
    forms, against the oracle: a slot count that is no multiple of 4 (the
    plan's scalar loads), no start positions (every slot starts at 0), start
    positions without a ring (ring rows are faults), out_loc with padding
    zeros, the latent output, and n_out past the step's rows (the padding
    rows' latent and pre-quant outputs zeroed over a sentinel).  Pool bytes
    exact given the GPU's fp32 rows, ring and fault count equal."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    n_req, n_new = {"odd_slots": (2801, 1), "no_start": (1400, 2)}.get(form, (2800, 1))
    cfg = W.decode_verify(seed=60 + len(form), n_req=n_req, n_new=n_new, ring_size=4,
                          max_prefix=512)
    start = None if form == "no_start" else cfg["start_pos"]
    ring0 = None if form == "no_ring" else cfg["ring"]
    p = oracle.plan(2, cfg["ext"], cfg["page_table"], cfg["page_bits"], start_pos=start)
    n_out = p["total"] + (300 if form == "padded" else 0)
    assert n_out <= 16 * sms, "the case must take the decode kernel"
    out_loc = None
    if form == "out_loc":
        out_loc = p["slot"].astype(np.int32)
        out_loc[::7] = 0
    pool = torch.full((cfg["pool_rows"] * 528,), 0xA5, dtype=torch.uint8, device="cuda")
    ring = None if ring0 is None else dev_bf16(ring0)
    pre = torch.full((n_out, 512), 7.0, dtype=torch.float32, device="cuda")
    lat = (torch.full((n_out, 512), 7.0, dtype=torch.bfloat16, device="cuda")
           if form in ("latent", "padded") else None)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.dsv4kv_compress_store(oracle.V41, 2, dev_bf16(cfg["rows"]), dev(cfg["ext"]), pool,
                            page_table=dev(cfg["page_table"]), page_bits=cfg["page_bits"],
                            rmsnorm_w=dev_bf16(cfg["norm_w"]), eps=cfg["eps"],
                            freqs_cis=dev(cfg["freqs"]), n_out=n_out,
                            out_loc=None if out_loc is None else dev(out_loc),
                            latent_out=lat, prequant_out=pre, err_word=err,
                            start_pos=None if start is None else dev(start), ring=ring)
    torch.cuda.synchronize()
    pre_h = pre.cpu().numpy()
    ref_pool = np.full(cfg["pool_rows"] * 528, 0xA5, np.uint8)
    ref_ring = None if ring0 is None else ring0.copy()
    ref = oracle.compress_store(oracle.V41, 2, cfg["rows"], cfg["ext"], page_table=cfg["page_table"],
                                page_bits=cfg["page_bits"], norm_w=cfg["norm_w"], eps=cfg["eps"],
                                freqs=cfg["freqs"], out_loc=out_loc, n_out=n_out, start_pos=start,
                                pool=ref_pool, pool_rows=cfg["pool_rows"], ring=ref_ring,
                                prequant_in=pre_h)
    assert int(err.item()) == ref["faults"]
    if form == "no_ring":
        assert ref["faults"] == int((cfg["start_pos"] % 2 == 1).sum()) > 0
    assert np.array_equal(pool.cpu().numpy(), ref_pool)
    if ref_ring is not None:
        assert np.array_equal(host_u16(ring).reshape(ref_ring.shape), ref_ring)
    if form == "padded":
        tot = p["total"]
        assert not pre[tot:].any() and not lat[tot:].any()
        assert np.isfinite(pre_h[:tot]).all()
    e2e = oracle.compress_store(oracle.V41, 2, cfg["rows"], cfg["ext"], page_table=cfg["page_table"],
                                page_bits=cfg["page_bits"], norm_w=cfg["norm_w"], eps=cfg["eps"],
                                freqs=cfg["freqs"], out_loc=out_loc, n_out=n_out, start_pos=start,
                                ring=None if ring0 is None else ring0.copy())
    ok = np.abs(e2e["prequant_f64"]).max(axis=1) > 0
    assert_prequant_close(pre_h[ok], e2e["prequant_f64"][ok])
    if lat is not None:
        lat_g = oracle.bf16_to_f64(host_u16(lat))
        lat_r = oracle.bf16_to_f64(e2e["latent"])
        tol = np.abs(lat_r) * 2.0 ** -7 + 1e-5 * np.abs(lat_r).max(axis=1, keepdims=True)
        assert np.all(np.abs(lat_g - lat_r) <= tol)


@pytest.mark.parametrize("rows_layout", ["packed", "shuffled"])
def test_decode_kernel_mixed_step_with_long_requests(B, rows_layout):
    """A step that mixes 600 decode requests with a few long ones, all in the
    decode kernel (at most 16 rows per SM): requests of 80 new tokens at an
    odd start make chunks of 40+ rows (overflow rows taken by other CTAs'
    spare warps) and 40 ring tokens each (more than the ring warp's 32
    stages, so it moves them in two batches); one request of 130 tokens at
    an odd start has n >= 2R, so its ring update follows its first row in
    that row's warp.  The requests' rows either packed back to back in slot
    order or in a shuffled order with gaps of 0-3 rows.  Ring, pool bytes
    (given the GPU's fp32 rows) and fault count equal the oracle's; pre-quant
    within tolerance."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    rng = np.random.default_rng(71)
    n_req, R = 600, 64
    lengths = [1] * n_req
    p0 = rng.integers(0, 2048, n_req).astype(np.int32)
    for r, n in ((5, 80), (6, 80), (300, 80), (599, 80), (301, 130)):
        lengths[r] = n
        p0[r] |= 1                                   # odd start: the first pair reads the ring
    if rows_layout == "packed":
        ext = W._ext(lengths)
    else:
        first, cursor = np.zeros(n_req, np.int64), 0
        for r in rng.permutation(n_req):
            first[r] = cursor + int(rng.integers(0, 4))
            cursor = int(first[r]) + lengths[r]
        ext = np.stack([first, np.array(lengths)]).astype(np.int32)
        assert (ext[0][1:] != ext[0][:-1] + ext[1][:-1]).any()
    rows = W.bf16_normal(rng, (int((ext[0] + ext[1]).max()), 1024))
    ring0 = W.bf16_normal(rng, (n_req, R, 1024))
    norm_w = W.bf16_from_f32(rng.uniform(0.5, 1.5, 512).astype(np.float32))
    max_c = (2048 + 130) // 2 + 1
    pt, n_pages = W._page_table(rng, [-(-max_c // 64)] * n_req)
    n_out = int(sum(((int(a) + n) >> 1) - (int(a) >> 1) for a, n in zip(p0, lengths)))
    assert n_out <= 16 * sms, "the step must take the decode kernel"
    cfg = dict(layout=oracle.V41, rows=rows, ext=ext, start_pos=p0, page_table=pt, page_bits=6,
               norm_w=norm_w, eps=1e-6, freqs=W.rope_table(2048 + 132), n_out=n_out,
               pool_rows=n_pages << 6)
    pool = torch.full((cfg["pool_rows"] * 528,), 0xA5, dtype=torch.uint8, device="cuda")
    ring = dev_bf16(ring0)
    pre, err = gpu_step(B, cfg, pool, ring)
    kw = dict(page_table=pt, page_bits=6, norm_w=norm_w, eps=1e-6, freqs=cfg["freqs"], n_out=n_out,
              start_pos=p0)
    ref_ring = ring0.copy()
    ref_pool = np.full(cfg["pool_rows"] * 528, 0xA5, np.uint8)
    ref = oracle.compress_store(oracle.V41, 2, rows, ext, pool=ref_pool, pool_rows=cfg["pool_rows"],
                                ring=ref_ring, **kw)
    assert err == ref["faults"] == 0
    assert np.array_equal(host_u16(ring).reshape(ref_ring.shape), ref_ring)
    assert_prequant_close(pre[:n_out], ref["prequant_f64"][:n_out])
    same_pool = np.full(cfg["pool_rows"] * 528, 0xA5, np.uint8)
    oracle.compress_store(oracle.V41, 2, rows, ext, pool=same_pool, pool_rows=cfg["pool_rows"],
                          ring=ring0.copy(), prequant_in=pre, **kw)
    assert np.array_equal(pool.cpu().numpy(), same_pool)


def test_decode_steps_in_a_cuda_graph_with_metadata_refreshed_in_place(B):
    """The serving loop's shape: one decode step (1024 requests x 1 new token,
    ring of 4) captured in a CUDA graph and replayed for 4 consecutive steps,
    with the new tokens' rows and the start positions written into the same
    device buffers before each replay (positions advance by one; n_out is the
    graph-static upper bound, so about half the rows are padding).  After
    every step the pool (given the GPU's fp32 rows) and the pair-state ring
    equal the oracle's, run step by step on the carried state."""
    rng = np.random.default_rng(81)
    n_req, R, steps = 1024, 4, 4
    p0 = rng.integers(0, 1024, n_req).astype(np.int32)
    norm_w = W.bf16_from_f32(rng.uniform(0.5, 1.5, 512).astype(np.float32))
    freqs = W.rope_table(1024 + steps + 2)
    pt, n_pages = W._page_table(rng, [-(-((1024 + steps) // 2 + 1) // 64)] * n_req)
    ext = W._ext([1] * n_req)
    ring0 = W.bf16_normal(rng, (n_req, R, 1024))
    pool_rows = n_pages << 6
    d_rows = torch.empty((n_req, 1024), dtype=torch.bfloat16, device="cuda")
    d_start = torch.empty(n_req, dtype=torch.int32, device="cuda")
    d_ext, d_pt = dev(ext), dev(pt)
    ring = dev_bf16(ring0)
    pool = torch.full((pool_rows * 528,), 0xA5, dtype=torch.uint8, device="cuda")
    pre = torch.zeros((n_req, 512), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    # preparing runs the launch once, and one more warms it outside the
    # capture: both on valid inputs, then the state is put back
    d_rows.zero_()
    d_start.copy_(dev(p0))
    keep_ring, keep_pool = ring.clone(), pool.clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        call = B.prepare_compress_store(1, 2, d_rows, d_ext, pool, page_table=d_pt, page_bits=6,
                                        rmsnorm_w=dev_bf16(norm_w), eps=1e-6,
                                        freqs_cis=dev(freqs), n_out=n_req, prequant_out=pre,
                                        err_word=err, stream=s, start_pos=d_start, ring=ring)
        call()
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ring.copy_(keep_ring)
    pool.copy_(keep_pool)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        call()
    ref_ring, ref_pool = ring0.copy(), np.full(pool_rows * 528, 0xA5, np.uint8)
    for step in range(steps):
        rows = W.bf16_normal(rng, (n_req, 1024))
        start = p0 + step
        d_rows.copy_(dev_bf16(rows))                      # refreshed in place
        d_start.copy_(dev(start.astype(np.int32)))
        graph.replay()
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        kw = dict(page_table=pt, page_bits=6, norm_w=norm_w, eps=1e-6, freqs=freqs, n_out=n_req,
                  start_pos=start.astype(np.int32))
        oracle.compress_store(oracle.V41, 2, rows, ext, pool=ref_pool, pool_rows=pool_rows,
                              ring=ref_ring, prequant_in=pre.cpu().numpy(), **kw)
        assert np.array_equal(host_u16(ring).reshape(ref_ring.shape), ref_ring), step
        assert np.array_equal(pool.cpu().numpy(), ref_pool), step


@pytest.mark.parametrize("n_slots", [0, 5])
def test_ring_form_step_without_new_tokens_writes_only_padding(B, n_slots):
    """A ring-form step with n_out > 0 but no new tokens (no request slots, or
    slots whose counts are all zero) takes the decode kernel and makes no
    rows: the pre-quant output is zeroed over its sentinel, the pool and the
    ring stay as they were, no fault."""
    rng = np.random.default_rng(5 + n_slots)
    R, n_out = 4, 8
    ext = np.zeros((2, n_slots), np.int32)
    p0 = rng.integers(0, 100, n_slots).astype(np.int32)
    ring0 = W.bf16_normal(rng, (max(n_slots, 1), R, 1024))
    rows = W.bf16_normal(rng, (4, 1024))
    pt = np.ones((max(n_slots, 1), 4), np.int32)
    pool = torch.full((4 * 64 * 528,), 0x33, dtype=torch.uint8, device="cuda")
    pre = torch.full((n_out, 512), 7.0, dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ring = dev_bf16(ring0)
    B.dsv4kv_compress_store(oracle.V41, 2, dev_bf16(rows), dev(ext), pool, page_table=dev(pt),
                            page_bits=6, n_out=n_out, prequant_out=pre, err_word=err,
                            start_pos=dev(p0), ring=ring)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert bool((pool == 0x33).all()) and not bool(pre.any())
    assert np.array_equal(host_u16(ring).reshape(ring0.shape), ring0)
