"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Covers the V41 round trip and ratio-2 compressor workloads, brute-force tiny
ragged cases over both layouts, both ratios and every norm/rope combination,
the padding / out_loc == 0 / fault rules, dequant of arbitrary bytes, the
top-k -> slot mapping, the reuse buffer, CUDA-graph replay with offsets
refreshed in place, and byte determinism with a negative control."""
import hashlib

import numpy as np
import pytest
import torch

import oracle
from deepseek_v4_compressed_c2_gb300 import workloads as W
from parity import (assert_bf16_equal_nan_aware, assert_prequant_close,
                    compare_rows_end_to_end, dev, dev_bf16, host_u16)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from deepseek_v4_compressed_c2_gb300 import build as b
    b.build()
    from deepseek_v4_compressed_c2_gb300 import binding
    binding.lib()
    return binding


def gpu_store(B, cfg, *, out_loc=None, n_out=None, pool_fill=0, want_pre=True, want_lat=True,
              score=None):
    rb = oracle.row_bytes(cfg["layout"])
    n_out = cfg["n_out"] if n_out is None else n_out
    pool = torch.full((cfg["pool_rows"] * rb,), pool_fill, dtype=torch.uint8, device="cuda")
    pre = torch.full((n_out, 512), 7.0, dtype=torch.float32, device="cuda") if want_pre else None
    lat = torch.full((n_out, 512), 7.0, dtype=torch.bfloat16, device="cuda") if want_lat else None
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.dsv4kv_compress_store(
        cfg["layout"], cfg["ratio"], dev_bf16(cfg["rows"]), dev(cfg["ext"]), pool,
        score=None if score is None else dev_bf16(score),
        page_table=None if cfg["page_table"] is None else dev(cfg["page_table"]),
        page_bits=cfg["page_bits"],
        rmsnorm_w=None if cfg["norm_w"] is None else dev_bf16(cfg["norm_w"]), eps=cfg["eps"],
        freqs_cis=None if cfg["freqs"] is None else dev(cfg["freqs"]),
        out_loc=None if out_loc is None else dev(out_loc), n_out=n_out,
        latent_out=lat, prequant_out=pre, err_word=err)
    torch.cuda.synchronize()
    return dict(pool=pool.cpu().numpy(), err=int(err.item()),
                pre=None if pre is None else pre.cpu().numpy(),
                lat=None if lat is None else host_u16(lat))


def oracle_store(cfg, *, out_loc=None, n_out=None, pool_fill=0, prequant_in=None, score=None):
    rb = oracle.row_bytes(cfg["layout"])
    pool = np.full(cfg["pool_rows"] * rb, pool_fill, np.uint8)
    res = oracle.compress_store(
        cfg["layout"], cfg["ratio"], cfg["rows"], cfg["ext"], score=score,
        page_table=cfg["page_table"], page_bits=cfg["page_bits"], norm_w=cfg["norm_w"],
        eps=cfg["eps"], freqs=cfg["freqs"], out_loc=out_loc,
        n_out=cfg["n_out"] if n_out is None else n_out, pool=pool, pool_rows=cfg["pool_rows"],
        prequant_in=prequant_in)
    res["pool"] = pool
    return res


def check_store(B, cfg, *, out_loc=None, min_allowed=0, exact_codes=False):
    """Full parity of one compress_store call: identical-input bytes, end-to-end
    tolerance, latent, padding, untouched bytes."""
    g = gpu_store(B, cfg, out_loc=out_loc, pool_fill=0xA5)
    ref = oracle_store(cfg, out_loc=out_loc, pool_fill=0xA5)
    same = oracle_store(cfg, out_loc=out_loc, pool_fill=0xA5, prequant_in=g["pre"])
    assert g["err"] == ref["faults"]
    # codes and scales bit-exact given the GPU's own fp32 pre-quant rows
    assert np.array_equal(g["pool"], same["pool"])
    total = ref["total"]
    assert_prequant_close(g["pre"][:total], ref["prequant_f64"][:total])
    assert not g["pre"][total:].any() and not g["lat"][total:].any()
    # latent (bf16, post-norm pre-RoPE) within the same tolerance
    lat_g = oracle.bf16_to_f64(g["lat"][:total])
    lat_r = oracle.bf16_to_f64(ref["latent"][:total])
    ulp = np.abs(lat_r) * 2.0 ** -7
    assert np.all(np.abs(lat_g - lat_r) <= ulp + 1e-5 * np.abs(lat_r).max(axis=1, keepdims=True))
    rb = oracle.row_bytes(cfg["layout"])
    gp = g["pool"].reshape(-1, rb)
    rp = ref["pool"].reshape(-1, rb)
    written = ~np.all(rp == 0xA5, axis=1) | ~np.all(gp == 0xA5, axis=1)
    assert np.array_equal(np.all(gp == 0xA5, axis=1), np.all(rp == 0xA5, axis=1))
    if exact_codes:
        assert np.array_equal(gp, rp)
    elif written.any():
        pre_by_slot = np.zeros((gp.shape[0], 512))
        slots = _slots_of(cfg, out_loc, total)
        ok = (slots > 0) & (slots < cfg["pool_rows"])
        pre_by_slot[slots[ok]] = ref["prequant_f64"][:total][ok]
        compare_rows_end_to_end(cfg["layout"], gp[written], rp[written], pre_by_slot[written],
                                min_allowed=min_allowed)
    return g, ref


def _slots_of(cfg, out_loc, total):
    if out_loc is not None:
        return np.asarray(out_loc[:total], np.int64)
    p = oracle.plan(cfg["ratio"], cfg["ext"], cfg["page_table"], cfg["page_bits"])
    return p["slot"]


# ---------------------------------------------------------------- configs
def test_v41_round_trip_256_rows_bit_exact(B):
    cfg = W.cfg1_v41_roundtrip()
    g, ref = check_store(B, cfg, exact_codes=True)
    ids = np.arange(64, 64 + 256, dtype=np.int32)
    out = B.dsv4kv_dequant_gather(cfg["layout"], dev(g["pool"]), dev(ids))
    want, _ = oracle.dequant_gather(cfg["layout"], ref["pool"], cfg["pool_rows"], ids)
    assert np.array_equal(host_u16(out), want)


def test_ratio2_compressor_4_requests(B):
    cfg = W.cfg2_ratio2_small()
    g, ref = check_store(B, cfg)
    assert ref["total"] == 1809
    # explicit out_loc from the plan, with some real rows marked 0 (not stored)
    p = oracle.plan(2, cfg["ext"], cfg["page_table"], cfg["page_bits"])
    out_loc = np.zeros(cfg["n_out"], np.int32)
    out_loc[:p["total"]] = p["slot"]
    out_loc[::7] = 0
    check_store(B, cfg, out_loc=out_loc)


def test_ratio2_separate_score_buffer_matches_fused(B):
    cfg = W.cfg2_ratio2_small()
    fused = gpu_store(B, cfg)
    split = dict(cfg)
    split["rows"] = np.ascontiguousarray(cfg["rows"][:, :512])
    score = np.ascontiguousarray(cfg["rows"][:, 512:])
    g = gpu_store(B, split, score=score)
    assert np.array_equal(g["pool"], fused["pool"])
    assert np.array_equal(g["pre"], fused["pre"])


# ------------------------------------------------------------ brute force
def _random_case(seed):
    rng = np.random.default_rng(1000 + seed)
    layout = [oracle.V41, oracle.V41_FP4, oracle.V4][seed % 3]
    ratio = 1 + (seed // 2) % 2
    norm = bool(rng.integers(0, 2))
    rope = bool(rng.integers(0, 2))
    n_req = int(rng.integers(0, 6))
    lens = [int(v) for v in rng.integers(0, 150, n_req)]
    if n_req and seed % 5 == 0:
        lens[0] = 1                                           # a lone (odd) token
    page_bits = int(rng.integers(0, 6))
    per = [n // ratio for n in lens]
    pages = [-(-p // (1 << page_bits)) for p in per]
    phys = rng.permutation(sum(pages) + 3) + 1
    max_pages = max([1] + pages)
    pt = np.zeros((max(n_req, 1) + 2, max_pages), np.int32)
    o = 0
    for r, p in enumerate(pages):
        pt[r, :p] = phys[o:o + p]
        o += p
    pool_rows = (sum(pages) + 4) << page_bits
    t = sum(lens) + 3
    scale = rng.choice([1.0, 1e-3, 30.0])
    x = (rng.standard_normal((t, 1024)) * scale).astype(np.float32)
    x[rng.random(x.shape) < 0.01] *= 50
    rows = W.bf16_from_f32(x)
    ext = np.zeros((2, max(n_req, 1) + 2), np.int32)
    ext[0, :n_req] = np.concatenate([[0], np.cumsum(lens)[:-1]]) if n_req else []
    ext[1, :n_req] = lens
    total = sum(per)
    n_out = total + int(rng.integers(0, 40))
    return dict(layout=layout, ratio=ratio, rows=rows, ext=ext, page_table=pt,
                page_bits=page_bits, norm_w=W.bf16_from_f32(rng.uniform(0.5, 1.5, 512).astype(np.float32)) if norm else None,
                freqs=W.rope_table(512) if rope else None, eps=1e-6, n_out=max(n_out, 1),
                pool_rows=pool_rows)


@pytest.mark.parametrize("seed", range(36))
def test_brute_force_tiny_cases(B, seed):
    cfg = _random_case(seed)
    check_store(B, cfg, min_allowed=2)


def test_every_layout_ratio_norm_rope_combination(B):
    base = W.cfg2_ratio2_small()
    for layout in (oracle.V41, oracle.V41_FP4, oracle.V4):
        for ratio in (1, 2):
            for norm in (False, True):
                for rope in (False, True):
                    cfg = dict(base, layout=layout, ratio=ratio,
                               norm_w=base["norm_w"] if norm else None,
                               freqs=base["freqs"] if rope else None, n_out=2048)
                    if ratio == 1:
                        cfg["n_out"] = 3620 + 20
                        cfg["pool_rows"] = 130 << 6
                        pt = np.zeros((8, 64), np.int32)
                        o = 1
                        for r, n in enumerate(base["lengths"]):
                            k = -(-n // 64)
                            pt[r, :k] = np.arange(o, o + k)
                            o += k
                        cfg["page_table"] = pt
                    check_store(B, cfg, min_allowed=3)


@pytest.mark.parametrize("layout", [oracle.V41, oracle.V41_FP4, oracle.V4])
def test_ratio1_store_only_row_states_and_faults(B, layout):
    """The store-only ratio-1 launch (one row per half-warp) against the
    oracle with rows of every state next to each other in a warp: valid rows,
    rows of a request that starts before the rows buffer or runs past it
    (faults; zeroed debug outputs), padding past the plan's total, and
    destinations that are padding (0), past the pool or negative (faults).
    Store-only rows are exact bf16, so the pool must equal the oracle's
    byte for byte."""
    rng = np.random.default_rng(41 + layout)
    lens = [37, 5, 64, 3, 90, 1]
    n_rows = sum(lens)
    rows = W.bf16_normal(rng, (n_rows, 512))
    ext = np.zeros((2, len(lens)), np.int32)
    ext[0] = np.concatenate([[0], np.cumsum(lens)[:-1]])
    ext[1] = lens
    ext[0, 1] = -3                       # starts before the rows buffer
    ext[0, 3] = n_rows - 1               # runs two rows past it
    total = n_rows
    n_out = total + 11                   # padding rows at the end
    pool_rows = 512
    out_loc = (rng.permutation(pool_rows - 1)[:n_out] + 1).astype(np.int32)
    out_loc[[4, 40, 41]] = 0             # padding destinations: not stored, no fault
    out_loc[[7, 100]] = pool_rows        # past the pool: faults
    out_loc[[12, 150]] = -9              # negative: faults
    cfg = dict(layout=layout, ratio=1, rows=rows, score=None, ext=ext, page_table=None,
               page_bits=6, norm_w=None, freqs=None, eps=1e-6, n_out=n_out,
               pool_rows=pool_rows)
    g, ref = check_store(B, cfg, out_loc=out_loc, exact_codes=True)
    assert g["err"] == ref["faults"] == 9
    # output rows of source rows -3..-1 (request 1) and n_rows, n_rows + 1
    # (request 3): faults with zeroed debug outputs
    bad = np.array([37, 38, 39, 107, 108])
    assert not g["pre"][bad].any() and not g["lat"][bad].any()


# ------------------------------------------------------------ edge cases
def test_empty_and_all_padding_calls(B):
    cfg = W.cfg1_v41_roundtrip()
    cfg0 = dict(cfg, ext=np.zeros((2, 3), np.int32), n_out=50,
                page_table=np.ones((3, 4), np.int32))
    g = gpu_store(B, cfg0, pool_fill=0x33)
    assert (g["pool"] == 0x33).all() and not g["pre"].any() and g["err"] == 0
    cfg_none = dict(cfg, ext=np.zeros((2, 0), np.int32), n_out=8)
    g = gpu_store(B, cfg_none, pool_fill=0x33)
    assert (g["pool"] == 0x33).all() and not g["pre"].any()
    pool = torch.zeros(100, dtype=torch.uint8, device="cuda")
    B.dsv4kv_compress_store(1, 1, dev_bf16(cfg["rows"]), dev(cfg["ext"]), pool,
                            page_table=dev(cfg["page_table"]), page_bits=6, n_out=0)
    out = B.dsv4kv_dequant_gather(1, pool, torch.zeros(0, dtype=torch.int32, device="cuda"))
    assert out.shape == (0, 512)


def test_device_faults_are_counted_not_trapped(B):
    cfg = W.cfg2_ratio2_small()
    bad = dict(cfg, ext=cfg["ext"].copy(), freqs=W.rope_table(600))
    bad["ext"][1, 3] = 2047 + 2000          # request 3 runs past the rows buffer
    bad["ext"][0, 2] = -5                   # a negative first row
    g = gpu_store(B, bad, pool_fill=0xA5)
    ref = oracle_store(bad, pool_fill=0xA5)
    assert g["err"] == ref["faults"] > 0
    same = oracle_store(bad, pool_fill=0xA5, prequant_in=g["pre"])
    assert np.array_equal(g["pool"], same["pool"])
    # destinations outside the pool and past the page table
    cfg1 = W.cfg1_v41_roundtrip()
    out_loc = np.arange(64, 64 + 256, dtype=np.int32)
    out_loc[[3, 9]] = [cfg1["pool_rows"], -7]
    g = gpu_store(B, cfg1, out_loc=out_loc, pool_fill=0xA5)
    assert g["err"] == 2
    short_pt = dict(cfg1, page_table=cfg1["page_table"][:, :2].copy())
    g = gpu_store(B, short_pt, pool_fill=0xA5)
    assert g["err"] == 128
    # gather: ids past the pool are faults and zero rows, negative ids zero rows
    pool = dev(oracle_store(cfg1)["pool"])
    ids = np.array([64, -1, 320, 1 << 30, 70], np.int32)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = host_u16(B.dsv4kv_dequant_gather(1, pool, dev(ids), err_word=err))
    want, faults = oracle.dequant_gather(1, pool.cpu().numpy(), cfg1["pool_rows"], ids)
    assert int(err.item()) == faults == 2
    assert np.array_equal(out, want)


def test_host_argument_errors_raise(B):
    cfg = W.cfg1_v41_roundtrip()
    pool = torch.zeros(cfg["pool_rows"] * 528, dtype=torch.uint8, device="cuda")
    with pytest.raises(B.DSV4KVError) as e:
        B.dsv4kv_compress_store(9, 1, dev_bf16(cfg["rows"]), dev(cfg["ext"]), pool,
                                page_table=dev(cfg["page_table"]), page_bits=6, n_out=4)
    assert e.value.status == -1
    with pytest.raises(B.DSV4KVError):
        B.dsv4kv_compress_store(1, 3, dev_bf16(cfg["rows"]), dev(cfg["ext"]), pool,
                                page_table=dev(cfg["page_table"]), page_bits=6, n_out=4)
    with pytest.raises(B.DSV4KVError):
        B.dsv4kv_dequant_gather(1, pool[1:], torch.zeros(4, dtype=torch.int32, device="cuda"))


@pytest.mark.parametrize("layout", [oracle.V41, oracle.V41_FP4, oracle.V4])
def test_dequant_of_arbitrary_bytes(B, layout):
    rng = np.random.default_rng(77 + layout)
    rb = oracle.row_bytes(layout)
    n = 777
    pool = rng.integers(0, 256, (n, rb), dtype=np.uint8)
    if layout == oracle.V41:
        pool[:, 512:] = rng.integers(0, 256, (n, 16), dtype=np.uint8)
        pool[:4, 512:] = [[0], [1], [254], [255]]           # scale-byte extremes
    if layout == oracle.V4:
        pool[:4, 576:] = [[0], [1], [254], [255]]
    ids = rng.permutation(n).astype(np.int32)
    out = host_u16(B.dsv4kv_dequant_gather(layout, dev(pool.reshape(-1)), dev(ids)))
    want, _ = oracle.dequant_gather(layout, pool.reshape(-1), n, ids)
    assert_bf16_equal_nan_aware(out, want)


@pytest.mark.parametrize("k,offset", [(333, 0), (332, 0), (332, 1), (2048, 0)])
def test_topk_to_slots_matches_oracle(B, k, offset):
    rng = np.random.default_rng(8 + k + offset)
    n_req, page_bits = 9, 4
    pt = rng.integers(1, 5000, (n_req, 40), dtype=np.int32)
    topk = rng.integers(-2, 40 << page_bits, (50, k), dtype=np.int32)
    topk[3, 5] = 45 << page_bits                              # past max_pages
    ttr = rng.integers(0, n_req, 50).astype(np.int32)
    ttr[7] = n_req + 3                                         # bad request
    valid = (rng.random(50) > 0.2).astype(np.uint8)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    # offset 1: topk and slots start 4 bytes past a 16-byte boundary
    topk_d = dev(np.concatenate([[0] * offset, topk.reshape(-1)]).astype(np.int32))[offset:].view(50, k)
    slots_buf = torch.empty(50 * k + offset, dtype=torch.int32, device="cuda")
    slots, lens = B.dsv4kv_topk_to_slots(topk_d, dev(ttr), dev(pt), page_bits, is_valid=dev(valid),
                                         slots=slots_buf[offset:].view(50, k), err_word=err)
    ws, wl, faults = oracle.topk_to_slots(topk, ttr, pt, page_bits, is_valid=valid)
    assert np.array_equal(slots.cpu().numpy(), ws)
    assert np.array_equal(lens.cpu().numpy(), wl)
    assert int(err.item()) == faults


def test_reuse_buffer_hits_equal_a_fresh_dequant(B):
    """Layers sharing a kv_source reuse one dequant; the reused rows equal a
    fresh dequant of the same rows (sglang PR #45909 verification)."""
    cfg = W.cfg2_ratio2_small()
    g = gpu_store(B, cfg)
    pool = dev(g["pool"])
    ids = dev(np.random.default_rng(3).permutation(np.arange(64, 4160))[:1500].astype(np.int32))
    buf = B.SparsePrefillKVBuffer(torch.empty((2048, 512), dtype=torch.bfloat16, device="cuda"))
    buf.dsv4kv_kvbuf_begin_forward()
    hits = []
    for _layer in range(4):
        rows, hit = buf.dsv4kv_kvbuf_get_with_head(1, pool, ids)
        hits.append(hit)
    assert hits == [False, True, True, True] and buf.dequants == 1
    fresh = B.dsv4kv_dequant_gather(1, pool, ids)
    assert torch.equal(rows.view(torch.int16), fresh.view(torch.int16))
    buf.dsv4kv_kvbuf_get(10)                                  # plain get forgets
    _, hit = buf.dsv4kv_kvbuf_get_with_head(1, pool, ids)
    assert not hit and buf.dequants == 2


def test_cuda_graph_replay_with_offsets_refreshed_in_place(B):
    cfg = W.cfg2_ratio2_small()
    rb = 528
    rows = dev_bf16(cfg["rows"])
    ext = dev(cfg["ext"])
    pt = dev(cfg["page_table"])
    w = dev_bf16(cfg["norm_w"])
    fr = dev(cfg["freqs"])
    pool = torch.zeros(cfg["pool_rows"] * rb, dtype=torch.uint8, device="cuda")
    ids = dev(np.arange(64, 64 + 512, dtype=np.int32))
    out = torch.empty((512, 512), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        B.dsv4kv_compress_store(1, 2, rows, ext, pool, page_table=pt, page_bits=6, rmsnorm_w=w,
                                freqs_cis=fr, n_out=2048)       # warm-up outside capture
        B.dsv4kv_dequant_gather(1, pool, ids, out)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        B.dsv4kv_compress_store(1, 2, rows, ext, pool, page_table=pt, page_bits=6, rmsnorm_w=w,
                                freqs_cis=fr, n_out=2048)
        B.dsv4kv_dequant_gather(1, pool, ids, out)
    for lens in ([37, 512, 1024, 2047], [100, 0, 900, 13], [0, 0, 0, 3000]):
        new_ext = W._ext(lens, n_slots=8, pad_first=sum(lens))
        ext.copy_(dev(new_ext))                                 # refreshed in place
        pool.zero_()
        graph.replay()
        torch.cuda.synchronize()
        c = dict(cfg, ext=new_ext)
        ref_pool = gpu_store(B, c)["pool"]
        assert np.array_equal(pool.cpu().numpy(), ref_pool)
        want = B.dsv4kv_dequant_gather(1, dev(ref_pool), ids)
        assert torch.equal(out.view(torch.int16), want.view(torch.int16))


def test_determinism_and_negative_control(B):
    cfg = W.cfg2_ratio2_small()
    h = []
    for eps in (1e-6, 1e-6, 1e-6 + 1e-3):
        g = gpu_store(B, dict(cfg, eps=eps))
        m = hashlib.sha256()
        m.update(g["pool"].tobytes())
        m.update(g["pre"].tobytes())
        m.update(g["lat"].tobytes())
        h.append(m.hexdigest())
    assert h[0] == h[1]
    assert h[2] != h[0]


@pytest.mark.parametrize("layout", [oracle.V41, oracle.V41_FP4, oracle.V4])
def test_pool_bytes_do_not_depend_on_the_debug_outputs(B, layout):
    """With RMSNorm the V41 store folds the norm scale into its power-of-two
    multiplier when no pre-quant output is requested; the bytes must equal
    those of the explicit path that writes prequant_out."""
    cfg = dict(W.cfg2_ratio2_small(), layout=layout)
    with_dbg = gpu_store(B, cfg, want_pre=True, want_lat=True)
    without = gpu_store(B, cfg, want_pre=False, want_lat=False)
    assert np.array_equal(with_dbg["pool"], without["pool"])


@pytest.mark.parametrize("layout,n_tok,k", [(oracle.V41, 37, 515), (oracle.V41_FP4, 37, 515),
                                            (oracle.V4, 37, 515), (oracle.V41, 101, 5),
                                            (oracle.V41_FP4, 77, 3)])
def test_fused_topk_gather_matches_oracle_composition(B, layout, n_tok, k):
    """dsv4kv_dequant_gather_topk == oracle top-k -> slots then gather, with
    lens and every fault kind (bad request, page past the table, slot past the
    pool), on a pool written by the store; k = 3 or 5 puts many tokens in one
    32-row tile of the bulk-copy gather."""
    cfg = dict(W.cfg2_ratio2_small(), layout=layout)
    pool = gpu_store(B, cfg)["pool"]
    rng = np.random.default_rng(31 + layout + k)
    pt = cfg["page_table"].copy()
    pt[7, 0] = 70                                   # a page past the pool (65 pages)
    topk = rng.integers(-3, 1100, (n_tok, k), dtype=np.int32)
    topk[2, :min(k, 7)] = 16 * 64 + np.arange(min(k, 7))   # page index 16 >= max_pages
    ttr = rng.integers(0, 8, n_tok).astype(np.int32)
    ttr[5] = 9                                      # request outside the table
    ttr[6] = 7
    topk[6, 0] = 5                                  # request 7, page 0 -> past the pool
    valid = (rng.random(n_tok) > 0.15).astype(np.uint8)
    valid[6] = 1
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    lens = torch.zeros(n_tok, dtype=torch.int32, device="cuda")
    out = B.dsv4kv_dequant_gather_topk(layout, dev(pool), dev(topk), dev(ttr), dev(pt), 6,
                                       is_valid=dev(valid), lens=lens, err_word=err)
    ws, wl, f1 = oracle.topk_to_slots(topk, ttr, pt, 6, is_valid=valid)
    want, f2 = oracle.dequant_gather(layout, pool, cfg["pool_rows"], ws.reshape(-1))
    assert_bf16_equal_nan_aware(host_u16(out), want)
    assert np.array_equal(lens.cpu().numpy(), wl)
    assert int(err.item()) == f1 + f2 and f1 > 0 and f2 > 0


@pytest.mark.parametrize("layout", [oracle.V41, oracle.V41_FP4, oracle.V4])
def test_page_entries_that_are_no_page_fault_and_give_zero_rows(B, layout):
    """A negative page-table entry, one whose slot would wrap a 32-bit shift
    back into the pool (2^26 pages of 64 rows), and one whose slot fits int32
    but lies past the pool: the standalone mapping and the fused gather both
    give slot -1 / a zero row and count one fault per entry, as the oracle
    does (64-bit slots, no wrap)."""
    cfg = dict(W.cfg2_ratio2_small(), layout=layout)
    pool = gpu_store(B, cfg)["pool"]
    pt = cfg["page_table"].copy()
    pt[0, 0] = -5
    pt[1, 0] = (1 << 26) + 2            # (2^26 + 2) << 6 wraps to slot 128 in 32 bits
    pt[2, 0] = (1 << 24)                # slot 2^30: fits int32, past the 65-page pool
    topk = np.tile(np.array([[3, 9, 40, 63, -1, 70]], np.int32), (6, 1))
    ttr = np.array([0, 1, 2, 3, 0, 1], np.int32)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    slots, lens = B.dsv4kv_topk_to_slots(dev(topk), dev(ttr), dev(pt), 6, err_word=err)
    ws, wl, f1 = oracle.topk_to_slots(topk, ttr, pt, 6)
    assert np.array_equal(slots.cpu().numpy(), ws)
    assert np.array_equal(lens.cpu().numpy(), wl)
    assert int(err.item()) == f1 and f1 == 16          # 4 ids x 4 tokens on entries 0 and 1
    assert (ws[[0, 1, 4, 5], :4] == -1).all() and (ws[2, :4] >= 1 << 30).all()
    err.zero_()
    lens = torch.zeros(6, dtype=torch.int32, device="cuda")
    out = B.dsv4kv_dequant_gather_topk(layout, dev(pool), dev(topk), dev(ttr), dev(pt), 6,
                                       lens=lens, err_word=err)
    want, f2 = oracle.dequant_gather(layout, pool, cfg["pool_rows"], ws.reshape(-1))
    assert_bf16_equal_nan_aware(host_u16(out), want)
    assert np.array_equal(lens.cpu().numpy(), wl)
    assert int(err.item()) == f1 + f2 and f2 == 4      # token 2's slots lie past the pool
    assert not host_u16(out).reshape(6, 6, 512)[[0, 1, 2, 4, 5], :4].any()


def test_fused_topk_reuse_buffer(B):
    cfg = W.cfg2_ratio2_small()
    pool = dev(gpu_store(B, cfg)["pool"])
    topk = dev(np.random.default_rng(4).integers(-1, 1000, (16, 256), dtype=np.int32))
    ttr = dev(np.arange(16, dtype=np.int32) % 4)
    pt = dev(cfg["page_table"])
    buf = B.SparsePrefillKVBuffer(torch.empty((4096, 512), dtype=torch.bfloat16, device="cuda"))
    buf.dsv4kv_kvbuf_begin_forward()
    hits = [buf.dsv4kv_kvbuf_get_with_head_topk(1, pool, topk, ttr, pt, 6)[1] for _ in range(4)]
    assert hits == [False, True, True, True] and buf.dequants == 1
    fresh = B.dsv4kv_dequant_gather_topk(1, pool, topk, ttr, pt, 6)
    assert torch.equal(buf.storage[:4096].view(torch.int16), fresh.view(torch.int16))


def test_maximum_slots_and_page_size(B):
    """4096 request slots (the plan's capacity, many of them empty or odd) and
    2^16-row pages (page_bits 16) against the oracle."""
    rng = np.random.default_rng(44)
    n_slots = 4096
    lens = rng.integers(0, 6, n_slots)
    lens[rng.random(n_slots) < 0.5] = 0
    rows = W.bf16_from_f32(rng.standard_normal((int(lens.sum()) + 1, 1024)).astype(np.float32))
    ext = W._ext([int(v) for v in lens])
    pt = np.zeros((n_slots, 1), np.int32)
    per = lens // 2
    # every request's rows fit in one 2^16-row page: give each slot its own
    # in-page window by using out_loc for the destination instead
    p = oracle.plan(2, ext, None, 0)
    out_loc = np.zeros(p["total"] + 7, np.int32)
    out_loc[:p["total"]] = 1 + rng.permutation(p["total"])
    cfg = dict(layout=oracle.V41, ratio=2, rows=rows, ext=ext, page_table=pt, page_bits=16,
               norm_w=None, freqs=W.rope_table(16), eps=1e-6, n_out=p["total"] + 7,
               pool_rows=p["total"] + 1)
    check_store(B, cfg, out_loc=out_loc, min_allowed=2)
    # page_bits 16 through the page table: 3 pages of 65536 rows
    big = dict(layout=oracle.V41_FP4, ratio=1, rows=W.bf16_from_f32(
        rng.standard_normal((70000, 512)).astype(np.float32)), ext=W._ext([70000]),
        page_table=np.array([[2, 1]], np.int32), page_bits=16, norm_w=None, freqs=None,
        eps=1e-6, n_out=70000, pool_rows=3 << 16)
    check_store(B, big, exact_codes=True)


def test_bounded_wait_reports_a_timeout_instead_of_hanging(B):
    """A wait on an mbarrier nothing arrives on gives up after its poll limit,
    reports exactly one timeout fault, the other waiter leaves through the
    abort flag, and the context stays usable."""
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    gave_up = torch.zeros(1, dtype=torch.int32, device="cuda")
    st = B.lib().dsv4kv_selftest_bounded_wait(1 << 14, err.data_ptr(), gave_up.data_ptr(),
                                              torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    assert int(err.item()) == 1 << 24 and int(gave_up.item()) == 2
    assert B.lib().dsv4kv_selftest_bounded_wait(0, err.data_ptr(), gave_up.data_ptr(), None) == -3
    # the context still works
    cfg = W.cfg1_v41_roundtrip()
    g = gpu_store(B, cfg)
    ref = oracle_store(cfg)
    assert np.array_equal(g["pool"], ref["pool"])


def test_fp4_quotient_matches_ieee_division_for_every_scale(B):
    """The FP4 quantizer divides by the e4m3 scale with a correctly rounded
    reciprocal and one correction step; it must equal the IEEE division bit
    for bit, for all 126 positive finite e4m3 divisors, on random fp32
    dividends over the quantizer's range and on dividends at and next to
    every e2m1 rounding midpoint times the divisor."""
    g = torch.Generator(device="cuda")
    g.manual_seed(123)
    codes = torch.arange(1, 127, dtype=torch.uint8, device="cuda")          # 0x01..0x7E
    s = torch.from_numpy(np.array([oracle.e4m3_value(c) for c in range(1, 127)], np.float32)).cuda()
    per = 1 << 17
    # random dividends: |x| up to 8 s, and tiny ones, both signs
    u = torch.rand((126, per), generator=g, device="cuda")
    x_rand = (u * 8 - 4) * s[:, None] * 2
    x_tiny = (torch.rand((126, per // 8), generator=g, device="cuda") - 0.5) * s[:, None] * 2.0 ** -20
    # near ties: t * s with the fp32 neighbours, t every e2m1 midpoint and value
    t = torch.tensor([0.25, 0.5, 0.75, 1, 1.25, 1.5, 1.75, 2, 2.5, 3, 3.5, 4, 5, 6, 7],
                     device="cuda")
    base = (t[None, :] * s[:, None]).contiguous()
    bits = base.view(torch.int32)
    near = torch.cat([(bits + d).view(torch.float32) for d in range(-8, 9)], dim=1)
    x = torch.cat([x_rand, x_tiny, near, -near], dim=1).contiguous()
    sc = codes[:, None].expand_as(x).contiguous()
    q_fast = torch.empty_like(x)
    q_ieee = torch.empty_like(x)
    st = B.lib().dsv4kv_selftest_fp4_quotient(x.data_ptr(), sc.data_ptr(), x.numel(),
                                              q_fast.data_ptr(), q_ieee.data_ptr(),
                                              torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    bad = q_fast.view(torch.int32) != q_ieee.view(torch.int32)
    assert int(bad.sum()) == 0, f"{int(bad.sum())} quotients differ, e.g. {x[bad][:4].tolist()}"


def test_fp4_reciprocal_is_the_ieee_reciprocal_for_every_scale(B):
    """The FP4 quantizer's reciprocal of the e4m3 scale (one Newton-Raphson
    step from the hardware approximation) equals the IEEE reciprocal, and
    hence the oracle's fp64 1/s rounded to fp32, for all 126 positive finite
    e4m3 codes."""
    codes = torch.arange(1, 127, dtype=torch.uint8, device="cuda")
    y_fast = torch.empty(126, dtype=torch.float32, device="cuda")
    y_ieee = torch.empty_like(y_fast)
    st = B.lib().dsv4kv_selftest_e4m3_recip(codes.data_ptr(), 126, y_fast.data_ptr(),
                                            y_ieee.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    want = np.array([1.0 / oracle.e4m3_value(c) for c in range(1, 127)]).astype(np.float32)
    assert np.array_equal(y_ieee.cpu().numpy().view(np.int32), want.view(np.int32))
    assert np.array_equal(y_fast.cpu().numpy().view(np.int32), want.view(np.int32))


@pytest.mark.parametrize("layout", [oracle.V41, oracle.V41_FP4, oracle.V4])
def test_guard_regions_around_pool_output_and_ring_stay_untouched(B, layout):
    """The pool, the gathered output and the ring sit inside larger buffers
    whose guard regions are sentinel-filled; no call writes outside its
    buffers (slots and ids include the first and last rows and out-of-range
    values)."""
    rb = oracle.row_bytes(layout)
    G = 1 << 16                                           # guard bytes each side
    cfg = dict(W.decode_verify(seed=21, n_req=48, n_new=5, ring_size=4, max_prefix=256),
               layout=layout)
    pool_bytes = cfg["pool_rows"] * rb
    big = torch.full((pool_bytes + 2 * G,), 0x5C, dtype=torch.uint8, device="cuda")
    pool = big[G:G + pool_bytes]
    ring_big = torch.full((cfg["ring"].size + 2 * G,), 0x1234, dtype=torch.int16, device="cuda")
    ring = ring_big[G:G + cfg["ring"].size].view(torch.bfloat16).view(cfg["ring"].shape)
    ring.copy_(dev_bf16(cfg["ring"]))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    # slots: the plan's, plus the pool's last row and out-of-range values
    p = oracle.plan(2, cfg["ext"], cfg["page_table"], cfg["page_bits"], start_pos=cfg["start_pos"])
    out_loc = p["slot"].astype(np.int32).copy()
    out_loc[:3] = [cfg["pool_rows"] - 1, cfg["pool_rows"], -1]
    B.dsv4kv_compress_store(layout, 2, dev_bf16(cfg["rows"]), dev(cfg["ext"]), pool,
                            page_table=dev(cfg["page_table"]), page_bits=cfg["page_bits"],
                            rmsnorm_w=dev_bf16(cfg["norm_w"]), eps=cfg["eps"],
                            freqs_cis=dev(cfg["freqs"]), out_loc=dev(out_loc),
                            err_word=err, start_pos=dev(cfg["start_pos"]), ring=ring)
    ids = np.array([0, cfg["pool_rows"] - 1, cfg["pool_rows"], -5, 1 << 30, 7], np.int32)
    out_big = torch.full(((len(ids) + 2) * 512,), 0x3A3A, dtype=torch.int16, device="cuda")
    out = out_big[512:512 + len(ids) * 512].view(torch.bfloat16).view(len(ids), 512)
    B.dsv4kv_dequant_gather(layout, pool, dev(ids), out, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 2 + 2                       # two bad slots, two bad ids
    assert bool((big[:G] == 0x5C).all()) and bool((big[G + pool_bytes:] == 0x5C).all())
    assert bool((ring_big[:G] == 0x1234).all()) and bool((ring_big[G + cfg["ring"].size:] == 0x1234).all())
    assert bool((out_big[:512] == 0x3A3A).all()) and bool((out_big[512 + len(ids) * 512:] == 0x3A3A).all())


def test_back_to_back_launches_see_the_previous_kernels_writes(B):
    """The store and the gather are launched to start early (programmatic
    dependent launch) and must still see what the kernel just before them
    wrote.  Each round: a torch kernel writes the store's input rows (a row
    permutation), the store writes the pool, the gather reads the rows just
    stored, the next round's torch kernel overwrites the inputs -- with no
    synchronisation anywhere.  The results equal a run synchronised after
    every launch."""
    cfg = W.cfg2_ratio2_small()
    base = dev_bf16(cfg["rows"])
    ext, pt = dev(cfg["ext"]), dev(cfg["page_table"])
    w, fr = dev_bf16(cfg["norm_w"]), dev(cfg["freqs"])
    plan = oracle.plan(2, cfg["ext"], cfg["page_table"], cfg["page_bits"])
    ids = dev(np.ascontiguousarray(plan["slot"][:plan["total"]]).astype(np.int32))
    g = torch.Generator(device="cuda")
    g.manual_seed(5)
    rounds = 6
    perms = [torch.randperm(base.shape[0], generator=g, device="cuda") for _ in range(rounds)]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")

    def run(sync):
        rows = torch.empty_like(base)
        pool = torch.zeros(cfg["pool_rows"] * 528, dtype=torch.uint8, device="cuda")
        outs = [torch.empty((ids.numel(), 512), dtype=torch.bfloat16, device="cuda")
                for _ in range(rounds)]
        for r in range(rounds):
            torch.index_select(base, 0, perms[r], out=rows)
            if sync:
                torch.cuda.synchronize()
            B.dsv4kv_compress_store(1, 2, rows, ext, pool, page_table=pt, page_bits=cfg["page_bits"],
                                    rmsnorm_w=w, eps=cfg["eps"], freqs_cis=fr,
                                    n_out=cfg["n_out"], err_word=err)
            if sync:
                torch.cuda.synchronize()
            B.dsv4kv_dequant_gather(1, pool, ids, outs[r], err_word=err)
            if sync:
                torch.cuda.synchronize()
        torch.cuda.synchronize()
        return [host_u16(o) for o in outs]

    fast, slow = run(False), run(True)
    assert int(err.item()) == 0
    for r in range(rounds):
        assert np.array_equal(fast[r], slow[r]), f"round {r}"
    assert not np.array_equal(slow[0], slow[1])          # the rounds do differ



@pytest.mark.parametrize("layout,k", [(oracle.V41, 512), (oracle.V41_FP4, 130), (oracle.V4, 7)])
def test_short_context_ids_and_fused_gather_match_oracle(B, layout, k):
    """dsv4kv_fill_all_compressed_indices == the oracle's fill, and
    dsv4kv_dequant_gather_all == oracle fill -> topk_to_slots -> gather (bit
    exact, lens, faults), on a pool written by the store."""
    cfg = dict(W.cfg2_ratio2_small(), layout=layout)
    pool = gpu_store(B, cfg)["pool"]
    rng = np.random.default_rng(41 + layout + k)
    n_tok = 45
    lens_in = rng.integers(-2, k + 40, n_tok).astype(np.int32)
    lens_in[:3] = [0, k, 1]
    pt = cfg["page_table"].copy()
    pt[7, 0] = 70                                   # a page past the pool (65 pages)
    ttr = rng.integers(0, 8, n_tok).astype(np.int32)
    ttr[5] = 9                                      # request outside the table
    ttr[6], lens_in[6] = 7, 3                       # request 7, page 0 -> past the pool
    valid = (rng.random(n_tok) > 0.15).astype(np.uint8)
    valid[6] = 1
    ids = B.dsv4kv_fill_all_compressed_indices(dev(lens_in), k)
    torch.cuda.synchronize()
    want_ids = oracle.fill_all_indices(lens_in, k)
    assert np.array_equal(ids.cpu().numpy(), want_ids)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    lens = torch.zeros(n_tok, dtype=torch.int32, device="cuda")
    out = B.dsv4kv_dequant_gather_all(layout, dev(pool), dev(lens_in), k, dev(ttr), dev(pt), 6,
                                      is_valid=dev(valid), lens=lens, err_word=err)
    ws, wl, f1 = oracle.topk_to_slots(want_ids, ttr, pt, 6, is_valid=valid)
    want, f2 = oracle.dequant_gather(layout, pool, cfg["pool_rows"], ws.reshape(-1))
    assert_bf16_equal_nan_aware(host_u16(out), want)
    assert np.array_equal(lens.cpu().numpy(), wl)
    assert int(err.item()) == f1 + f2 and f1 > 0 and f2 > 0


@pytest.mark.parametrize("layout", [oracle.V41, oracle.V41_FP4, oracle.V4])
def test_fake_quant_matches_oracle_and_store_then_gather(B, layout):
    """dsv4kv_fake_quant == the oracle's dequant(store_row(x)) bit for bit
    (rows with outliers, all-zero rows), from a strided input and in place,
    and == a store-only dsv4kv_compress_store followed by dsv4kv_dequant_gather."""
    rng = np.random.default_rng(61 + layout)
    n = 333
    x32 = rng.standard_normal((n, 512)).astype(np.float32)
    x32[rng.random((n, 512)) < 0.01] *= 50
    x32[7] = 0.0
    x = W.bf16_from_f32(x32)
    want = oracle.bf16_bits(oracle.dequant_rows(layout, oracle.quantize_rows(layout, oracle.bf16_to_f64(x))))
    wide = torch.zeros((n, 1024), dtype=torch.bfloat16, device="cuda")
    wide[:, :512] = dev_bf16(x)
    out = B.dsv4kv_fake_quant(layout, wide[:, :512])
    torch.cuda.synchronize()
    assert np.array_equal(host_u16(out), want)
    inplace = dev_bf16(x).contiguous()
    B.dsv4kv_fake_quant(layout, inplace, inplace)
    torch.cuda.synchronize()
    assert np.array_equal(host_u16(inplace), want)
    # the same through the pool: store-only rows 1..n, gathered back
    rb = oracle.row_bytes(layout)
    pool = torch.zeros((n + 1) * rb, dtype=torch.uint8, device="cuda")
    ext = torch.tensor([[0], [n]], dtype=torch.int32, device="cuda")
    B.dsv4kv_compress_store(layout, 1, dev_bf16(x), ext, pool,
                            out_loc=torch.arange(1, n + 1, dtype=torch.int32, device="cuda"),
                            n_out=n)
    back = B.dsv4kv_dequant_gather(layout, pool, torch.arange(1, n + 1, dtype=torch.int32,
                                                             device="cuda"))
    torch.cuda.synchronize()
    assert np.array_equal(host_u16(back), want)


def test_requests_past_65536_rows_plan_and_store_bit_exact(B):
    """No 16-bit limit in the plan: one request of 70,001 rows and another of
    65,536 (ratio 1, store-only, random permuted page table) store every row
    at its page-table slot, bit-exact against the oracle."""
    rng = np.random.default_rng(65)
    lens = [70001, 65536, 3]
    n_rows = sum(lens)
    rows = W.bf16_from_f32(rng.standard_normal((n_rows, 512)).astype(np.float32))
    ext = np.array([[0, lens[0], lens[0] + lens[1]], lens], np.int32)
    pages = [-(-n // 64) for n in lens]
    perm = rng.permutation(sum(pages)).astype(np.int32) + 1
    pt = np.zeros((3, max(pages)), np.int32)
    o = 0
    for r, p in enumerate(pages):
        pt[r, :p] = perm[o:o + p]
        o += p
    pool_rows = (sum(pages) + 1) * 64
    cfg = dict(layout=oracle.V41, ratio=1, rows=rows, ext=ext, page_table=pt, page_bits=6,
               norm_w=None, eps=1e-6, freqs=None, n_out=n_rows, pool_rows=pool_rows)
    g = gpu_store(B, cfg, pool_fill=0xA5, want_pre=False, want_lat=False)
    ref = oracle_store(cfg, pool_fill=0xA5)
    assert g["err"] == ref["faults"] == 0 and ref["total"] == n_rows
    assert np.array_equal(g["pool"], ref["pool"])
