"""Host-side checks of the C ABI that need no GPU: the library builds and
loads, exports every function include/dsv4kv.h declares, reports the page's
row sizes, rejects host-checkable bad arguments before touching CUDA, and its
reuse-buffer head follows the reference model's trace (sglang PR #45909)."""
import ctypes
import json
import os
import re

import pytest

from oracle.kvbuf_model import KVBufModel

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def B():
    from deepseek_v4_compressed_c2_gb300 import build as b
    b.build()
    from deepseek_v4_compressed_c2_gb300 import binding
    binding.lib()
    return binding


def _declared():
    with open(os.path.join(ROOT, "include", "dsv4kv.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dsv4kv_\w+)\s*\(", text)))


def test_every_declared_symbol_is_exported(B):
    names = _declared()
    assert "dsv4kv_compress_store" in names and "dsv4kv_dequant_gather" in names
    lib = ctypes.CDLL(B._LIB_PATH)
    for n in names:
        assert hasattr(lib, n), f"{n} declared but not exported"


def test_row_bytes_and_status_strings(B, golden_dir):
    with open(os.path.join(golden_dir, "kvlayout_row_bytes.json")) as f:
        rb = json.load(f)["row_bytes"]
    L = B.lib()
    assert L.dsv4kv_row_bytes(0) == rb["V4"]
    assert L.dsv4kv_row_bytes(1) == rb["V41"]
    assert L.dsv4kv_row_bytes(2) == rb["V41_FP4"]
    assert L.dsv4kv_row_bytes(3) == -1
    for s in (0, -1, -2, -3, -4, -99):
        assert L.dsv4kv_status_string(s)


FAKE = 1 << 20          # a 16-B aligned non-null stand-in; never dereferenced


def _store(L, **kw):
    a = dict(layout=1, ratio=2, rows=FAKE, n_rows=100, row_stride=1024, score=None,
             score_stride=0, ext=FAKE, n_slots=4, pt=FAKE, max_pages=4, page_bits=6,
             w=None, eps=1e-6, freqs=None, max_pos=0, out_loc=None, n_out=10, pool=FAKE,
             pool_rows=1000, lat=None, pre=None, err=None, stream=None)
    a.update(kw)
    return L.dsv4kv_compress_store(*a.values())


def test_compress_store_rejects_bad_arguments_before_any_launch(B):
    L = B.lib()
    assert _store(L, layout=7) == -1
    assert _store(L, layout=-1) == -1
    assert _store(L, ratio=3) == -1
    assert _store(L, page_bits=17) == -1
    assert _store(L, n_out=-1) == -1
    assert _store(L, n_slots=5000) == -3
    assert _store(L, pool_rows=1 << 31) == -3
    assert _store(L, rows=None) == -1
    assert _store(L, rows=FAKE + 8) == -1                  # misaligned
    assert _store(L, row_stride=1000) == -1                # fused ratio 2 needs 1024
    assert _store(L, row_stride=1028) == -1                # not a 16-B multiple
    assert _store(L, pt=None) == -1                        # no out_loc and no table
    assert _store(L, freqs=FAKE, max_pos=0) == -1
    assert _store(L, eps=-1.0) == -1
    assert _store(L, score=FAKE, ratio=1, row_stride=512) == -1
    assert _store(L, n_out=0) == 0                         # no-op, nothing launched


def test_dequant_and_topk_reject_bad_arguments(B):
    L = B.lib()
    assert L.dsv4kv_dequant_gather(5, FAKE, 10, FAKE, 4, FAKE, None, None) == -1
    assert L.dsv4kv_dequant_gather(0, FAKE, 10, None, 4, FAKE, None, None) == -1
    assert L.dsv4kv_dequant_gather(1, FAKE, 10, FAKE, -1, FAKE, None, None) == -1
    assert L.dsv4kv_dequant_gather(1, FAKE, 10, None, 4, FAKE, None, None) == -1
    assert L.dsv4kv_dequant_gather(1, FAKE, 10, FAKE, 4, FAKE + 2, None, None) == -1
    assert L.dsv4kv_dequant_gather(1, FAKE, 1 << 31, FAKE, 4, FAKE, None, None) == -3
    assert L.dsv4kv_dequant_gather(1, None, 10, None, 0, None, None, None) == 0
    assert L.dsv4kv_topk_to_slots(FAKE, 4, 70000, FAKE, None, FAKE, 2, 2, 6, FAKE, None, None, None) == -3
    assert L.dsv4kv_topk_to_slots(FAKE, 4, 8, FAKE, None, FAKE, 2, 2, 20, FAKE, None, None, None) == -1
    assert L.dsv4kv_topk_to_slots(FAKE, 0, 8, FAKE, None, FAKE, 2, 2, 6, FAKE, None, None, None) == 0


SOURCES = {"A": (1, 0x1000, 4096, 0x9000), "B": (1, 0x2000, 4096, 0xA000),
           "A2": (1, 0x1000, 4096, 0xB000)}


def test_reuse_head_follows_the_reference_trace(B, golden_dir):
    with open(os.path.join(golden_dir, "kvbuf_trace.json")) as f:
        g = json.load(f)
    L = B.lib()
    buf = B.dsv4kv_kvbuf()
    model = KVBufModel(g["capacity"])
    assert L.dsv4kv_kvbuf_init(ctypes.byref(buf), FAKE, g["capacity"]) == 0
    hit = ctypes.c_int()
    for op in g["ops"]:
        if op[0] == "begin_forward":
            L.dsv4kv_kvbuf_begin_forward(ctypes.byref(buf))
            model.begin_forward()
        elif op[0] == "get":
            assert L.dsv4kv_kvbuf_get(ctypes.byref(buf), op[1], None) == 0
            model.get(op[1])
        elif op[0] == "realloc":
            assert L.dsv4kv_kvbuf_init(ctypes.byref(buf), FAKE + 4096, op[1]) == 0
            model.realloc(op[1])
        else:
            layout, pool, rows, ids = SOURCES[op[1]]
            assert L.dsv4kv_kvbuf_lookup(ctypes.byref(buf), layout, pool, rows, ids, op[2],
                                         ctypes.byref(hit)) == 0
            want = model.get_with_head(layout, pool, rows, ids, op[2])
            assert bool(hit.value) == want == op[3]
    # capacity: ERANGE, and the head is left as it was
    assert L.dsv4kv_kvbuf_lookup(ctypes.byref(buf), 1, 1, 1, 1, g["capacity"] + 1,
                                 ctypes.byref(hit)) == -3
    assert L.dsv4kv_kvbuf_get(ctypes.byref(buf), g["capacity"] + 1, None) == -3


def test_get_with_head_of_zero_rows_needs_no_launch(B):
    L = B.lib()
    buf = B.dsv4kv_kvbuf()
    assert L.dsv4kv_kvbuf_init(ctypes.byref(buf), FAKE, 8) == 0
    hit = ctypes.c_int()
    rows = ctypes.c_void_p()
    for want in (0, 1, 1):
        assert L.dsv4kv_kvbuf_get_with_head(ctypes.byref(buf), 1, FAKE, 10, FAKE, 0,
                                            ctypes.byref(rows), ctypes.byref(hit), None, None) == 0
        assert hit.value == want and rows.value == FAKE
    assert L.dsv4kv_kvbuf_init(ctypes.byref(buf), FAKE + 8, 8) == -1   # misaligned storage


def _ring(L, **kw):
    a = dict(layout=1, ratio=2, rows=FAKE, n_rows=100, row_stride=1024, score=None,
             score_stride=0, ext=FAKE, n_slots=4, start=FAKE, ring=FAKE, ring_size=4, pt=FAKE,
             max_pages=4, page_bits=6, w=None, eps=1e-6, freqs=None, max_pos=0, out_loc=None,
             n_out=10, pool=FAKE, pool_rows=1000, lat=None, pre=None, err=None, stream=None)
    a.update(kw)
    return L.dsv4kv_compress_store_ring(*a.values())


def test_ring_and_fused_gather_reject_bad_arguments(B):
    L = B.lib()
    assert _ring(L, ratio=1) == -1                  # the ring holds pairs: ratio 2 only
    assert _ring(L, ring_size=0) == -1
    assert _ring(L, ring=FAKE + 8) == -1            # misaligned ring
    assert _ring(L, ring=None, ring_size=3) == -1
    assert _ring(L, start=FAKE + 2) == -1           # misaligned start positions
    assert _ring(L, layout=5) == -1
    assert _ring(L, n_out=0) == 0
    g = L.dsv4kv_dequant_gather_topk
    assert g(1, FAKE, 10, FAKE, 4, 70000, FAKE, None, FAKE, 2, 2, 6, FAKE, None, None, None) == -3
    assert g(1, FAKE, 10, FAKE, 4, 8, FAKE, None, FAKE, 2, 2, 17, FAKE, None, None, None) == -1
    assert g(1, FAKE, 10, FAKE, 4, 8, None, None, FAKE, 2, 2, 6, FAKE, None, None, None) == -1
    assert g(1, FAKE, 10, FAKE, 4, 8, FAKE, None, FAKE, 2, 2, 6, FAKE + 8, None, None, None) == -1
    assert g(7, FAKE, 10, FAKE, 4, 8, FAKE, None, FAKE, 2, 2, 6, FAKE, None, None, None) == -1
    assert g(1, FAKE, 10, FAKE, 0, 8, FAKE, None, FAKE, 2, 2, 6, FAKE, None, None, None) == 0


def test_topk_reuse_head_covers_the_id_mapping(B):
    """The top-k form's head includes the mapping arguments: the same top-k
    buffer through another page table, token map, validity mask, page size or
    k is a miss.  n_tok = 0 rows, so nothing is launched."""
    L = B.lib()
    buf = B.dsv4kv_kvbuf()
    assert L.dsv4kv_kvbuf_init(ctypes.byref(buf), FAKE, 64) == 0
    rows, hit, lens = ctypes.c_void_p(), ctypes.c_int(), ctypes.c_int()
    base = [1, FAKE, 1000, FAKE + 256, 0, 8, FAKE + 512, None, FAKE + 1024, 4, 16, 6]

    def call(**kw):
        a = list(base)
        for i, v in kw.items():
            a[int(i[1:])] = v
        st = L.dsv4kv_kvbuf_get_with_head_topk(ctypes.byref(buf), *a, ctypes.byref(rows), None,
                                               ctypes.byref(hit), None, None)
        assert st == 0
        return hit.value

    assert call() == 0 and call() == 1                       # same source: hit
    assert call(a8=FAKE + 2048) == 0 and call(a8=FAKE + 2048) == 1   # other page table
    assert call(a6=FAKE + 4096) == 0                         # other token -> request map
    assert call(a7=FAKE + 8192) == 0                         # a validity mask
    assert call(a11=5) == 0                                  # other page size
    assert call(a5=7) == 0                                   # other k (n_tok * k still 0)
    L.dsv4kv_kvbuf_begin_forward(ctypes.byref(buf))
    assert call() == 0 and call() == 1
    # every field of the head alone: a change is a miss, the same again a hit
    for field, value in (("a0", 2), ("a1", FAKE + 64), ("a2", 999), ("a3", FAKE + 128),
                         ("a5", 4), ("a6", FAKE + 4096), ("a7", FAKE + 8192),
                         ("a8", FAKE + 2048), ("a9", 5), ("a10", 17), ("a11", 7)):
        assert call() in (0, 1)
        assert call() == 1
        assert call(**{field: value}) == 0, field
        assert call(**{field: value}) == 1, field
        assert call() == 0, field
    # the head is kept exactly as given (struct layout shared with C)
    call(a9=3, a10=12, a11=4)
    assert (buf.head_valid, buf.head_form, buf.head_layout, buf.head_k, buf.head_n_req,
            buf.head_max_pages, buf.head_page_bits) == (1, 1, 1, 8, 3, 12, 4)
    assert (buf.head_pool, buf.head_pool_rows, buf.head_ids, buf.head_token_to_req,
            buf.head_page_table, buf.head_is_valid) == (FAKE, 1000, FAKE + 256, FAKE + 512,
                                                        FAKE + 1024, None)


def test_short_context_calls_reject_bad_arguments(B):
    L = B.lib()
    f = L.dsv4kv_fill_all_compressed_indices
    assert f(FAKE, 4, 70000, FAKE, None) == -3
    assert f(FAKE, -1, 8, FAKE, None) == -1
    assert f(None, 4, 8, FAKE, None) == -1
    assert f(FAKE, 4, 8, FAKE + 2, None) == -1
    assert f(None, 0, 8, None, None) == 0                     # nothing to do
    g = L.dsv4kv_dequant_gather_all
    assert g(1, FAKE, 10, FAKE, 4, 70000, FAKE, None, FAKE, 2, 2, 6, FAKE, None, None, None) == -3
    assert g(1, FAKE, 10, None, 4, 8, FAKE, None, FAKE, 2, 2, 6, FAKE, None, None, None) == -1
    assert g(1, FAKE, 10, FAKE, 4, 8, FAKE, None, FAKE, 2, 2, 17, FAKE, None, None, None) == -1
    assert g(1, FAKE, 10, FAKE, 4, 8, FAKE, None, FAKE, 2, 2, 6, FAKE + 8, None, None, None) == -1
    assert g(9, FAKE, 10, FAKE, 4, 8, FAKE, None, FAKE, 2, 2, 6, FAKE, None, None, None) == -1
    assert g(1, FAKE, 10, FAKE, 0, 8, FAKE, None, FAKE, 2, 2, 6, FAKE, None, None, None) == 0
    # the reuse head of the short-context form is its own source
    buf = B.dsv4kv_kvbuf()
    assert L.dsv4kv_kvbuf_init(ctypes.byref(buf), FAKE, 64) == 0
    rows, hit = ctypes.c_void_p(), ctypes.c_int()
    args = (1, FAKE, 1000, FAKE + 256, 0, 8, FAKE + 512, None, FAKE + 1024, 4, 16, 6)
    for fn, want in ((L.dsv4kv_kvbuf_get_with_head_all, 0), (L.dsv4kv_kvbuf_get_with_head_all, 1),
                     (L.dsv4kv_kvbuf_get_with_head_topk, 0), (L.dsv4kv_kvbuf_get_with_head_all, 0)):
        assert fn(ctypes.byref(buf), *args, ctypes.byref(rows), None, ctypes.byref(hit), None,
                  None) == 0
        assert hit.value == want


def test_fake_quant_rejects_bad_arguments(B):
    L = B.lib()
    f = L.dsv4kv_fake_quant
    assert f(3, FAKE, 10, 512, FAKE, None) == -1            # layout
    assert f(1, FAKE, -1, 512, FAKE, None) == -1
    assert f(1, FAKE + 8, 10, 512, FAKE, None) == -1        # misaligned input
    assert f(1, FAKE, 10, 512, FAKE + 4, None) == -1        # misaligned output
    assert f(1, FAKE, 10, 500, FAKE, None) == -1            # stride below 512
    assert f(1, FAKE, 10, 516, FAKE, None) == -1            # stride not a multiple of 8
    assert f(1, None, 0, 512, None, None) == 0              # nothing to do


def test_selftests_reject_bad_arguments(B):
    """The self-test calls validate on the host like the others: no launch for
    a negative count or a null or misaligned pointer; n = 0 is a no-op."""
    L = B.lib()
    q = L.dsv4kv_selftest_fp4_quotient
    assert q(FAKE, FAKE, -1, FAKE, FAKE, None) == -1
    assert q(None, FAKE, 4, FAKE, FAKE, None) == -1
    assert q(FAKE + 2, FAKE, 4, FAKE, FAKE, None) == -1     # misaligned fp32 input
    assert q(None, None, 0, None, None, None) == 0
    r = L.dsv4kv_selftest_e4m3_recip
    assert r(FAKE, -1, FAKE, FAKE, None) == -1
    assert r(None, 4, FAKE, FAKE, None) == -1
    assert r(FAKE, 4, FAKE + 2, FAKE, None) == -1           # misaligned fp32 output
    assert r(FAKE, 4, FAKE, None, None) == -1
    assert r(None, 0, None, None, None) == 0
    w = L.dsv4kv_selftest_bounded_wait
    assert w(0, FAKE, FAKE, None) == -3                      # polls outside 1..2^24: ERANGE
    assert w(100, None, FAKE, None) == -1
