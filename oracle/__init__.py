"""CPU oracle for the DeepSeek-V4.1 compressed-KV write/read path.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py``, never by the product package.  It
shares no code with the CUDA library.  The arithmetic lives in
``dsv4kv_oracle.c`` (plain C, fp64); this module compiles it with gcc into
``oracle/_build/liboracle.so`` on first use and marshals numpy arrays.

Sources are cited in the C file: sglang PR #39652 "dsv4.1: compression, KV
I/O, and metadata kernels" (KVLayout, PagedKV::row, store_row, c1/c2,
dequantizers, the ue8m0 review), sglang PR #46230 (extend offsets, fused
| kv | score | projection), sglang PR #45909 (SparsePrefillKVBuffer reuse,
modelled in ``kvbuf_model.py``) and flashinfer_sparse.py
(_compressed_topk_to_slots).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

V4, V41, V41_FP4 = 0, 1, 2
D = 512

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dsv4kv_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (ISO C11, no FP contraction, no fast-math)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P, I, L, F, Dd = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64,
                          ctypes.c_float, ctypes.c_double)
        sig = {
            "orc_row_bytes": (I, [I]),
            "orc_e4m3_value": (Dd, [ctypes.c_uint]),
            "orc_e2m1_value": (Dd, [ctypes.c_uint]),
            "orc_e4m3_encode": (ctypes.c_uint, [Dd]),
            "orc_e2m1_encode": (ctypes.c_uint, [Dd]),
            "orc_ue8m0": (ctypes.c_uint, [F]),
            "orc_bf16_bits": (ctypes.c_uint16, [Dd]),
            "orc_quantize_row": (I, [I, P, P]),
            "orc_dequant_row": (I, [I, P, P]),
            "orc_row_offset": (L, [I, I, L]),
            "orc_plan": (L, [I, P, I, P, P, I, I, L, P, P, P, P, P, P]),
            "orc_compress_store": (L, [I, I, P, L, L, P, L, P, I, P, P, I, P, I, I, P, F,
                                       P, I, P, L, P, L, P, L, P, P, P, P, P]),
            "orc_dequant_gather": (L, [I, P, L, P, L, P]),
            "orc_topk_to_slots": (L, [P, L, I, P, P, P, I, I, I, P, P]),
            "orc_fill_all_indices": (None, [L, I, P, P]),
            "orc_ue8m0_many": (None, [P, L, P]),
            "orc_e4m3_encode_many": (None, [P, L, P]),
            "orc_e2m1_encode_many": (None, [P, L, P]),
            "orc_bf16_bits_many": (None, [P, L, P]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def _c(a, dtype):
    """Contiguous array of the given dtype (None passes through)."""
    if a is None:
        return None
    return np.ascontiguousarray(a, dtype=dtype)


# --------------------------------------------------------------------------
# scalar / vector primitives
# --------------------------------------------------------------------------
def row_bytes(layout: int) -> int:
    return _load().orc_row_bytes(layout)


def e4m3_value(code: int) -> float:
    return _load().orc_e4m3_value(code)


def e2m1_value(nib: int) -> float:
    return _load().orc_e2m1_value(nib)


def e4m3_encode(x) -> np.ndarray:
    x = _c(np.atleast_1d(x), np.float64)
    out = np.empty(x.shape, np.uint8)
    _load().orc_e4m3_encode_many(_ptr(x), x.size, _ptr(out))
    return out


def e2m1_encode(x) -> np.ndarray:
    x = _c(np.atleast_1d(x), np.float64)
    out = np.empty(x.shape, np.uint8)
    _load().orc_e2m1_encode_many(_ptr(x), x.size, _ptr(out))
    return out


def ue8m0(amax) -> np.ndarray:
    a = _c(np.atleast_1d(amax), np.float32)
    out = np.empty(a.shape, np.uint8)
    _load().orc_ue8m0_many(_ptr(a), a.size, _ptr(out))
    return out


def bf16_bits(x) -> np.ndarray:
    x = _c(np.atleast_1d(x), np.float64)
    out = np.empty(x.shape, np.uint16)
    _load().orc_bf16_bits_many(_ptr(x), x.size, _ptr(out))
    return out


def bf16_to_f64(bits) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    # a signaling-NaN pattern (arbitrary bytes) widens to a quiet NaN; some
    # hosts flag that conversion as an invalid operation, which is expected here
    with np.errstate(invalid="ignore"):
        return b.view(np.float32).astype(np.float64)


# --------------------------------------------------------------------------
# rows
# --------------------------------------------------------------------------
def quantize_rows(layout: int, x_f32: np.ndarray) -> np.ndarray:
    """fp32 [n, 512] -> uint8 [n, row_bytes] (store_row on each row)."""
    x = _c(x_f32, np.float32).reshape(-1, D)
    rb = row_bytes(layout)
    out = np.zeros((x.shape[0], rb), np.uint8)
    lib = _load()
    for i in range(x.shape[0]):
        rc = lib.orc_quantize_row(layout, x[i:].ctypes.data, out[i:].ctypes.data)
        if rc != 0:
            raise ValueError(f"orc_quantize_row: layout {layout} not supported")
    return out


def dequant_rows(layout: int, rows: np.ndarray) -> np.ndarray:
    """uint8 [n, row_bytes] -> fp64 [n, 512] (exact)."""
    r = _c(rows, np.uint8).reshape(-1, row_bytes(layout))
    out = np.zeros((r.shape[0], D), np.float64)
    lib = _load()
    for i in range(r.shape[0]):
        rc = lib.orc_dequant_row(layout, r[i:].ctypes.data, out[i:].ctypes.data)
        if rc != 0:
            raise ValueError(f"orc_dequant_row: layout {layout} not supported")
    return out


def row_offset(layout: int, page_bits: int, slot: int) -> int:
    return _load().orc_row_offset(layout, page_bits, slot)


def plan(ratio, ext, page_table=None, page_bits=0, start_pos=None):
    """Write plan: dict of per-output-row arrays (req, j, c, src, pos, slot);
    src = -1 marks a pair whose first token comes from the ring."""
    ext = _c(ext, np.int32)
    n_slots = ext.shape[-1]
    pt = _c(page_table, np.int32)
    sp = _c(start_pos, np.int32)
    max_pages = 0 if pt is None else pt.shape[-1]
    lib = _load()
    total = lib.orc_plan(ratio, _ptr(ext), n_slots, _ptr(sp), _ptr(pt), max_pages, page_bits,
                         0, None, None, None, None, None, None)
    req = np.zeros(total, np.int32)
    jj = np.zeros(total, np.int32)
    cc = np.zeros(total, np.int64)
    src = np.zeros(total, np.int64)
    pos = np.zeros(total, np.int64)
    slot = np.zeros(total, np.int64)
    lib.orc_plan(ratio, _ptr(ext), n_slots, _ptr(sp), _ptr(pt), max_pages, page_bits,
                 total, _ptr(req), _ptr(jj), _ptr(cc), _ptr(src), _ptr(pos), _ptr(slot))
    return dict(total=int(total), req=req, j=jj, c=cc, src=src, pos=pos, slot=slot)


def compress_store(layout, ratio, rows, ext, *, score=None, page_table=None,
                   page_bits=0, norm_w=None, eps=1e-6, freqs=None, out_loc=None,
                   n_out=None, pool=None, pool_rows=None, prequant_in=None,
                   want_f64=True, want_f32=True, want_latent=True, which=None,
                   start_pos=None, ring=None):
    """Run the fp64 compressor.  rows/score are bf16 bit arrays (uint16) with
    rows of width >= 512 (the fused | kv | score | layout when ratio == 2 and
    score is None).  start_pos (int32 [n_slots]) and ring (uint16 bf16 bits
    [n_slots, R, 1024], updated in place) follow orc_plan / the C header.
    pool (uint8, flat) is updated in place.  `which` (int64
    output-row indices) restricts the work to those rows; per-row outputs and
    prequant_in are then indexed by position in `which`.  Returns a dict
    with total, faults and the requested per-row outputs."""
    rows = _c(rows, np.uint16)
    n_rows, row_stride = rows.shape
    score = _c(score, np.uint16)
    score_stride = 0 if score is None else score.shape[1]
    ext = _c(ext, np.int32)
    n_slots = ext.shape[-1]
    pt = _c(page_table, np.int32)
    max_pages = 0 if pt is None else pt.shape[-1]
    norm_w = _c(norm_w, np.uint16)
    freqs = _c(freqs, np.float32)
    max_pos = 0 if freqs is None else freqs.shape[0]
    out_loc = _c(out_loc, np.int32)
    sp = _c(start_pos, np.int32)
    if ring is not None:
        assert ring.dtype == np.uint16 and ring.flags.c_contiguous and ring.ndim == 3
    ring_size = 0 if ring is None else ring.shape[1]
    if n_out is None:
        n_out = out_loc.shape[0] if out_loc is not None else \
            plan(ratio, ext, pt, page_bits, start_pos=sp)["total"]
    if pool is not None:
        assert pool.dtype == np.uint8 and pool.flags.c_contiguous
        if pool_rows is None:
            pool_rows = pool.size // row_bytes(layout)
    pre_in = _c(prequant_in, np.float32)
    which = _c(which, np.int64)
    n_rows_out = n_out if which is None else which.size
    f64 = np.zeros((n_rows_out, D), np.float64) if want_f64 else None
    f32 = np.zeros((n_rows_out, D), np.float32) if want_f32 else None
    lat = np.zeros((n_rows_out, D), np.uint16) if want_latent else None
    faults = ctypes.c_int64(0)
    total = _load().orc_compress_store(
        layout, ratio, _ptr(rows), n_rows, row_stride, _ptr(score), score_stride,
        _ptr(ext), n_slots, _ptr(sp), _ptr(ring), ring_size, _ptr(pt), max_pages, page_bits,
        _ptr(norm_w), eps,
        _ptr(freqs), max_pos, _ptr(out_loc), n_out, _ptr(which),
        0 if which is None else which.size, _ptr(pool),
        0 if pool_rows is None else pool_rows, _ptr(pre_in), _ptr(f64), _ptr(f32),
        _ptr(lat), ctypes.addressof(faults))
    if total < 0:
        raise ValueError(f"orc_compress_store rejected its arguments ({total})")
    return dict(total=int(total), faults=int(faults.value), prequant_f64=f64,
                prequant_f32=f32, latent=lat)


def dequant_gather(layout, pool, pool_rows, ids):
    """bf16 bits [n, 512] of the gathered rows; returns (out, faults)."""
    ids = _c(ids, np.int32)
    out = np.zeros((ids.size, D), np.uint16)
    pool = _c(pool, np.uint8)
    faults = _load().orc_dequant_gather(layout, _ptr(pool), pool_rows, _ptr(ids),
                                        ids.size, _ptr(out))
    if faults < 0:
        raise ValueError("orc_dequant_gather: layout not supported")
    return out, int(faults)


def fill_all_indices(lens, k):
    """Short-context ids: int32 [n_tok, k], row t = 0..lens[t]-1 then -1."""
    lens = _c(lens, np.int32)
    out = np.zeros((lens.size, k), np.int32)
    _load().orc_fill_all_indices(lens.size, k, _ptr(lens), _ptr(out))
    return out


def topk_to_slots(topk, token_to_req, page_table, page_bits, is_valid=None):
    topk = _c(topk, np.int32)
    n_tok, k = topk.shape
    ttr = _c(token_to_req, np.int32)
    pt = _c(page_table, np.int32)
    n_req, max_pages = pt.shape
    iv = _c(is_valid, np.uint8)
    slots = np.zeros((n_tok, k), np.int32)
    lens = np.zeros(n_tok, np.int32)
    faults = _load().orc_topk_to_slots(_ptr(topk), n_tok, k, _ptr(ttr), _ptr(iv),
                                       _ptr(pt), n_req, max_pages, page_bits,
                                       _ptr(slots), _ptr(lens))
    return slots, lens, int(faults)
