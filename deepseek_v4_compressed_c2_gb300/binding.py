"""Thin Python binding of the dsv4kv C ABI (include/dsv4kv.h).

Argument marshalling only: every step of the compressed-KV write and read
runs in the CUDA library ``_build/libdsv4kv.so``.  PyTorch provides device
memory and the current stream.  The library must have been built
(``__graft_entry__.build()`` or ``python -m deepseek_v4_compressed_c2_gb300.build``);
there is no fallback -- if it is missing, every call raises.

Function names are the C names.  Shapes, dtypes and the error convention are
documented in the header; a negative status raises ``DSV4KVError``.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from .build import LIB as _LIB_PATH

V4, V41, V41_FP4 = 0, 1, 2
DIM = 512
_ROW_BYTES = {V4: 584, V41: 528, V41_FP4: 288}

_lock = threading.Lock()
_lib = None


class DSV4KVError(RuntimeError):
    def __init__(self, fn, status, lib):
        msg = lib.dsv4kv_status_string(status).decode()
        if status == -4:
            msg += f" (cudaError {lib.dsv4kv_last_cuda_error()})"
        super().__init__(f"{fn}: status {status}: {msg}")
        self.status = status


class dsv4kv_kvbuf(ctypes.Structure):
    _fields_ = [("storage", ctypes.c_void_p), ("capacity_rows", ctypes.c_longlong),
                ("head_valid", ctypes.c_int), ("head_layout", ctypes.c_int),
                ("head_pool", ctypes.c_void_p), ("head_pool_rows", ctypes.c_longlong),
                ("head_ids", ctypes.c_void_p), ("head_n", ctypes.c_longlong),
                ("head_form", ctypes.c_int), ("head_k", ctypes.c_int),
                ("head_token_to_req", ctypes.c_void_p), ("head_is_valid", ctypes.c_void_p),
                ("head_page_table", ctypes.c_void_p), ("head_n_req", ctypes.c_int),
                ("head_max_pages", ctypes.c_int), ("head_page_bits", ctypes.c_int)]


def lib():
    """The loaded CUDA library; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"dsv4kv CUDA library not built ({_LIB_PATH} missing); "
                               "run __graft_entry__.build() first")
        L = ctypes.CDLL(_LIB_PATH)
        P, I, LL, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_longlong, ctypes.c_float
        KB = ctypes.POINTER(dsv4kv_kvbuf)
        sig = {
            "dsv4kv_row_bytes": (I, [I]),
            "dsv4kv_last_cuda_error": (I, []),
            "dsv4kv_status_string": (ctypes.c_char_p, [I]),
            "dsv4kv_compress_store": (I, [I, I, P, LL, LL, P, LL, P, I, P, I, I, P, F, P, I,
                                          P, I, P, LL, P, P, P, P]),
            "dsv4kv_compress_store_ring": (I, [I, I, P, LL, LL, P, LL, P, I, P, P, I, P, I, I, P,
                                               F, P, I, P, I, P, LL, P, P, P, P]),
            "dsv4kv_dequant_gather": (I, [I, P, LL, P, LL, P, P, P]),
            "dsv4kv_topk_to_slots": (I, [P, I, I, P, P, P, I, I, I, P, P, P, P]),
            "dsv4kv_dequant_gather_topk": (I, [I, P, LL, P, I, I, P, P, P, I, I, I, P, P, P, P]),
            "dsv4kv_kvbuf_get_with_head_topk": (I, [KB, I, P, LL, P, I, I, P, P, P, I, I, I,
                                                    ctypes.POINTER(ctypes.c_void_p), P,
                                                    ctypes.POINTER(ctypes.c_int), P, P]),
            "dsv4kv_kvbuf_get_with_head_all": (I, [KB, I, P, LL, P, I, I, P, P, P, I, I, I,
                                                   ctypes.POINTER(ctypes.c_void_p), P,
                                                   ctypes.POINTER(ctypes.c_int), P, P]),
            "dsv4kv_fill_all_compressed_indices": (I, [P, I, I, P, P]),
            "dsv4kv_fake_quant": (I, [I, P, LL, LL, P, P]),
            "dsv4kv_dequant_gather_all": (I, [I, P, LL, P, I, I, P, P, P, I, I, I, P, P, P, P]),
            "dsv4kv_selftest_bounded_wait": (I, [I, P, P, P]),
            "dsv4kv_selftest_fp4_quotient": (I, [P, P, LL, P, P, P]),
            "dsv4kv_selftest_e4m3_recip": (I, [P, LL, P, P, P]),
            "dsv4kv_kvbuf_init": (I, [KB, P, LL]),
            "dsv4kv_kvbuf_begin_forward": (None, [KB]),
            "dsv4kv_kvbuf_get": (I, [KB, LL, ctypes.POINTER(ctypes.c_void_p)]),
            "dsv4kv_kvbuf_lookup": (I, [KB, I, P, LL, P, LL, ctypes.POINTER(ctypes.c_int)]),
            "dsv4kv_kvbuf_get_with_head": (I, [KB, I, P, LL, P, LL, ctypes.POINTER(ctypes.c_void_p),
                                               ctypes.POINTER(ctypes.c_int), P, P]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
        return L


def _check(fn, status):
    if status != 0:
        raise DSV4KVError(fn, status, lib())


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _need(t, dtype, name):
    if t is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")


def _pool_rows(pool, layout, pool_rows):
    """Rows of the layout the pool tensor holds, or a checked explicit count."""
    pool_bytes = pool.numel() * pool.element_size()
    if pool_rows is None:
        return pool_bytes // _ROW_BYTES.get(layout, 1)
    if pool_rows * _ROW_BYTES.get(layout, 0) > pool_bytes:
        raise ValueError("pool_rows exceeds the pool tensor")
    return pool_rows


def dsv4kv_row_bytes(layout: int) -> int:
    rb = lib().dsv4kv_row_bytes(layout)
    _check("dsv4kv_row_bytes", rb if rb < 0 else 0)
    return rb


def dsv4kv_compress_store(layout, ratio, rows, extend_offsets, pool, *, score=None,
                          page_table=None, page_bits=0, rmsnorm_w=None, eps=1e-6,
                          freqs_cis=None, out_loc=None, n_out=None, pool_rows=None,
                          latent_out=None, prequant_out=None, err_word=None, stream=None,
                          start_pos=None, ring=None):
    """Fused compress -> RMSNorm -> RoPE -> quantize -> paged store.
    rows: bf16 [n_rows, row_stride] (unit column stride); extend_offsets: int32
    [2, n_slots]; pool: uint8 tensor of pool_rows * row_bytes bytes.  With
    start_pos (int32 [n_slots]) and/or ring (bf16 [n_slots, R, 1024]) this is
    dsv4kv_compress_store_ring."""
    _need(start_pos, torch.int32, "start_pos")
    _need(ring, torch.bfloat16, "ring")
    if start_pos is not None and start_pos.numel() < extend_offsets.shape[1]:
        raise ValueError("start_pos must hold n_slots positions")
    if ring is not None and (ring.dim() != 3 or ring.shape[2] != 2 * DIM or not ring.is_contiguous()
                             or ring.shape[0] < extend_offsets.shape[1]):
        raise ValueError("ring must be a contiguous [>= n_slots, R, 1024] tensor")
    _need(rows, torch.bfloat16, "rows")
    _need(score, torch.bfloat16, "score")
    _need(extend_offsets, torch.int32, "extend_offsets")
    _need(page_table, torch.int32, "page_table")
    _need(rmsnorm_w, torch.bfloat16, "rmsnorm_w")
    _need(freqs_cis, torch.float32, "freqs_cis")
    _need(out_loc, torch.int32, "out_loc")
    _need(latent_out, torch.bfloat16, "latent_out")
    _need(prequant_out, torch.float32, "prequant_out")
    _need(err_word, torch.int32, "err_word")
    if rows.dim() != 2 or rows.stride(1) != 1:
        raise ValueError("rows must be 2-D with unit column stride")
    if extend_offsets.dim() != 2 or extend_offsets.shape[0] != 2 or not extend_offsets.is_contiguous():
        raise ValueError("extend_offsets must be a contiguous [2, n_slots] tensor")
    if n_out is None:
        if out_loc is None:
            raise ValueError("n_out is required when out_loc is None")
        n_out = out_loc.numel()
    pool_rows = _pool_rows(pool, layout, pool_rows)
    if out_loc is not None and out_loc.numel() < n_out:
        raise ValueError("out_loc has fewer than n_out entries")
    for name, t in (("latent_out", latent_out), ("prequant_out", prequant_out)):
        if t is not None and (t.numel() < n_out * DIM or not t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous tensor of >= n_out x 512")
    if score is not None and (score.dim() != 2 or score.stride(1) != 1
                              or score.shape[0] < rows.shape[0]):
        raise ValueError("score must be 2-D, unit column stride, with >= n_rows rows")
    if rows.shape[1] < (2 * DIM if ratio == 2 and score is None else DIM):
        raise ValueError("rows are narrower than the layout needs")
    if rmsnorm_w is not None and rmsnorm_w.numel() < DIM:
        raise ValueError("rmsnorm_w must hold 512 weights")
    if freqs_cis is not None and (freqs_cis.dim() != 2 or freqs_cis.shape[1] != 64
                                  or not freqs_cis.is_contiguous()):
        raise ValueError("freqs_cis must be a contiguous [max_pos, 64] tensor")
    if page_table is not None and (page_table.dim() != 2 or not page_table.is_contiguous()
                                   or page_table.shape[0] < extend_offsets.shape[1]):
        raise ValueError("page_table must be a contiguous [>= n_slots, max_pages] tensor")
    s_stride = 0 if score is None else score.stride(0)
    st = lib().dsv4kv_compress_store_ring(
        layout, ratio, _ptr(rows), rows.shape[0], rows.stride(0), _ptr(score), s_stride,
        _ptr(extend_offsets), extend_offsets.shape[1], _ptr(start_pos), _ptr(ring),
        0 if ring is None else ring.shape[1], _ptr(page_table),
        0 if page_table is None else page_table.shape[1], page_bits, _ptr(rmsnorm_w), eps,
        _ptr(freqs_cis), 0 if freqs_cis is None else freqs_cis.shape[0], _ptr(out_loc), n_out,
        _ptr(pool), pool_rows, _ptr(latent_out), _ptr(prequant_out), _ptr(err_word),
        _stream(stream))
    _check("dsv4kv_compress_store_ring" if (start_pos is not None or ring is not None)
           else "dsv4kv_compress_store", st)


def dsv4kv_dequant_gather(layout, pool, ids, out=None, *, pool_rows=None, err_word=None,
                          stream=None):
    """bf16 [n, 512] rows of the pool at `ids` (int32); returns `out`."""
    _need(ids, torch.int32, "ids")
    _need(out, torch.bfloat16, "out")
    _need(err_word, torch.int32, "err_word")
    n = ids.numel()
    if not ids.is_contiguous():
        raise ValueError("ids must be contiguous")
    if out is None:
        out = torch.empty((n, DIM), dtype=torch.bfloat16, device=ids.device)
    elif out.numel() < n * DIM or not out.is_contiguous():
        raise ValueError("out must be a contiguous tensor of >= n x 512")
    pool_rows = _pool_rows(pool, layout, pool_rows)
    st = lib().dsv4kv_dequant_gather(layout, _ptr(pool), pool_rows, _ptr(ids), n, _ptr(out),
                                     _ptr(err_word), _stream(stream))
    _check("dsv4kv_dequant_gather", st)
    return out


def dsv4kv_topk_to_slots(topk, token_to_req, page_table, page_bits, *, is_valid=None,
                         slots=None, lens=None, err_word=None, stream=None):
    """Request-local top-k ids -> pool slots (int32 [n_tok, k]) and lens."""
    n_tok, k = _topk_args(topk, token_to_req, page_table, is_valid)
    if slots is None:
        slots = torch.empty((n_tok, k), dtype=torch.int32, device=topk.device)
    if lens is None:
        lens = torch.empty((n_tok,), dtype=torch.int32, device=topk.device)
    st = lib().dsv4kv_topk_to_slots(_ptr(topk), n_tok, k, _ptr(token_to_req), _ptr(is_valid),
                                    _ptr(page_table), page_table.shape[0], page_table.shape[1],
                                    page_bits, _ptr(slots), _ptr(lens), _ptr(err_word),
                                    _stream(stream))
    _check("dsv4kv_topk_to_slots", st)
    return slots, lens


def _topk_args(topk, token_to_req, page_table, is_valid):
    _need(topk, torch.int32, "topk")
    _need(token_to_req, torch.int32, "token_to_req")
    _need(page_table, torch.int32, "page_table")
    _need(is_valid, torch.uint8, "is_valid")
    n_tok, k = topk.shape
    if not (topk.is_contiguous() and page_table.is_contiguous()) or token_to_req.numel() < n_tok \
            or (is_valid is not None and is_valid.numel() < n_tok):
        raise ValueError("topk / page_table must be contiguous; token_to_req, is_valid >= n_tok")
    return n_tok, k


def dsv4kv_dequant_gather_topk(layout, pool, topk, token_to_req, page_table, page_bits, out=None,
                               *, is_valid=None, lens=None, pool_rows=None, err_word=None,
                               stream=None):
    """Fused top-k -> slot -> gather-dequant; returns out [n_tok * k, 512]."""
    n_tok, k = _topk_args(topk, token_to_req, page_table, is_valid)
    _need(out, torch.bfloat16, "out")
    _need(lens, torch.int32, "lens")
    _need(err_word, torch.int32, "err_word")
    n = n_tok * k
    if out is None:
        out = torch.empty((n, DIM), dtype=torch.bfloat16, device=topk.device)
    elif out.numel() < n * DIM or not out.is_contiguous():
        raise ValueError("out must be a contiguous tensor of >= n_tok * k x 512")
    if lens is not None and lens.numel() < n_tok:
        raise ValueError("lens must hold n_tok counts")
    pool_rows = _pool_rows(pool, layout, pool_rows)
    st = lib().dsv4kv_dequant_gather_topk(layout, _ptr(pool), pool_rows, _ptr(topk), n_tok, k,
                                          _ptr(token_to_req), _ptr(is_valid), _ptr(page_table),
                                          page_table.shape[0], page_table.shape[1], page_bits,
                                          _ptr(out), _ptr(lens), _ptr(err_word), _stream(stream))
    _check("dsv4kv_dequant_gather_topk", st)
    return out


def dsv4kv_fill_all_compressed_indices(lens_in, k, out=None, *, stream=None):
    """Short-context ids: int32 [n_tok, k], row t = 0 .. lens_in[t]-1 then -1."""
    _need(lens_in, torch.int32, "lens_in")
    _need(out, torch.int32, "out")
    n_tok = lens_in.numel()
    if not lens_in.is_contiguous():
        raise ValueError("lens_in must be contiguous")
    if out is None:
        out = torch.empty((n_tok, k), dtype=torch.int32, device=lens_in.device)
    elif out.numel() < n_tok * k or not out.is_contiguous():
        raise ValueError("out must be a contiguous tensor of >= n_tok x k")
    st = lib().dsv4kv_fill_all_compressed_indices(_ptr(out), n_tok, k, _ptr(lens_in),
                                                  _stream(stream))
    _check("dsv4kv_fill_all_compressed_indices", st)
    return out


def dsv4kv_fake_quant(layout, x, out=None, *, stream=None):
    """bf16 [n, >=512] rows -> bf16 [n, 512]: quantized with the layout's
    store_row and dequantized (out may be x when x is [n, 512])."""
    _need(x, torch.bfloat16, "x")
    _need(out, torch.bfloat16, "out")
    if x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be 2-D with unit column stride")
    n = x.shape[0]
    if out is None:
        out = torch.empty((n, DIM), dtype=torch.bfloat16, device=x.device)
    elif out.numel() < n * DIM or not out.is_contiguous():
        raise ValueError("out must be a contiguous tensor of >= n x 512")
    st = lib().dsv4kv_fake_quant(layout, _ptr(x), n, x.stride(0), _ptr(out), _stream(stream))
    _check("dsv4kv_fake_quant", st)
    return out


def _all_args(lens_in, token_to_req, page_table, is_valid):
    _need(lens_in, torch.int32, "lens_in")
    _need(token_to_req, torch.int32, "token_to_req")
    _need(page_table, torch.int32, "page_table")
    _need(is_valid, torch.uint8, "is_valid")
    n_tok = lens_in.numel()
    if not (lens_in.is_contiguous() and page_table.is_contiguous()) \
            or token_to_req.numel() < n_tok or (is_valid is not None and is_valid.numel() < n_tok):
        raise ValueError("lens_in / page_table must be contiguous; token_to_req, is_valid >= n_tok")
    return n_tok


def dsv4kv_dequant_gather_all(layout, pool, lens_in, k, token_to_req, page_table, page_bits,
                              out=None, *, is_valid=None, lens=None, pool_rows=None,
                              err_word=None, stream=None):
    """Fused short-context gather: row t*k + j = compressed row j of token t's
    request when j < lens_in[t], else zeros; returns out [n_tok * k, 512]."""
    n_tok = _all_args(lens_in, token_to_req, page_table, is_valid)
    _need(out, torch.bfloat16, "out")
    _need(lens, torch.int32, "lens")
    _need(err_word, torch.int32, "err_word")
    n = n_tok * k
    if out is None:
        out = torch.empty((n, DIM), dtype=torch.bfloat16, device=lens_in.device)
    elif out.numel() < n * DIM or not out.is_contiguous():
        raise ValueError("out must be a contiguous tensor of >= n_tok * k x 512")
    if lens is not None and lens.numel() < n_tok:
        raise ValueError("lens must hold n_tok counts")
    pool_rows = _pool_rows(pool, layout, pool_rows)
    st = lib().dsv4kv_dequant_gather_all(layout, _ptr(pool), pool_rows, _ptr(lens_in), n_tok, k,
                                         _ptr(token_to_req), _ptr(is_valid), _ptr(page_table),
                                         page_table.shape[0], page_table.shape[1], page_bits,
                                         _ptr(out), _ptr(lens), _ptr(err_word), _stream(stream))
    _check("dsv4kv_dequant_gather_all", st)
    return out


class SparsePrefillKVBuffer:
    """The shared bf16 buffer sparse-prefill layers read, with the reuse head
    (sglang PR #45909).  Wraps a caller-owned dsv4kv_kvbuf struct and a
    storage tensor of capacity_rows x 512 bf16."""

    def __init__(self, storage: torch.Tensor):
        _need(storage, torch.bfloat16, "storage")
        self.buf = dsv4kv_kvbuf()
        self.dequants = 0
        self.dsv4kv_kvbuf_init(storage)

    def dsv4kv_kvbuf_init(self, storage: torch.Tensor):
        """(Re)allocation: new storage, head forgotten."""
        self.storage = storage
        _check("dsv4kv_kvbuf_init",
               lib().dsv4kv_kvbuf_init(ctypes.byref(self.buf), _ptr(storage), storage.shape[0]))

    def dsv4kv_kvbuf_begin_forward(self):
        lib().dsv4kv_kvbuf_begin_forward(ctypes.byref(self.buf))

    def dsv4kv_kvbuf_get(self, n: int) -> torch.Tensor:
        p = ctypes.c_void_p()
        _check("dsv4kv_kvbuf_get", lib().dsv4kv_kvbuf_get(ctypes.byref(self.buf), n, ctypes.byref(p)))
        return self.storage[:n]

    def dsv4kv_kvbuf_lookup(self, layout, pool, pool_rows, ids, n) -> bool:
        hit = ctypes.c_int(0)
        _check("dsv4kv_kvbuf_lookup",
               lib().dsv4kv_kvbuf_lookup(ctypes.byref(self.buf), layout, _ptr(pool), pool_rows,
                                         _ptr(ids), n, ctypes.byref(hit)))
        return bool(hit.value)

    def dsv4kv_kvbuf_get_with_head(self, layout, pool, ids, *, pool_rows=None, err_word=None,
                                   stream=None):
        """(rows, hit): on a miss the gather-dequant fills the storage."""
        n = ids.numel()
        pool_rows = _pool_rows(pool, layout, pool_rows)
        if not ids.is_contiguous():
            raise ValueError("ids must be contiguous")
        p = ctypes.c_void_p()
        hit = ctypes.c_int(0)
        st = lib().dsv4kv_kvbuf_get_with_head(ctypes.byref(self.buf), layout, _ptr(pool),
                                              pool_rows, _ptr(ids), n, ctypes.byref(p),
                                              ctypes.byref(hit), _ptr(err_word), _stream(stream))
        _check("dsv4kv_kvbuf_get_with_head", st)
        if not hit.value and n > 0:
            self.dequants += 1
        return self.storage[:n], bool(hit.value)

    def dsv4kv_kvbuf_get_with_head_topk(self, layout, pool, topk, token_to_req, page_table,
                                        page_bits, *, is_valid=None, lens=None, pool_rows=None,
                                        err_word=None, stream=None):
        """(rows, hit) with request-local top-k ids as the gather ids; on a
        miss the fused top-k gather-dequant fills the storage."""
        n_tok, k = _topk_args(topk, token_to_req, page_table, is_valid)
        pool_rows = _pool_rows(pool, layout, pool_rows)
        p = ctypes.c_void_p()
        hit = ctypes.c_int(0)
        st = lib().dsv4kv_kvbuf_get_with_head_topk(
            ctypes.byref(self.buf), layout, _ptr(pool), pool_rows, _ptr(topk), n_tok, k,
            _ptr(token_to_req), _ptr(is_valid), _ptr(page_table), page_table.shape[0],
            page_table.shape[1], page_bits, ctypes.byref(p), _ptr(lens), ctypes.byref(hit),
            _ptr(err_word), _stream(stream))
        _check("dsv4kv_kvbuf_get_with_head_topk", st)
        if not hit.value and n_tok * k > 0:
            self.dequants += 1
        return self.storage[:n_tok * k], bool(hit.value)

    def dsv4kv_kvbuf_get_with_head_all(self, layout, pool, lens_in, k, token_to_req, page_table,
                                       page_bits, *, is_valid=None, lens=None, pool_rows=None,
                                       err_word=None, stream=None):
        """(rows, hit) with the short-context ids (dsv4kv_dequant_gather_all)."""
        n_tok = _all_args(lens_in, token_to_req, page_table, is_valid)
        pool_rows = _pool_rows(pool, layout, pool_rows)
        p = ctypes.c_void_p()
        hit = ctypes.c_int(0)
        st = lib().dsv4kv_kvbuf_get_with_head_all(
            ctypes.byref(self.buf), layout, _ptr(pool), pool_rows, _ptr(lens_in), n_tok, k,
            _ptr(token_to_req), _ptr(is_valid), _ptr(page_table), page_table.shape[0],
            page_table.shape[1], page_bits, ctypes.byref(p), _ptr(lens), ctypes.byref(hit),
            _ptr(err_word), _stream(stream))
        _check("dsv4kv_kvbuf_get_with_head_all", st)
        if not hit.value and n_tok * k > 0:
            self.dequants += 1
        return self.storage[:n_tok * k], bool(hit.value)


class PreparedCall:
    """A C-ABI call whose arguments were marshalled once (tensor pointers,
    sizes, stream); calling it issues the launch again with the same
    arguments.  For loops that relaunch the same step (a prefill loop without
    a CUDA graph): per call the host cost is one ctypes call, and the C side
    still checks every argument."""

    def __init__(self, name, args, keep):
        self._fn = getattr(lib(), name)
        self._name = name
        self._args = args
        self._keep = keep            # tensors whose pointers are baked in

    def __call__(self):
        st = self._fn(*self._args)
        if st != 0:
            raise DSV4KVError(self._name, st, lib())


def prepare_compress_store(layout, ratio, rows, extend_offsets, pool, *, score=None,
                           page_table=None, page_bits=0, rmsnorm_w=None, eps=1e-6,
                           freqs_cis=None, out_loc=None, n_out=None, pool_rows=None,
                           latent_out=None, prequant_out=None, err_word=None, stream=None,
                           start_pos=None, ring=None):
    """dsv4kv_compress_store (or, with start_pos / ring, the _ring entry) with
    its arguments marshalled once.  The checked first call below runs the
    launch once (a ring step advances the ring)."""
    if n_out is None:
        n_out = out_loc.numel()
    if pool_rows is None:
        pool_rows = pool.numel() * pool.element_size() // _ROW_BYTES.get(layout, 1)
    head = (layout, ratio, _ptr(rows), rows.shape[0], rows.stride(0), _ptr(score),
            0 if score is None else score.stride(0), _ptr(extend_offsets),
            extend_offsets.shape[1])
    tail = (_ptr(page_table), 0 if page_table is None else page_table.shape[1], page_bits,
            _ptr(rmsnorm_w), eps, _ptr(freqs_cis), 0 if freqs_cis is None else freqs_cis.shape[0],
            _ptr(out_loc), n_out, _ptr(pool), pool_rows, _ptr(latent_out), _ptr(prequant_out),
            _ptr(err_word), _stream(stream))
    use_ring = start_pos is not None or ring is not None
    if use_ring:
        name = "dsv4kv_compress_store_ring"
        args = head + (_ptr(start_pos), _ptr(ring), 0 if ring is None else ring.shape[1]) + tail
    else:
        name, args = "dsv4kv_compress_store", head + tail
    # one checked call validates shapes through the same path as the plain binding
    dsv4kv_compress_store(layout, ratio, rows, extend_offsets, pool, score=score,
                          page_table=page_table, page_bits=page_bits, rmsnorm_w=rmsnorm_w,
                          eps=eps, freqs_cis=freqs_cis, out_loc=out_loc, n_out=n_out,
                          pool_rows=pool_rows, latent_out=latent_out, prequant_out=prequant_out,
                          err_word=err_word, stream=stream, start_pos=start_pos, ring=ring)
    return PreparedCall(name, args,
                        (rows, extend_offsets, pool, score, page_table, rmsnorm_w, freqs_cis,
                         out_loc, latent_out, prequant_out, err_word, start_pos, ring))


def prepare_topk_to_slots(topk, token_to_req, page_table, page_bits, slots, lens, *,
                          is_valid=None, err_word=None, stream=None):
    dsv4kv_topk_to_slots(topk, token_to_req, page_table, page_bits, is_valid=is_valid,
                         slots=slots, lens=lens, err_word=err_word, stream=stream)
    n_tok, k = topk.shape
    args = (_ptr(topk), n_tok, k, _ptr(token_to_req), _ptr(is_valid), _ptr(page_table),
            page_table.shape[0], page_table.shape[1], page_bits, _ptr(slots), _ptr(lens),
            _ptr(err_word), _stream(stream))
    return PreparedCall("dsv4kv_topk_to_slots", args,
                        (topk, token_to_req, page_table, slots, lens, is_valid, err_word))


def prepare_dequant_gather(layout, pool, ids, out, *, pool_rows=None, err_word=None, stream=None):
    dsv4kv_dequant_gather(layout, pool, ids, out, pool_rows=pool_rows, err_word=err_word,
                          stream=stream)
    if pool_rows is None:
        pool_rows = pool.numel() * pool.element_size() // _ROW_BYTES.get(layout, 1)
    args = (layout, _ptr(pool), pool_rows, _ptr(ids), ids.numel(), _ptr(out), _ptr(err_word),
            _stream(stream))
    return PreparedCall("dsv4kv_dequant_gather", args, (pool, ids, out, err_word))


def prepare_dequant_gather_topk(layout, pool, topk, token_to_req, page_table, page_bits, out, *,
                                is_valid=None, pool_rows=None, err_word=None, stream=None):
    """dsv4kv_dequant_gather_topk with its arguments marshalled once."""
    dsv4kv_dequant_gather_topk(layout, pool, topk, token_to_req, page_table, page_bits, out,
                               is_valid=is_valid, pool_rows=pool_rows, err_word=err_word,
                               stream=stream)
    n_tok, k = topk.shape
    if pool_rows is None:
        pool_rows = pool.numel() * pool.element_size() // _ROW_BYTES.get(layout, 1)
    args = (layout, _ptr(pool), pool_rows, _ptr(topk), n_tok, k, _ptr(token_to_req),
            _ptr(is_valid), _ptr(page_table), page_table.shape[0], page_table.shape[1], page_bits,
            _ptr(out), None, _ptr(err_word), _stream(stream))
    return PreparedCall("dsv4kv_dequant_gather_topk", args,
                        (pool, topk, token_to_req, page_table, is_valid, out, err_word))


def prepare_get_with_head_topk(kvbuf, layout, pool, topk, token_to_req, page_table, page_bits, *,
                               is_valid=None, pool_rows=None, err_word=None, stream=None):
    """SparsePrefillKVBuffer.get_with_head_topk with its arguments marshalled
    once; the returned callable gives the hit flag."""
    n_tok, k = _topk_args(topk, token_to_req, page_table, is_valid)
    if pool_rows is None:
        pool_rows = pool.numel() * pool.element_size() // _ROW_BYTES.get(layout, 1)
    hit = ctypes.c_int(0)
    rows = ctypes.c_void_p()
    fn = lib().dsv4kv_kvbuf_get_with_head_topk
    args = (ctypes.byref(kvbuf.buf), layout, _ptr(pool), pool_rows, _ptr(topk), n_tok, k,
            _ptr(token_to_req), _ptr(is_valid), _ptr(page_table), page_table.shape[0],
            page_table.shape[1], page_bits, ctypes.byref(rows), None, ctypes.byref(hit),
            _ptr(err_word), _stream(stream))
    keep = (pool, topk, token_to_req, page_table, is_valid, err_word, kvbuf)

    def call():
        st = fn(*args)
        if st != 0:
            raise DSV4KVError("dsv4kv_kvbuf_get_with_head_topk", st, lib())
        if not hit.value and n_tok * k > 0:
            kvbuf.dequants += 1
        return bool(hit.value)
    call.keep = keep
    return call


def prepare_get_with_head(kvbuf, layout, pool, ids, *, pool_rows=None, err_word=None,
                          stream=None):
    """SparsePrefillKVBuffer.get_with_head with its arguments marshalled once;
    the returned callable gives the hit flag."""
    if pool_rows is None:
        pool_rows = pool.numel() * pool.element_size() // _ROW_BYTES.get(layout, 1)
    hit = ctypes.c_int(0)
    rows = ctypes.c_void_p()
    fn = lib().dsv4kv_kvbuf_get_with_head
    args = (ctypes.byref(kvbuf.buf), layout, _ptr(pool), pool_rows, _ptr(ids), ids.numel(),
            ctypes.byref(rows), ctypes.byref(hit), _ptr(err_word), _stream(stream))
    keep = (pool, ids, err_word, kvbuf)

    def call():
        st = fn(*args)
        if st != 0:
            raise DSV4KVError("dsv4kv_kvbuf_get_with_head", st, lib())
        if not hit.value and ids.numel() > 0:
            kvbuf.dequants += 1
        return bool(hit.value)
    call.keep = keep
    return call
