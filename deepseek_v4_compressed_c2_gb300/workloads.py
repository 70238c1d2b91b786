"""Seeded synthetic inputs for the compressed-KV write/read path.

This module is the one thing the CUDA path and the CPU oracle share: it builds
input arrays (numpy, host memory) and holds none of the method's arithmetic --
no pooling, normalisation, rotation, quantization, plan or slot computation.
Each workload mirrors the shapes, value distributions and ragged structure of
the DeepSeek-V4.1 prefill / decode cases the sglang pages describe (512-dim
bf16 latents, ragged extend lengths, random permuted page tables, a padded
output-row count for the prefill CUDA graph, a top-k id list per request).

Generators: numpy ``default_rng(seed)`` (PCG64); bf16 values are float32
samples rounded to nearest even.  The RoPE table (``freqs_cis``) is a model
buffer the compressor reads, built here as cos/sin of pos * theta^(-2i/64).
"""
from __future__ import annotations

import math

import numpy as np

D = 512
V4, V41, V41_FP4 = 0, 1, 2


def bf16_from_f32(a: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit pattern (uint16), round to nearest even; finite inputs."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    out = np.empty(a.shape, np.uint16)
    flat_in = a.reshape(-1).view(np.uint32)
    flat_out = out.reshape(-1)
    step = 1 << 24
    for s in range(0, flat_in.size, step):
        u = flat_in[s:s + step].astype(np.uint64)
        u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
        flat_out[s:s + step] = u.astype(np.uint16)
    return out


def bf16_normal(rng: np.random.Generator, shape) -> np.ndarray:
    """bf16 bits of float32 N(0, 1) samples, generated in chunks."""
    n = int(np.prod(shape))
    out = np.empty(n, np.uint16)
    step = 1 << 24
    for s in range(0, n, step):
        m = min(step, n - s)
        out[s:s + m] = bf16_from_f32(rng.standard_normal(m, dtype=np.float32))
    return out.reshape(shape)


def rope_table(max_pos: int, theta: float = 10000.0, rope_dim: int = 64) -> np.ndarray:
    """freqs_cis as fp32 [max_pos, rope_dim]: (cos, sin) of pos * theta^(-2i/rope_dim)
    for the rope_dim/2 complex pairs, interleaved."""
    i = np.arange(rope_dim // 2, dtype=np.float64)
    inv = theta ** (-2.0 * i / rope_dim)
    ang = np.arange(max_pos, dtype=np.float64)[:, None] * inv[None, :]
    t = np.empty((max_pos, rope_dim), np.float64)
    t[:, 0::2] = np.cos(ang)
    t[:, 1::2] = np.sin(ang)
    return t.astype(np.float32)


def _page_table(rng, pages_per_req, max_pages=None, permute=True):
    """int32 [n_req, max_pages]; physical page 0 is reserved (never handed out)."""
    total = int(sum(pages_per_req))
    phys = (rng.permutation(total) + 1) if permute else np.arange(1, total + 1)
    if max_pages is None:
        max_pages = max(1, max(pages_per_req) if pages_per_req else 1)
    pt = np.zeros((len(pages_per_req), max_pages), np.int32)
    o = 0
    for r, p in enumerate(pages_per_req):
        pt[r, :p] = phys[o:o + p]
        o += p
    return pt, total + 1


def _ext(lengths, n_slots=None, pad_first=None):
    """int32 [2, n_slots]: first row and row count per request slot; slots past
    the batch hold no rows."""
    n_slots = len(lengths) if n_slots is None else n_slots
    ext = np.zeros((2, n_slots), np.int32)
    first = np.concatenate([[0], np.cumsum(lengths)[:-1]]) if len(lengths) else []
    ext[0, :len(lengths)] = first
    ext[1, :len(lengths)] = lengths
    if pad_first is not None:
        ext[0, len(lengths):] = pad_first
    return ext


def cfg1_v41_roundtrip(seed: int = 0):
    """V41 fp8 round trip: 256 tokens x 512 bf16 N(0,1) with 1% of entries x50,
    ratio 1 store-only, page size 64, identity page table (logical p ->
    physical p + 1, page 0 reserved); then dequant the 256 written rows."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((256, D), dtype=np.float32)
    n_out = int(0.01 * x.size)
    idx = rng.choice(x.size, n_out, replace=False)
    x.reshape(-1)[idx] *= np.float32(50.0)
    page_bits = 6
    pt, n_pages = _page_table(rng, [256 >> page_bits], permute=False)
    return dict(name="v41_roundtrip_256x512", layout=V41, ratio=1,
                rows=bf16_from_f32(x), score=None, ext=_ext([256]),
                page_table=pt, page_bits=page_bits, norm_w=None, freqs=None,
                eps=1e-6, n_out=256, pool_rows=n_pages << page_bits,
                lengths=[256])


def cfg2_ratio2_small(seed: int = 2):
    """Ratio-2 fused compressor, V41: 4 requests with extend lengths
    {37, 512, 1024, 2047}; fused | kv | score | bf16 N(0,1) rows (padded to
    4096 rows: DP padding rows belong to no request; 8 request slots, slots
    past the batch hold no rows); RMSNorm weight U(0.5, 1.5); RoPE theta
    10000; page size 64 with a random permutation of physical pages 1..64;
    2048 output rows, those past the plan's total are padding."""
    rng = np.random.default_rng(seed)
    lengths = [37, 512, 1024, 2047]
    t_pad = 4096
    rows = bf16_normal(rng, (t_pad, 2 * D))
    w = bf16_from_f32(rng.uniform(0.5, 1.5, D).astype(np.float32))
    page_bits = 6
    rows_per_req = [n // 2 for n in lengths]
    pages = [-(-n // (1 << page_bits)) for n in rows_per_req]
    # physical pages drawn from a permutation of 1..64 (page 0 reserved)
    perm = rng.permutation(64) + 1
    pt = np.zeros((8, 16), np.int32)
    o = 0
    for r, p in enumerate(pages):
        pt[r, :p] = perm[o:o + p]
        o += p
    return dict(name="ratio2_v41_4req_3620tok", layout=V41, ratio=2, rows=rows,
                score=None, ext=_ext(lengths, n_slots=8, pad_first=sum(lengths)),
                page_table=pt, page_bits=page_bits, norm_w=w,
                freqs=rope_table(4096), eps=1e-6, n_out=2048,
                pool_rows=65 << page_bits, lengths=lengths)


def cfg3_fp4_store(seed: int = 3, tokens: int = 32768):
    """V41_FP4: ratio-1 store of 32768 tokens x 512 bf16 N(0,1) into page size
    128 (one request, logical p -> physical p + 1), then full dequant."""
    rng = np.random.default_rng(seed)
    rows = bf16_normal(rng, (tokens, D))
    page_bits = 7
    pt, n_pages = _page_table(rng, [-(-tokens // (1 << page_bits))], permute=False)
    return dict(name=f"fp4_store_{tokens}x512", layout=V41_FP4, ratio=1, rows=rows,
                score=None, ext=_ext([tokens]), page_table=pt, page_bits=page_bits,
                norm_w=None, freqs=None, eps=1e-6, n_out=tokens,
                pool_rows=n_pages << page_bits, lengths=[tokens])


def cfg4_gather(seed: int = 4, pool_rows: int = 1 << 20, n_ids: int = 1 << 18,
                page_bits: int = 6):
    """Sparse-prefill gather-dequant: a V41 pool of 1,048,576 rows (page 0
    reserved, the rest filled by the ratio-1 store-only path from bf16 N(0,1)
    latents), then 262,144 unique shuffled row ids from the filled rows,
    read by 4 layers that share one kv_source."""
    rng = np.random.default_rng(seed)
    filled = pool_rows - (1 << page_bits)
    rows = bf16_normal(rng, (filled, D))
    pt, _ = _page_table(rng, [filled >> page_bits], permute=False)
    ids = (rng.choice(filled, n_ids, replace=False) + (1 << page_bits)).astype(np.int32)
    return dict(name=f"gather_v41_{n_ids}_of_{pool_rows}", layout=V41, ratio=1,
                rows=rows, score=None, ext=_ext([filled]), page_table=pt,
                page_bits=page_bits, norm_w=None, freqs=None, eps=1e-6,
                n_out=filled, pool_rows=pool_rows, ids=ids, layers=4,
                lengths=[filled])


def cfg5_lengths(seed: int = 7, n_req: int = 64, target: int = 262144):
    """Lognormal(ln 4096, 0.6) request lengths, clipped to [2, 32768],
    rescaled to sum ~ target and rounded."""
    rng = np.random.default_rng(seed)
    raw = np.clip(rng.lognormal(math.log(4096.0), 0.6, n_req), 2, 32768)
    lens = np.clip(np.rint(raw * (target / raw.sum())), 2, 32768).astype(np.int64)
    return rng, [int(v) for v in lens]


def cfg5_long_prefill(seed: int = 7, n_req: int = 64, target: int = 262144,
                      topk: int = 2048, page_bits: int = 6):
    """Long prefill batch: 64 requests with lognormal lengths (median 4096,
    capped at 32768, ~262k tokens), ratio-2 compressors writing V41 rows at
    page size 64 over random permuted page tables; then each request's
    top-2048 compressed ids (min(2048, rows) unique random ids, -1 padded)
    for one gather-dequant.  bf16 N(0,1) fused | kv | score | inputs,
    RMSNorm weight U(0.5, 1.5), RoPE theta 10000."""
    rng, lens = cfg5_lengths(seed, n_req, target)
    total = sum(lens)
    rows = bf16_normal(rng, (total, 2 * D))
    w = bf16_from_f32(rng.uniform(0.5, 1.5, D).astype(np.float32))
    rows_per_req = [n // 2 for n in lens]
    pages = [-(-n // (1 << page_bits)) for n in rows_per_req]
    pt, n_pages = _page_table(rng, pages)
    top = np.full((n_req, topk), -1, np.int32)
    for r, n in enumerate(rows_per_req):
        m = min(topk, n)
        top[r, :m] = rng.choice(n, m, replace=False)
    n_out = sum(rows_per_req)
    return dict(name=f"long_prefill_{n_req}req_{total}tok", layout=V41, ratio=2,
                rows=rows, score=None, ext=_ext(lens), page_table=pt,
                page_bits=page_bits, norm_w=w, freqs=rope_table(32768), eps=1e-6,
                n_out=n_out, pool_rows=n_pages << page_bits, lengths=lens,
                topk=top, token_to_req=np.arange(n_req, dtype=np.int32))


def decode_verify(seed: int = 11, n_req: int = 512, n_new: int = 4, ring_size: int = 4,
                  max_prefix: int = 8192, page_bits: int = 6):
    """Ratio-2 decode / speculative-verify step: n_req requests, each with a
    cached prefix of random length (so half start at an odd position and
    complete their first pair with the token held in the pair-state ring),
    n_new new tokens (1 = decode, 1 + draft = verify); fused | kv | score |
    bf16 N(0,1) rows; a ring [n_req, ring_size, 1024] pre-filled with bf16
    N(0,1) entries standing for earlier steps' tokens; RMSNorm weight
    U(0.5, 1.5); RoPE theta 10000; random permuted page tables."""
    rng = np.random.default_rng(seed)
    p0 = rng.integers(0, max_prefix, n_req).astype(np.int32)
    rows = bf16_normal(rng, (n_req * n_new, 2 * D))
    ring = bf16_normal(rng, (n_req, ring_size, 2 * D))
    w = bf16_from_f32(rng.uniform(0.5, 1.5, D).astype(np.float32))
    max_c = (max_prefix + n_new) // 2 + 1
    pages = -(-max_c // (1 << page_bits))
    pt, n_pages = _page_table(rng, [pages] * n_req)
    ext = _ext([n_new] * n_req)
    n_out = int(sum(((int(a) + n_new) >> 1) - (int(a) >> 1) for a in p0))
    return dict(name=f"decode_verify_{n_req}req_{n_new}tok", layout=V41, ratio=2, rows=rows,
                score=None, ext=ext, start_pos=p0, ring=ring, page_table=pt,
                page_bits=page_bits, norm_w=w, freqs=rope_table(max_prefix + n_new + 2),
                eps=1e-6, n_out=n_out, pool_rows=n_pages << page_bits,
                lengths=[n_new] * n_req)


def c1_page_table(lengths, seed: int = 107, page_bits: int = 6):
    """Random permuted page tables for one compressed row per token (the
    ratio-1 compressor over a batch of requests of these lengths): int32
    [n_req, max_pages] and the pool's row count (page 0 reserved)."""
    rng = np.random.default_rng(seed)
    pt, n_pages = _page_table(rng, [-(-n // (1 << page_bits)) for n in lengths])
    return pt, n_pages << page_bits


def c1_long_prefill(seed: int = 7, n_req: int = 64, target: int = 262144, page_bits: int = 6):
    """The long-prefill batch through the ratio-1 compressor with RMSNorm and
    RoPE (the full c1 form): the same 64 lognormal requests, fused
    | kv | score | bf16 rows (the score columns unused), RMSNorm weight and
    RoPE table as the ratio-2 batch; one V41 row per token at its position,
    page size 64 over random permuted page tables (seed + 100)."""
    c = cfg5_long_prefill(seed, n_req, target, page_bits=page_bits)
    pt, pool_rows = c1_page_table(c["lengths"], seed + 100, page_bits)
    return dict(c, name=f"c1_long_prefill_{n_req}req_{sum(c['lengths'])}tok", ratio=1,
                page_table=pt, n_out=sum(c["lengths"]), pool_rows=pool_rows, topk=None)


CONFIGS = {
    1: cfg1_v41_roundtrip,
    2: cfg2_ratio2_small,
    3: cfg3_fp4_store,
    4: cfg4_gather,
    5: cfg5_long_prefill,
}
