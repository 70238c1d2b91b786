/*
 * dsv4kv -- DeepSeek-V4.1 compressed-KV write and read on one GB300 (sm_103a).
 *
 * Plain C ABI.  Every pointer argument is a DEVICE pointer owned by the caller
 * unless marked "host"; the library keeps no reference to any of them after a
 * call returns (the reuse buffer only remembers the caller's storage pointer
 * and the identity of the last source it filled).  Every call that touches the
 * GPU is asynchronous on `stream` (a cudaStream_t passed as void*; NULL = the
 * legacy default stream), never synchronises the host, allocates no memory,
 * and reads its metadata (offsets, page tables, out_loc, ids) on the device,
 * so a sequence of calls can be captured into a CUDA graph and replayed with
 * the metadata refreshed in place.
 *
 * Return value: DSV4KV_OK (0) or a negative status; see the enum below.
 * Host-checkable argument errors return before anything is launched.  Faults
 * that only the device can see (an id or slot outside the pool, a request
 * whose rows run past the input, a position past the RoPE table) never trap:
 * the affected row is written as zeros or skipped, as each call documents,
 * and one is added to *err_word (a caller-zeroed device int32; may be NULL).
 *
 * Sources, cited by page title and section:
 *   [KVL]  sglang PR #39652 "dsv4.1: compression, KV I/O, and metadata
 *          kernels" -- Summary: KVLayout, PagedKV<layout, page_bits>::row,
 *          v41::store_row; the c1/c2 compressors; the V4.1 dequantizers;
 *          review: store_row_fp8's ue8m0 formula, clear_negative_zero.
 *   [EXT]  sglang PR #46230 (ratio-2 fused compressor in the prefill CUDA
 *          graph) -- low_ratio_extend_offsets; the | kv | score | projection.
 *   [BUF]  sglang PR #45909 (sparse-prefill KV dequant reuse) --
 *          SparsePrefillKVBuffer and get_with_head.
 *   [TOPK] flashinfer_sparse.py -- _compressed_topk_to_slots and
 *          compressed_block_size = block_size // compress_ratio.
 */
#ifndef DSV4KV_H
#define DSV4KV_H

#ifdef __cplusplus
extern "C" {
#endif

/* Paged main-KV row formats [KVL, KVLayout bullet].  One row = one 512-dim
 * compressed latent (dims 0..447 "nope", 448..511 "rope").
 *   DSV4KV_V4      584 B: 448 e4m3 nope codes (byte d = dim d), then the 64
 *                  rope dims as bf16 (bytes 448..575), then 7 ue8m0 scales
 *                  (byte 576+g scales dims 64g..64g+63) and a zero byte.
 *                  Rows are 8-byte aligned only.
 *   DSV4KV_V41     528 B: 512 e4m3 codes (byte d = dim d), then 16 ue8m0
 *                  scale bytes (byte 512+g scales dims 32g..32g+31).
 *   DSV4KV_V41_FP4 288 B: 256 bytes of e2m1 codes (byte i holds dim 2i in
 *                  its low nibble, dim 2i+1 in its high nibble), then 32 e4m3
 *                  scale bytes (byte 256+g scales dims 16g..16g+15). */
typedef enum {
    DSV4KV_V4 = 0,
    DSV4KV_V41 = 1,
    DSV4KV_V41_FP4 = 2
} dsv4kv_layout;

enum {
    DSV4KV_OK = 0,
    DSV4KV_EINVAL = -1,  /* NULL / misaligned pointer, bad enum, negative size */
    DSV4KV_ENOTSUP = -2, /* a layout or mode that is not built */
    DSV4KV_ERANGE = -3,  /* a size past a documented limit */
    DSV4KV_ECUDA = -4    /* a CUDA launch failed; see dsv4kv_last_cuda_error */
};

/* Limits of this build. */
#define DSV4KV_DIM 512
#define DSV4KV_MAX_SLOTS 4096          /* request slots per compress_store call */
#define DSV4KV_MAX_POOL_ROWS 2147483647LL /* slots and ids are int32 */

/* Bytes per row of `layout` (584 / 528 / 288), or DSV4KV_EINVAL.  Host only. */
int dsv4kv_row_bytes(int layout);

/* The cudaError_t of the last DSV4KV_ECUDA on this host thread (0 if none). */
int dsv4kv_last_cuda_error(void);

/* Static description of a status code.  Host only. */
const char *dsv4kv_status_string(int status);

/*
 * Fused compressor: pool -> RMSNorm -> RoPE -> quantize -> paged store.
 * [KVL, c1/c2 bullet: "pair-pooling (ratio 2), RMSNorm, RoPE and the main-KV
 * write in one launch, returning the pre-RoPE latent; out_loc == 0 marks a
 * padded graph row"; EXT for the offsets and the fused projection.]
 *
 * Plan.  extend_offsets is int32 [2, n_slots]: row 0 = first source row of
 * each request slot, row 1 = its source row count (<= 0: no rows).  Output
 * rows are numbered request by request: request r contributes
 * count_r / ratio rows (an odd trailing token of a ratio-2 request yields no
 * row), row j of request r pools source rows first_r + ratio*j + t, t < ratio,
 * and sits at position ratio*j.  Output rows k >= the plan's total are
 * padding: nothing is stored and latent_out / prequant_out rows are zeroed.
 *
 * Per row (fp32 on the device):
 *   ratio 1: x = kv[first_r + j]
 *   ratio 2: x[d] = sum_t softmax_t(score[src+t][d]) * kv[src+t][d]
 *   RMSNorm (if rmsnorm_w): x = x / sqrt(mean(x^2) + eps) * w
 *   latent_out (if given) = bf16(x)                    (post-norm, pre-RoPE)
 *   RoPE (if freqs_cis): pairs (448+2i, 449+2i), i < 32, rotated by
 *        (c, s) = freqs_cis[pos][2i], freqs_cis[pos][2i+1]
 *   prequant_out (if given) = x                        (what is quantized)
 *   store_row:  V41 (V4: per 64 nope dims, rope dims kept as bf16):
 *        per 32 dims e = max((bits(amax)>>23) - 8 +
 *        ((bits(amax) & 0x7FFFFF) > 0x600000), 114), the ue8m0 byte equal to
 *        127 + ceil(log2(max(amax/448, 1e-4))); codes e4m3_rn_satfinite(
 *        x * 2^(127-e)).  V41_FP4: per 16 dims s = e4m3_rn_satfinite(amax/6),
 *        codes e2m1_rn_satfinite(x / s) (IEEE fp32 divisions), 0 if s == 0.
 *        A code that rounds to -0 is stored as +0.
 *   slot = out_loc[k] if out_loc, else
 *        page_table[r][j >> page_bits] << page_bits | (j & (2^page_bits - 1))
 *        (compressed pages hold 2^page_bits rows [TOPK]); slot 0 = do not
 *        store (page 0 is reserved); the row lands at
 *        pool + (slot >> page_bits) * (row_bytes << page_bits)
 *             + (slot & (2^page_bits - 1)) * row_bytes      [KVL, PagedKV].
 *
 * Arguments:
 *   layout        DSV4KV_V4, DSV4KV_V41 or DSV4KV_V41_FP4.
 *   ratio         1 or 2.
 *   rows          bf16 [n_rows, row_stride], 16-B aligned; kv in columns
 *                 0..511.  For ratio 2 with score == NULL the score sits in
 *                 columns 512..1023 (the fused | kv | score | projection).
 *   row_stride    elements, multiple of 8, >= 512 (>= 1024 fused ratio 2).
 *   score         NULL or bf16 [n_rows, score_stride] (ratio 2 only).
 *   extend_offsets, n_slots   see Plan; 0 <= n_slots <= DSV4KV_MAX_SLOTS.
 *   page_table    int32 [n_slots, max_pages]; required when out_loc == NULL.
 *   page_bits     log2 rows per page, 0..16.
 *   rmsnorm_w     NULL (no norm) or bf16 [512], 16-B aligned; eps >= 0.
 *   freqs_cis     NULL (no RoPE) or fp32 [max_pos, 64], 16-B aligned.
 *   out_loc       NULL or int32 [n_out].
 *   n_out         output rows (>= the plan's total to store every row);
 *                 0 is a no-op.
 *   pool          [pool_rows * row_bytes] bytes, 16-B aligned;
 *                 1 <= pool_rows <= DSV4KV_MAX_POOL_ROWS.
 *   latent_out    NULL or bf16 [n_out, 512], 16-B aligned.
 *   prequant_out  NULL or fp32 [n_out, 512], 16-B aligned.
 * Device faults (+1 on err_word each): source rows outside [0, n_rows) or a
 * position >= max_pos (row not computed: zero latent/prequant, not stored);
 * a slot < 0 or >= pool_rows, or a page index >= max_pages (row computed,
 * not stored).
 */
int dsv4kv_compress_store(int layout, int ratio,
                          const void *rows, long long n_rows, long long row_stride,
                          const void *score, long long score_stride,
                          const int *extend_offsets, int n_slots,
                          const int *page_table, int max_pages, int page_bits,
                          const void *rmsnorm_w, float eps,
                          const float *freqs_cis, int max_pos,
                          const int *out_loc, int n_out,
                          void *pool, long long pool_rows,
                          void *latent_out, float *prequant_out,
                          int *err_word, void *stream);

/*
 * dsv4kv_compress_store with per-request start positions and the ratio-2
 * pair-state ring: the general extend step that covers prefill with a
 * cached prefix (chunked prefill), decode (one new token per request) and
 * speculative verify (1 + draft tokens) [KVL, c1/c2 bullet: the ratio-2
 * decode compressor keeps a pair-state ring; review: the c2 kernel completes
 * a pair at an odd position and loads RoPE frequencies at pos - 1].
 *
 *   start_pos   NULL (every slot starts at 0) or int32 [n_slots]: position
 *               p0 of slot r's first new token; new token t (t < count_r) is
 *               at position p0 + t in source row first_r + t.  Positions
 *               start at 0: a row, or a ring token, at a negative position
 *               counts one fault in err_word and is neither stored nor
 *               written to the ring.
 *   Rows: compressed row c pools the tokens at positions ratio*c ..
 *         ratio*c + ratio - 1 and is produced by the step that holds its
 *         last token: ratio 1: c in [p0, p0 + n); ratio 2: c in
 *         [p0 / 2, (p0 + n) / 2).  Output rows stay numbered request by
 *         request; the page-table index of a row is c; RoPE position ratio*c.
 *   ring        NULL or bf16 [n_slots, ring_size, 1024] (ratio 2 only),
 *               16-B aligned, caller-owned state that lives across steps:
 *               entry (q / 2) % ring_size holds the kv | score of the token
 *               at even position q.  When p0 is odd, the first pair reads
 *               token p0 - 1 from the ring (with ring == NULL that row is a
 *               fault).  After the step, each even-position new token among
 *               the step's last 2 * ring_size positions is written to the
 *               ring, so ring_size >= 1 + (draft tokens) / 2 keeps every
 *               token a rolled-back verify step can need.
 *   ring_size   entries per request (0 when ring is NULL).
 * Every other argument is as in dsv4kv_compress_store (which is this call
 * with start_pos = ring = NULL).  Within one call the ring is read before
 * it is written; calls on one stream see each other's ring updates.
 */
int dsv4kv_compress_store_ring(int layout, int ratio,
                               const void *rows, long long n_rows, long long row_stride,
                               const void *score, long long score_stride,
                               const int *extend_offsets, int n_slots,
                               const int *start_pos, void *ring, int ring_size,
                               const int *page_table, int max_pages, int page_bits,
                               const void *rmsnorm_w, float eps,
                               const float *freqs_cis, int max_pos,
                               const int *out_loc, int n_out,
                               void *pool, long long pool_rows,
                               void *latent_out, float *prequant_out,
                               int *err_word, void *stream);

/*
 * Paged gather-dequant [KVL, dequantize_k_cache_paged for the V4.1 layouts]:
 *   out_bf16[i][d] = bf16(code(ids[i], d) * scale(ids[i], d)), i < n.
 * V41 / V4: scale = 2^(e - 127) of the group's ue8m0 byte (V4 rope dims are
 * copied); V41_FP4: the group's e4m3 scale.  Products are exact in bf16 for every row store_row writes.
 * ids[i] < 0 gives a zero row; ids[i] >= pool_rows gives a zero row and one
 * fault.  The pool is addressed as rows of row_bytes (pages are unpadded, so
 * a slot's byte offset is slot * row_bytes whatever the page size).
 *   pool      [pool_rows * row_bytes] bytes, 16-B aligned.
 *   ids       int32 [n].
 *   out_bf16  bf16 [n, 512], 16-B aligned.
 *   n         0 <= n < 2^31; 0 is a no-op.
 */
int dsv4kv_dequant_gather(int layout, const void *pool, long long pool_rows,
                          const int *ids, long long n, void *out_bf16,
                          int *err_word, void *stream);

/*
 * Fused top-k gather-dequant: dsv4kv_topk_to_slots followed by
 * dsv4kv_dequant_gather in one launch, without the slot buffer [TOPK; KVL,
 * dequantize_k_cache_paged]:
 *   out_bf16[t*k + c] = dequant(pool row slot(t, c)), slot as in
 *   dsv4kv_topk_to_slots; slot -1 gives a zero row, a slot >= pool_rows a
 *   zero row and one fault.
 * lens (nullable int32 [n_tok]) must be zeroed by the caller; the call adds
 * each token's number of slots >= 0.  Argument rules as for the two calls it
 * fuses; out_bf16 is [n_tok * k, 512].
 */
int dsv4kv_dequant_gather_topk(int layout, const void *pool, long long pool_rows,
                               const int *topk, int n_tok, int k,
                               const int *token_to_req, const unsigned char *is_valid,
                               const int *page_table, int n_req, int max_pages, int page_bits,
                               void *out_bf16, int *lens, int *err_word, void *stream);

/*
 * Short-context ids [KVL test table: fill_all_compressed_indices; TOPK: the
 * indexer's "short-context bypass", where every compressed row a token can
 * see is selected]: topk_out[t*k + j] = j for j < lens_in[t], else -1
 * (lens_in[t] < 0 selects nothing; only the first k are written).  lens_in
 * is the caller's per-token visible compressed length, e.g. (position + 1) /
 * ratio in a causal prefill.  topk_out: int32 [n_tok, k] device; lens_in:
 * int32 [n_tok] device.  DSV4KV_ERANGE if k > 65536.
 */
int dsv4kv_fill_all_compressed_indices(int *topk_out, int n_tok, int k, const int *lens_in,
                                       void *stream);

/*
 * dsv4kv_dequant_gather_topk with the short-context ids of
 * dsv4kv_fill_all_compressed_indices made on the fly (no id buffer): row
 * t*k + j gathers compressed row j of token t's request when j < lens_in[t],
 * a zero row otherwise.  Same arguments, lens and faults as
 * dsv4kv_dequant_gather_topk with lens_in in place of topk.
 */
int dsv4kv_dequant_gather_all(int layout, const void *pool, long long pool_rows,
                              const int *lens_in, int n_tok, int k,
                              const int *token_to_req, const unsigned char *is_valid,
                              const int *page_table, int n_req, int max_pages, int page_bits,
                              void *out_bf16, int *lens, int *err_word, void *stream);

/*
 * Request-local top-k compressed ids -> physical pool slots [TOPK,
 * _compressed_topk_to_slots, single-rank branch]:
 *   slots[t][c] = page_table[req][id >> page_bits] << page_bits
 *                 | (id & (2^page_bits - 1)),  id = topk[t][c], req = token_to_req[t]
 * (formed in 64 bits) or -1 when id < 0, when is_valid (nullable uint8
 * [n_tok]) is 0 for t, or on a fault: req outside [0, n_req) (one fault per
 * token), a page index >= max_pages, a negative page entry, or a slot past
 * 2^31 - 1 (one fault per entry).  lens (nullable int32 [n_tok]) = number of
 * slots >= 0 in the row.
 *   topk int32 [n_tok, k]; token_to_req int32 [n_tok];
 *   page_table int32 [n_req, max_pages]; slots int32 [n_tok, k];
 *   0 <= k <= 65536, page_bits 0..16.
 */
int dsv4kv_topk_to_slots(const int *topk, int n_tok, int k,
                         const int *token_to_req, const unsigned char *is_valid,
                         const int *page_table, int n_req, int max_pages, int page_bits,
                         int *slots, int *lens, int *err_word, void *stream);

/*
 * Self-test of the bounded waits (no counterpart on the pages; failure
 * detection of this library).  Every pipelined kernel waits on mbarriers
 * with a poll limit; when a limit runs out the kernel adds
 * DSV4KV_FAULT_TIMEOUT to err_word and returns instead of hanging.  This call
 * runs that wait on a barrier nothing arrives on: one warp gives up after
 * `polls` polls (1..2^24) and a second warp must see its abort flag and give
 * up too.  Expected result: *err_word += DSV4KV_FAULT_TIMEOUT and
 * *gave_up += 2 (both device int32, caller-zeroed).
 * After any call reports DSV4KV_FAULT_TIMEOUT, everything that launch wrote
 * (pool rows, gathered rows, ring entries, lens) is undefined, rows of other
 * CTAs included: a copy still in flight when a CTA gave up may land in shared
 * memory that a later CTA uses.
 */
#define DSV4KV_FAULT_TIMEOUT (1 << 24)
int dsv4kv_selftest_bounded_wait(int polls, int *err_word, int *gave_up, void *stream);

/*
 * Self-test of the V41_FP4 quantizer's division (no counterpart on the pages):
 * for each i, with s = the e4m3 value of scale_codes[i], writes the
 * quantizer's quotient x[i] / s (reciprocal plus one correction step, in
 * the paired fp32 form the quantizer uses: elements 2j and 2j + 1 together)
 * to q_fast[i] and the IEEE division to q_ieee[i]; the two must agree bit
 * for bit.  x, q_fast, q_ieee: fp32 [n] device; scale_codes: uint8 [n]
 * device.
 */
int dsv4kv_selftest_fp4_quotient(const float *x, const unsigned char *scale_codes, long long n,
                                 float *q_fast, float *q_ieee, void *stream);

/*
 * Self-test of the reciprocal that the V41_FP4 quantizer's division starts
 * from (no counterpart on the pages): for each i, with s = the e4m3 value of
 * codes[i], writes the quantizer's reciprocal (one Newton-Raphson step from
 * the hardware approximation) to y_fast[i] and the IEEE reciprocal to
 * y_ieee[i]; for every positive finite code (0x01..0x7E) the two must agree
 * bit for bit.  codes: uint8 [n] device; y_fast, y_ieee: fp32 [n] device.
 * Returns DSV4KV_EINVAL for n < 0, a null or misaligned pointer.
 */
int dsv4kv_selftest_e4m3_recip(const unsigned char *codes, long long n, float *y_fast,
                               float *y_ieee, void *stream);

/*
 * Fake quantization [KVL test table: fake_quant_compressed_kv,
 * fake_quant_fp4]: out_bf16[i] = bf16(dequant(store_row(in_bf16[i]))) for
 * each of n rows, with the layout's own store_row and dequantizer, so the
 * result equals dsv4kv_compress_store (store-only) followed by
 * dsv4kv_dequant_gather of that row, bit for bit.  in_bf16: [n, in_stride]
 * (in_stride >= 512, a multiple of 8 elements), out_bf16: [n, 512]; both
 * 16-byte aligned; out_bf16 == in_bf16 (in_stride 512) is allowed.
 */
int dsv4kv_fake_quant(int layout, const void *in_bf16, long long n, long long in_stride,
                      void *out_bf16, void *stream);

/*
 * Source-reuse buffer [BUF]: the shared bf16 buffer the sparse-prefill layers
 * read.  It remembers the source it last dequantized -- (layout, pool,
 * pool_rows, ids pointer, n) -- and a get_with_head for that same source is a
 * hit: the rows are already there and nothing is launched.  A plain get, a
 * re-init (reallocation) or begin_forward forgets the head.  Reuse is sound
 * while no call between the fill and the hit writes the pool rows or the ids
 * (within one forward no later layer writes the source cache, and graph
 * replay keeps layer order).
 *
 * The struct is host memory owned by the caller; `storage` is the caller's
 * device buffer of capacity_rows x 512 bf16, 16-B aligned.
 */
typedef struct dsv4kv_kvbuf {
    void *storage;
    long long capacity_rows;
    /* the head: the source the storage holds, compared field by field */
    int head_valid;
    int head_layout;
    const void *head_pool;
    long long head_pool_rows;
    const int *head_ids;               /* ids, top-k ids, or short-context lengths */
    long long head_n;                  /* rows gathered */
    int head_form;                     /* DSV4KV_KVBUF_IDS / _TOPK / _ALL */
    int head_k;                        /* top-k and short-context forms: ids per token */
    const int *head_token_to_req;      /* the id mapping (0 / NULL for the ids form) */
    const unsigned char *head_is_valid;
    const int *head_page_table;
    int head_n_req;
    int head_max_pages;
    int head_page_bits;
} dsv4kv_kvbuf;

/* head_form values: which gather filled the storage */
#define DSV4KV_KVBUF_IDS 0             /* dsv4kv_dequant_gather (pool slots) */
#define DSV4KV_KVBUF_TOPK 1            /* dsv4kv_dequant_gather_topk */
#define DSV4KV_KVBUF_ALL 2             /* dsv4kv_dequant_gather_all */

/* (Re)initialise: set storage and capacity, forget the head.  Host only. */
int dsv4kv_kvbuf_init(dsv4kv_kvbuf *buf, void *storage_bf16, long long capacity_rows);

/* Start of a new forward: forget the head.  Host only. */
void dsv4kv_kvbuf_begin_forward(dsv4kv_kvbuf *buf);

/* Plain get of the first n rows (host pointer *rows = storage): forgets the
 * head.  DSV4KV_ERANGE if n > capacity.  Host only. */
int dsv4kv_kvbuf_get(dsv4kv_kvbuf *buf, long long n, void **rows);

/* The head decision alone: *hit = 1 if (layout, pool, pool_rows, ids, n) is
 * the head, else 0 and the head becomes that source.  Launches nothing; for
 * callers that run their own dequant on a miss.  Host only. */
int dsv4kv_kvbuf_lookup(dsv4kv_kvbuf *buf, int layout, const void *pool,
                        long long pool_rows, const int *ids, long long n, int *hit);

/* get_with_head: *rows = storage; on a miss runs dsv4kv_dequant_gather into
 * the storage and sets the head (cleared again if the launch fails); on a hit
 * launches nothing.  Same argument rules as dsv4kv_dequant_gather. */
int dsv4kv_kvbuf_get_with_head(dsv4kv_kvbuf *buf, int layout, const void *pool,
                               long long pool_rows, const int *ids, long long n,
                               void **rows, int *hit, int *err_word, void *stream);

/* get_with_head whose gather ids are request-local top-k ids: the head is
 * (layout, pool, pool_rows, topk pointer, n_tok * k) and every mapping
 * argument (the token_to_req, is_valid and page_table pointers, n_req,
 * max_pages, page_bits, k), compared exactly, so the same top-k buffer
 * mapped through another table is a miss; on a miss runs
 * dsv4kv_dequant_gather_topk into the storage (lens as there, written only
 * on a miss), on a hit launches nothing. */
int dsv4kv_kvbuf_get_with_head_topk(dsv4kv_kvbuf *buf, int layout, const void *pool,
                                    long long pool_rows, const int *topk, int n_tok, int k,
                                    const int *token_to_req, const unsigned char *is_valid,
                                    const int *page_table, int n_req, int max_pages, int page_bits,
                                    void **rows, int *lens, int *hit, int *err_word, void *stream);

/* get_with_head whose ids are the short-context ids (dsv4kv_dequant_gather_all):
 * the head is (layout, pool, pool_rows, lens_in pointer, n_tok * k) and the
 * mapping arguments as for the top-k form, with its own head_form, so a
 * top-k fill never hits for it; a miss runs dsv4kv_dequant_gather_all into
 * the storage, a hit launches nothing. */
int dsv4kv_kvbuf_get_with_head_all(dsv4kv_kvbuf *buf, int layout, const void *pool,
                                   long long pool_rows, const int *lens_in, int n_tok, int k,
                                   const int *token_to_req, const unsigned char *is_valid,
                                   const int *page_table, int n_req, int max_pages, int page_bits,
                                   void **rows, int *lens, int *hit, int *err_word, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* DSV4KV_H */
