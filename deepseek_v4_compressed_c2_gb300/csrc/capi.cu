// The C ABI (include/dsv4kv.h): argument validation, dispatch to the
// launchers, and the source-reuse buffer's head (host state only).
//
// Every host-checkable error is rejected here, before any CUDA call, so a
// failing call launches nothing.  Device-only faults are counted by the
// kernels in the caller's err_word.
#include <atomic>
#include <cstdint>
#include <cuda_runtime.h>

#include "dsv4kv.h"
#include "internal.cuh"
#include "launchers.cuh"
#include "layout.cuh"

namespace dsv4kv {

static_assert(kMaxSlots == DSV4KV_MAX_SLOTS, "plan capacity matches the header");

static thread_local int g_last_cuda_error = 0;

static int cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return DSV4KV_OK;
  g_last_cuda_error = (int)e;
  return DSV4KV_ECUDA;
}

static bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// SMs of the current device, cached per device (atomics: host threads may
// launch concurrently; a race only repeats the query)
int device_sm_count() {
  constexpr int kMaxDevices = 64;
  static std::atomic<int> cache[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 148;
  if (dev < kMaxDevices) {
    const int seen = cache[dev].load(std::memory_order_relaxed);
    if (seen > 0) return seen;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
  if (dev < kMaxDevices) cache[dev].store(n, std::memory_order_relaxed);
  return n;
}

// layouts usable by store / dequant: all three KVLayout members
static int check_rw_layout(int layout) {
  if (layout == DSV4KV_V4 || layout == DSV4KV_V41 || layout == DSV4KV_V41_FP4) return DSV4KV_OK;
  return DSV4KV_EINVAL;
}

static int check_gather(int layout, const void* pool, long long pool_rows, const int* ids,
                        long long n, const void* out) {
  int st = check_rw_layout(layout);
  if (st != DSV4KV_OK) return st;
  if (n < 0 || pool_rows < 0) return DSV4KV_EINVAL;
  if (n > 2147483647LL || pool_rows > DSV4KV_MAX_POOL_ROWS) return DSV4KV_ERANGE;
  if (n == 0) return DSV4KV_OK;
  if (!pool || !ids || !out) return DSV4KV_EINVAL;
  if (!aligned16(pool) || !aligned16(out) || ((uintptr_t)ids & 3u)) return DSV4KV_EINVAL;
  return DSV4KV_OK;
}

}  // namespace dsv4kv

using namespace dsv4kv;

extern "C" {

int dsv4kv_row_bytes(int layout) {
  const int rb = row_bytes_of(layout);
  return rb > 0 ? rb : DSV4KV_EINVAL;
}

int dsv4kv_last_cuda_error(void) { return g_last_cuda_error; }

const char* dsv4kv_status_string(int status) {
  switch (status) {
    case DSV4KV_OK: return "ok";
    case DSV4KV_EINVAL: return "invalid argument (null or misaligned pointer, bad enum, negative size)";
    case DSV4KV_ENOTSUP: return "not supported in this build";
    case DSV4KV_ERANGE: return "size outside a documented limit";
    case DSV4KV_ECUDA: return "CUDA launch failed (see dsv4kv_last_cuda_error)";
    default: return "unknown status";
  }
}

int dsv4kv_compress_store(int layout, int ratio, const void* rows, long long n_rows,
                          long long row_stride, const void* score, long long score_stride,
                          const int* extend_offsets, int n_slots, const int* page_table,
                          int max_pages, int page_bits, const void* rmsnorm_w, float eps,
                          const float* freqs_cis, int max_pos, const int* out_loc, int n_out,
                          void* pool, long long pool_rows, void* latent_out, float* prequant_out,
                          int* err_word, void* stream) {
  return dsv4kv_compress_store_ring(layout, ratio, rows, n_rows, row_stride, score, score_stride,
                                    extend_offsets, n_slots, nullptr, nullptr, 0, page_table,
                                    max_pages, page_bits, rmsnorm_w, eps, freqs_cis, max_pos,
                                    out_loc, n_out, pool, pool_rows, latent_out, prequant_out,
                                    err_word, stream);
}

int dsv4kv_compress_store_ring(int layout, int ratio, const void* rows, long long n_rows,
                               long long row_stride, const void* score, long long score_stride,
                               const int* extend_offsets, int n_slots, const int* start_pos,
                               void* ring, int ring_size, const int* page_table, int max_pages,
                               int page_bits, const void* rmsnorm_w, float eps,
                               const float* freqs_cis, int max_pos, const int* out_loc, int n_out,
                               void* pool, long long pool_rows, void* latent_out,
                               float* prequant_out, int* err_word, void* stream) {
  if (ring && (ratio != 2 || ring_size < 1 || !aligned16(ring))) return DSV4KV_EINVAL;
  if (!ring && ring_size != 0) return DSV4KV_EINVAL;
  if (start_pos && ((uintptr_t)start_pos & 3u)) return DSV4KV_EINVAL;
  int st = check_rw_layout(layout);
  if (st != DSV4KV_OK) return st;
  if (ratio != 1 && ratio != 2) return DSV4KV_EINVAL;
  if (n_out < 0 || n_rows < 0 || n_slots < 0 || pool_rows < 0) return DSV4KV_EINVAL;
  if (page_bits < 0 || page_bits > 16) return DSV4KV_EINVAL;
  if (n_slots > DSV4KV_MAX_SLOTS || pool_rows > DSV4KV_MAX_POOL_ROWS) return DSV4KV_ERANGE;
  if (!(eps >= 0.f)) return DSV4KV_EINVAL;
  if (n_out == 0) return DSV4KV_OK;
  if (!rows || (n_slots > 0 && !extend_offsets) || !pool || pool_rows < 1) return DSV4KV_EINVAL;
  if (!aligned16(rows) || !aligned16(pool) || (row_stride % 8) != 0) return DSV4KV_EINVAL;
  if (row_stride < DSV4KV_DIM || (ratio == 2 && !score && row_stride < 2 * DSV4KV_DIM))
    return DSV4KV_EINVAL;
  if (score && (ratio != 2 || !aligned16(score) || (score_stride % 8) != 0 ||
                score_stride < DSV4KV_DIM))
    return DSV4KV_EINVAL;
  if (!out_loc && (!page_table || max_pages < 1)) return DSV4KV_EINVAL;
  if (page_table && max_pages < 1) return DSV4KV_EINVAL;
  if (rmsnorm_w && !aligned16(rmsnorm_w)) return DSV4KV_EINVAL;
  if (freqs_cis && (!aligned16(freqs_cis) || max_pos < 1)) return DSV4KV_EINVAL;
  if ((latent_out && !aligned16(latent_out)) || (prequant_out && !aligned16(prequant_out)))
    return DSV4KV_EINVAL;
  if (((uintptr_t)extend_offsets & 3u) || (out_loc && ((uintptr_t)out_loc & 3u)) ||
      (page_table && ((uintptr_t)page_table & 3u)))
    return DSV4KV_EINVAL;

  StoreParams p;
  p.rows = static_cast<const __nv_bfloat16*>(rows);
  p.n_rows = n_rows;
  p.row_stride = row_stride;
  p.score = static_cast<const __nv_bfloat16*>(score);
  p.score_stride = score_stride;
  p.ext = extend_offsets;
  p.n_slots = n_slots;
  p.page_table = page_table;
  p.max_pages = page_table ? max_pages : 0;
  p.page_bits = page_bits;
  p.norm_w = static_cast<const __nv_bfloat16*>(rmsnorm_w);
  p.eps = eps;
  p.freqs = freqs_cis;
  p.max_pos = freqs_cis ? max_pos : 0;
  p.out_loc = out_loc;
  p.n_out = n_out;
  p.pool = static_cast<uint8_t*>(pool);
  p.pool_rows = pool_rows;
  p.latent_out = static_cast<__nv_bfloat16*>(latent_out);
  p.prequant_out = prequant_out;
  p.err = err_word;
  p.start_pos = start_pos;
  p.ring = static_cast<__nv_bfloat16*>(ring);
  p.ring_size = ring ? ring_size : 0;
  return cuda_status(launch_compress_store(p, layout, ratio, static_cast<cudaStream_t>(stream)));
}

int dsv4kv_dequant_gather(int layout, const void* pool, long long pool_rows, const int* ids,
                          long long n, void* out_bf16, int* err_word, void* stream) {
  int st = check_gather(layout, pool, pool_rows, ids, n, out_bf16);
  if (st != DSV4KV_OK || n == 0) return st;
  return cuda_status(launch_dequant_gather(layout, static_cast<const uint8_t*>(pool), pool_rows,
                                           ids, n, static_cast<__nv_bfloat16*>(out_bf16),
                                           err_word, static_cast<cudaStream_t>(stream)));
}

static int check_topk(const int* topk, int n_tok, int k, const int* token_to_req,
                      const int* page_table, int n_req, int max_pages, int page_bits) {
  if (n_tok < 0 || k < 0 || n_req < 0 || max_pages < 0) return DSV4KV_EINVAL;
  if (page_bits < 0 || page_bits > 16) return DSV4KV_EINVAL;
  if (k > 65536) return DSV4KV_ERANGE;
  if (n_tok == 0 || k == 0) return DSV4KV_OK;
  if (!token_to_req || !topk) return DSV4KV_EINVAL;
  if (n_req > 0 && max_pages > 0 && !page_table) return DSV4KV_EINVAL;
  if (((uintptr_t)topk & 3u) || ((uintptr_t)token_to_req & 3u) || ((uintptr_t)page_table & 3u))
    return DSV4KV_EINVAL;
  return DSV4KV_OK;
}

int dsv4kv_dequant_gather_topk(int layout, const void* pool, long long pool_rows, const int* topk,
                               int n_tok, int k, const int* token_to_req,
                               const unsigned char* is_valid, const int* page_table, int n_req,
                               int max_pages, int page_bits, void* out_bf16, int* lens,
                               int* err_word, void* stream) {
  int st = check_topk(topk, n_tok, k, token_to_req, page_table, n_req, max_pages, page_bits);
  if (st != DSV4KV_OK) return st;
  const long long n = (long long)n_tok * k;
  st = check_gather(layout, pool, pool_rows, topk, n, out_bf16);
  if (st != DSV4KV_OK || n == 0) return st;
  if ((uintptr_t)lens & 3u) return DSV4KV_EINVAL;
  return cuda_status(launch_dequant_gather_topk(
      layout, static_cast<const uint8_t*>(pool), pool_rows, topk, nullptr, n_tok, k, token_to_req,
      is_valid, page_table, n_req, max_pages, page_bits, static_cast<__nv_bfloat16*>(out_bf16),
      lens, err_word, static_cast<cudaStream_t>(stream)));
}

int dsv4kv_dequant_gather_all(int layout, const void* pool, long long pool_rows,
                              const int* lens_in, int n_tok, int k, const int* token_to_req,
                              const unsigned char* is_valid, const int* page_table, int n_req,
                              int max_pages, int page_bits, void* out_bf16, int* lens,
                              int* err_word, void* stream) {
  // the top-k checks with lens_in standing where the ids would be
  int st = check_topk(lens_in, n_tok, k, token_to_req, page_table, n_req, max_pages, page_bits);
  if (st != DSV4KV_OK) return st;
  const long long n = (long long)n_tok * k;
  st = check_gather(layout, pool, pool_rows, lens_in, n, out_bf16);
  if (st != DSV4KV_OK || n == 0) return st;
  if ((uintptr_t)lens & 3u) return DSV4KV_EINVAL;
  return cuda_status(launch_dequant_gather_topk(
      layout, static_cast<const uint8_t*>(pool), pool_rows, nullptr, lens_in, n_tok, k,
      token_to_req, is_valid, page_table, n_req, max_pages, page_bits,
      static_cast<__nv_bfloat16*>(out_bf16), lens, err_word, static_cast<cudaStream_t>(stream)));
}

int dsv4kv_fill_all_compressed_indices(int* topk_out, int n_tok, int k, const int* lens_in,
                                       void* stream) {
  if (n_tok < 0 || k < 0) return DSV4KV_EINVAL;
  if (k > 65536) return DSV4KV_ERANGE;
  if (n_tok == 0 || k == 0) return DSV4KV_OK;
  if (!topk_out || !lens_in || ((uintptr_t)topk_out & 3u) || ((uintptr_t)lens_in & 3u))
    return DSV4KV_EINVAL;
  return cuda_status(launch_fill_all_indices(topk_out, n_tok, k, lens_in,
                                             static_cast<cudaStream_t>(stream)));
}

int dsv4kv_topk_to_slots(const int* topk, int n_tok, int k, const int* token_to_req,
                         const unsigned char* is_valid, const int* page_table, int n_req,
                         int max_pages, int page_bits, int* slots, int* lens, int* err_word,
                         void* stream) {
  if (n_tok < 0 || k < 0 || n_req < 0 || max_pages < 0) return DSV4KV_EINVAL;
  if (page_bits < 0 || page_bits > 16) return DSV4KV_EINVAL;
  if (k > 65536) return DSV4KV_ERANGE;
  if (n_tok == 0) return DSV4KV_OK;
  if (!token_to_req || !slots || (k > 0 && !topk)) return DSV4KV_EINVAL;
  if (n_req > 0 && max_pages > 0 && !page_table) return DSV4KV_EINVAL;
  if (((uintptr_t)topk & 3u) || ((uintptr_t)token_to_req & 3u) || ((uintptr_t)slots & 3u) ||
      ((uintptr_t)page_table & 3u) || ((uintptr_t)lens & 3u))
    return DSV4KV_EINVAL;
  return cuda_status(launch_topk_to_slots(topk, n_tok, k, token_to_req, is_valid, page_table, n_req,
                                          max_pages, page_bits, slots, lens, err_word,
                                          static_cast<cudaStream_t>(stream)));
}

int dsv4kv_fake_quant(int layout, const void* in_bf16, long long n, long long in_stride,
                      void* out_bf16, void* stream) {
  int st = check_rw_layout(layout);
  if (st != DSV4KV_OK) return st;
  if (n < 0 || in_stride < 0) return DSV4KV_EINVAL;
  if (n == 0) return DSV4KV_OK;
  if (!in_bf16 || !out_bf16 || !aligned16(in_bf16) || !aligned16(out_bf16)) return DSV4KV_EINVAL;
  if (in_stride < DSV4KV_DIM || (in_stride % 8) != 0) return DSV4KV_EINVAL;
  return cuda_status(launch_fake_quant(layout, static_cast<const __nv_bfloat16*>(in_bf16), n,
                                       in_stride, static_cast<__nv_bfloat16*>(out_bf16),
                                       static_cast<cudaStream_t>(stream)));
}

int dsv4kv_selftest_bounded_wait(int polls, int* err_word, int* gave_up, void* stream) {
  if (polls < 1 || polls > (1 << 24)) return DSV4KV_ERANGE;
  if (!err_word || !gave_up || ((uintptr_t)err_word & 3u) || ((uintptr_t)gave_up & 3u))
    return DSV4KV_EINVAL;
  return cuda_status(launch_bounded_wait_selftest((uint32_t)polls, err_word, gave_up,
                                                  static_cast<cudaStream_t>(stream)));
}

int dsv4kv_selftest_fp4_quotient(const float* x, const unsigned char* scale_codes, long long n,
                                 float* q_fast, float* q_ieee, void* stream) {
  if (n < 0) return DSV4KV_EINVAL;
  if (n == 0) return DSV4KV_OK;
  if (!x || !scale_codes || !q_fast || !q_ieee || ((uintptr_t)x & 3u) ||
      ((uintptr_t)q_fast & 3u) || ((uintptr_t)q_ieee & 3u))
    return DSV4KV_EINVAL;
  return cuda_status(launch_fp4_quotient_selftest(x, scale_codes, n, q_fast, q_ieee,
                                                  static_cast<cudaStream_t>(stream)));
}

int dsv4kv_selftest_e4m3_recip(const unsigned char* codes, long long n, float* y_fast,
                               float* y_ieee, void* stream) {
  if (n < 0) return DSV4KV_EINVAL;
  if (n == 0) return DSV4KV_OK;
  if (!codes || !y_fast || !y_ieee || ((uintptr_t)y_fast & 3u) || ((uintptr_t)y_ieee & 3u))
    return DSV4KV_EINVAL;
  return cuda_status(launch_e4m3_recip_selftest(codes, n, y_fast, y_ieee,
                                                static_cast<cudaStream_t>(stream)));
}

// ----------------------------------------------------------------- reuse
}  // extern "C"

namespace {

// What the reuse buffer's storage holds: the gathered source, and for the
// top-k and short-context forms the id mapping, every field kept as given.
struct KvbufKey {
  int form;
  int layout;
  const void* pool;
  long long pool_rows;
  const int* ids;
  long long n;
  int k;
  const int* token_to_req;
  const unsigned char* is_valid;
  const int* page_table;
  int n_req, max_pages, page_bits;
};

KvbufKey ids_key(int layout, const void* pool, long long pool_rows, const int* ids, long long n) {
  return KvbufKey{DSV4KV_KVBUF_IDS, layout, pool, pool_rows, ids, n, 0, nullptr, nullptr, nullptr,
                  0, 0, 0};
}

KvbufKey mapped_key(int form, int layout, const void* pool, long long pool_rows, const int* ids,
                    int n_tok, int k, const int* token_to_req, const unsigned char* is_valid,
                    const int* page_table, int n_req, int max_pages, int page_bits) {
  return KvbufKey{form,         layout,   pool,       pool_rows, ids,       (long long)n_tok * k,
                  k,            token_to_req, is_valid, page_table, n_req, max_pages, page_bits};
}

void kvbuf_clear(dsv4kv_kvbuf* buf) {
  buf->head_valid = 0;
  buf->head_form = DSV4KV_KVBUF_IDS;
  buf->head_layout = -1;
  buf->head_pool = nullptr;
  buf->head_pool_rows = 0;
  buf->head_ids = nullptr;
  buf->head_n = 0;
  buf->head_k = 0;
  buf->head_token_to_req = nullptr;
  buf->head_is_valid = nullptr;
  buf->head_page_table = nullptr;
  buf->head_n_req = 0;
  buf->head_max_pages = 0;
  buf->head_page_bits = 0;
}

// The head decision: a hit when every field equals the head's; on a miss the
// key becomes the head.
int kvbuf_lookup_key(dsv4kv_kvbuf* buf, const KvbufKey& q, int* hit) {
  if (!buf || !hit || q.n < 0) return DSV4KV_EINVAL;
  if (q.n > buf->capacity_rows) return DSV4KV_ERANGE;
  const bool same = buf->head_valid && buf->head_form == q.form &&
                    buf->head_layout == q.layout && buf->head_pool == q.pool &&
                    buf->head_pool_rows == q.pool_rows && buf->head_ids == q.ids &&
                    buf->head_n == q.n && buf->head_k == q.k &&
                    buf->head_token_to_req == q.token_to_req &&
                    buf->head_is_valid == q.is_valid && buf->head_page_table == q.page_table &&
                    buf->head_n_req == q.n_req && buf->head_max_pages == q.max_pages &&
                    buf->head_page_bits == q.page_bits;
  if (same) {
    *hit = 1;
    return DSV4KV_OK;
  }
  *hit = 0;
  buf->head_valid = 1;
  buf->head_form = q.form;
  buf->head_layout = q.layout;
  buf->head_pool = q.pool;
  buf->head_pool_rows = q.pool_rows;
  buf->head_ids = q.ids;
  buf->head_n = q.n;
  buf->head_k = q.k;
  buf->head_token_to_req = q.token_to_req;
  buf->head_is_valid = q.is_valid;
  buf->head_page_table = q.page_table;
  buf->head_n_req = q.n_req;
  buf->head_max_pages = q.max_pages;
  buf->head_page_bits = q.page_bits;
  return DSV4KV_OK;
}

}  // namespace

extern "C" {

int dsv4kv_kvbuf_init(dsv4kv_kvbuf* buf, void* storage_bf16, long long capacity_rows) {
  if (!buf || capacity_rows < 0) return DSV4KV_EINVAL;
  if (capacity_rows > 0 && (!storage_bf16 || !aligned16(storage_bf16))) return DSV4KV_EINVAL;
  buf->storage = storage_bf16;
  buf->capacity_rows = capacity_rows;
  kvbuf_clear(buf);
  return DSV4KV_OK;
}

void dsv4kv_kvbuf_begin_forward(dsv4kv_kvbuf* buf) {
  if (buf) buf->head_valid = 0;
}

int dsv4kv_kvbuf_get(dsv4kv_kvbuf* buf, long long n, void** rows) {
  if (!buf || n < 0) return DSV4KV_EINVAL;
  if (n > buf->capacity_rows) return DSV4KV_ERANGE;
  buf->head_valid = 0;
  if (rows) *rows = buf->storage;
  return DSV4KV_OK;
}

int dsv4kv_kvbuf_lookup(dsv4kv_kvbuf* buf, int layout, const void* pool, long long pool_rows,
                        const int* ids, long long n, int* hit) {
  return kvbuf_lookup_key(buf, ids_key(layout, pool, pool_rows, ids, n), hit);
}

int dsv4kv_kvbuf_get_with_head(dsv4kv_kvbuf* buf, int layout, const void* pool,
                               long long pool_rows, const int* ids, long long n, void** rows,
                               int* hit, int* err_word, void* stream) {
  if (!buf || !hit) return DSV4KV_EINVAL;
  int st = check_gather(layout, pool, pool_rows, ids, n, buf->storage);
  if (st != DSV4KV_OK) return st;
  st = dsv4kv_kvbuf_lookup(buf, layout, pool, pool_rows, ids, n, hit);
  if (st != DSV4KV_OK) return st;
  if (rows) *rows = buf->storage;
  if (*hit || n == 0) return DSV4KV_OK;
  st = dsv4kv_dequant_gather(layout, pool, pool_rows, ids, n, buf->storage, err_word, stream);
  if (st != DSV4KV_OK) buf->head_valid = 0;
  return st;
}

int dsv4kv_kvbuf_get_with_head_all(dsv4kv_kvbuf* buf, int layout, const void* pool,
                                   long long pool_rows, const int* lens_in, int n_tok, int k,
                                   const int* token_to_req, const unsigned char* is_valid,
                                   const int* page_table, int n_req, int max_pages, int page_bits,
                                   void** rows, int* lens, int* hit, int* err_word, void* stream) {
  if (!buf || !hit) return DSV4KV_EINVAL;
  int st = check_topk(lens_in, n_tok, k, token_to_req, page_table, n_req, max_pages, page_bits);
  if (st != DSV4KV_OK) return st;
  const long long n = (long long)n_tok * k;
  st = check_gather(layout, pool, pool_rows, lens_in, n, buf->storage);
  if (st != DSV4KV_OK) return st;
  st = kvbuf_lookup_key(buf,
                        mapped_key(DSV4KV_KVBUF_ALL, layout, pool, pool_rows, lens_in, n_tok, k,
                                   token_to_req, is_valid, page_table, n_req, max_pages, page_bits),
                        hit);
  if (st != DSV4KV_OK) return st;
  if (rows) *rows = buf->storage;
  if (*hit || n == 0) return DSV4KV_OK;
  st = dsv4kv_dequant_gather_all(layout, pool, pool_rows, lens_in, n_tok, k, token_to_req,
                                 is_valid, page_table, n_req, max_pages, page_bits, buf->storage,
                                 lens, err_word, stream);
  if (st != DSV4KV_OK) buf->head_valid = 0;
  return st;
}

int dsv4kv_kvbuf_get_with_head_topk(dsv4kv_kvbuf* buf, int layout, const void* pool,
                                    long long pool_rows, const int* topk, int n_tok, int k,
                                    const int* token_to_req, const unsigned char* is_valid,
                                    const int* page_table, int n_req, int max_pages, int page_bits,
                                    void** rows, int* lens, int* hit, int* err_word, void* stream) {
  if (!buf || !hit) return DSV4KV_EINVAL;
  int st = check_topk(topk, n_tok, k, token_to_req, page_table, n_req, max_pages, page_bits);
  if (st != DSV4KV_OK) return st;
  const long long n = (long long)n_tok * k;
  st = check_gather(layout, pool, pool_rows, topk, n, buf->storage);
  if (st != DSV4KV_OK) return st;
  st = kvbuf_lookup_key(buf,
                        mapped_key(DSV4KV_KVBUF_TOPK, layout, pool, pool_rows, topk, n_tok, k,
                                   token_to_req, is_valid, page_table, n_req, max_pages, page_bits),
                        hit);
  if (st != DSV4KV_OK) return st;
  if (rows) *rows = buf->storage;
  if (*hit || n == 0) return DSV4KV_OK;
  st = dsv4kv_dequant_gather_topk(layout, pool, pool_rows, topk, n_tok, k, token_to_req, is_valid,
                                  page_table, n_req, max_pages, page_bits, buf->storage, lens,
                                  err_word, stream);
  if (st != DSV4KV_OK) buf->head_valid = 0;
  return st;
}

}  // extern "C"
