// Decode / speculative-verify steps of the ratio-2 compressor: one launch
// for a step of a few new tokens per request that makes at most 16
// compressed rows per SM.
//
// sglang PR #39652 "dsv4.1: compression, KV I/O, and metadata kernels",
// Summary (c1/c2 bullet) and the review of the c2 kernel: the ratio-2 decode
// compressor keeps a pair-state ring, completes a pair at an odd position and
// rotates it with the RoPE frequencies of pos - 1; sglang PR #46230: the
// offsets are read on the device, so the launch can sit in a CUDA graph whose
// metadata is refreshed in place.
//
// Such a step is latency-bound (a few MB, L2-resident), so the launch is
// shaped for latency: no row waits for a plan of the whole step before its
// loads and its arithmetic.  The request slots are cut into G chunks of
// S <= 32 consecutive slots, one per CTA (G = one CTA per SM, and at least
// n_out / 16), and each CTA has 20 warps:
//  * 16 row warps.  Together they first copy every slot's new-token count and
//    start position into shared memory with the slot's rows (8 slots per
//    thread); warp 0 also reads its chunk's slots (lane l: slot S * b + l)
//    and scans their rows.  Row warp w then takes the chunk's local row w,
//    finds its slot by a ballot, issues every load of the row (the ring
//    entry for a pair whose first token precedes the step, the new token's
//    kv | score, the RoPE row, the page-table entry) and does the row's
//    arithmetic.  Only its writes wait for the scan, which gives the row its
//    output index chunk_base[b] + w (rows at or past n_out are not written).
//  * 3 scan warps: the rows of every chunk, from the counts in shared
//    memory, and their prefix chunk_base, which numbers the rows request by
//    request.
//  * the ring warp: this chunk's ring tokens, staged in shared memory by bulk
//    copies.
// A chunk with more than 16 rows has overflow rows; after the scan they are
// numbered across chunks and taken, in order, by the spare row warps (a CTA
// whose chunk has t < 16 rows below n_out has 16 - t), which exist whenever
// n_out <= 16 G.
//
// The ring.  Each even-position new token among the last 2R positions of a
// request goes to entry (q / 2) % R.  A row reads a ring entry only at a
// request's first row with an odd start, and an update can write that same
// entry only when the step has n >= 2R tokens; such a request's update is
// done by the warp that computes that first row, after the row (program
// order), or by scan warp 0 when the row falls at or past n_out.  The ring
// warp does every other update; none of them touches an entry that a row of
// the launch reads, so no order between CTAs is needed.
#include <atomic>
#include <cstddef>

#include "compress_row.cuh"
#include "internal.cuh"
#include "launchers.cuh"
#include "tma.cuh"

namespace dsv4kv {

constexpr int kDecRows = kDecodeRowsPerCta;                // row warps
constexpr int kDecAuxWarps = 4;                            // 3 scan warps and the ring warp
constexpr int kDecScanWarps = 3;
constexpr int kDecWarps = kDecRows + kDecAuxWarps;
constexpr int kDecThreads = kDecWarps * 32;
constexpr int kDecScanThreads = kDecScanWarps * 32;
constexpr int kDecSlotsPerRowThread = kMaxSlots / (kDecRows * 32);   // 8
constexpr int kDecChunksPerLane = kDecodeMaxGrid / 32;
constexpr int kDecStages = 32;                             // ring tokens in shared memory
constexpr uint32_t kDecTokBytes = 2 * kDim * sizeof(__nv_bfloat16);   // kv | score
constexpr int kBarRows = 1, kBarAux = 2, kBarData = 3;     // named barriers
static_assert(kDecodeMaxChunk == 32, "one chunk slot per lane of warp 0");
static_assert(kDecSlotsPerRowThread == 8 && kDecodeMaxGrid % 32 == 0, "scan shapes");

struct DecodeShared {
  uint4 norm_w[64];                      // the RMSNorm weight row, bf16 [512]
  uint64_t scan_bar;                     // the scan's results are published
  uint64_t ring_bar;                     // the ring tokens' bulk copies
  int abort;                             // a bounded wait gave up
  unsigned t_loc;                        // rows of this chunk (saturated at n_out)
  int m_first[kDecodeMaxChunk], m_count[kDecodeMaxChunk], m_start[kDecodeMaxChunk];
  unsigned m_off[kDecodeMaxChunk], m_n[kDecodeMaxChunk];   // this chunk's local rows per slot
  unsigned chunk_tot[kDecodeMaxGrid];    // rows per chunk (each slot's rows capped at n_out)
  unsigned chunk_base[kDecodeMaxGrid + 1];   // their prefix, saturated at n_out
};
static_assert(kDecodeMaxGrid * kDecodeRowsPerCta <= 65535, "a slot's capped rows fit 16 bits");

// Dynamic shared memory: every slot's new-token count, start position and
// rows (capped at n_out), written by the row warps, and the ring stages.
struct DecodeSmem {
  int* count;
  int* start;
  uint16_t* rows;
  uint8_t* stage;
};
constexpr size_t kDecArrayBytes = sizeof(int) * (size_t)kMaxSlots;
constexpr size_t kDecRowsBytes = sizeof(uint16_t) * (size_t)kMaxSlots;
constexpr size_t kDecSmemBytes =
    2 * kDecArrayBytes + kDecRowsBytes + (size_t)kDecStages * kDecTokBytes;

__device__ __forceinline__ unsigned sat_add(unsigned a, unsigned b, unsigned cap) {
  const unsigned s = a + b;    // a, b <= cap < 2^31: no wrap
  return s < cap ? s : cap;
}

// rows_of_slot<2> capped at cap, in 32 bits: for n > 0,
// floor((p0 + n) / 2) - floor(p0 / 2) = floor((n + (p0 & 1)) / 2) for every
// int p0 (odd p0, negative ones included, completes one pair more).
__device__ __forceinline__ unsigned capped_rows(int n, int p0, unsigned cap) {
  if (n <= 0) return 0u;
  const unsigned r = ((unsigned)n + ((unsigned)p0 & 1u)) >> 1;
  return r < cap ? r : cap;
}

__device__ __forceinline__ bool aligned16(const void* q) {
  return (reinterpret_cast<uintptr_t>(q) & 15) == 0;
}

// Descriptor of row j of request slot r (ratio 2 with start positions):
// compressed index c = p0 / 2 + j at position 2c; the pair's first token is
// in the ring when 2c < p0.  The state rules are plan_row's.
template <bool ROPE>
__device__ __forceinline__ RowDesc decode_row_desc(const StoreParams& p, int r, long long j,
                                                   int first, int p0, long long& src) {
  RowDesc d;
  const long long c = ((long long)p0 >> 1) + j;
  const long long pos = 2 * c;
  d.r = r;
  d.c = (int)c;
  d.pos = (int)pos;
  src = (long long)first + (pos - p0);
  if (pos < p0) {
    const bool ok = p.ring != nullptr && first >= 0 && (long long)first + 1 <= p.n_rows &&
                    pos >= 0 && (!ROPE || pos < p.max_pos);
    d.state = ok ? kRowOkRing : kRowBad;
  } else {
    const bool ok = src >= 0 && src + 2 <= p.n_rows && pos >= 0 && (!ROPE || pos < p.max_pos);
    d.state = ok ? kRowOk : kRowBad;
  }
  return d;
}

// The ring tokens of a request: the even positions q, q + 2, ... among the
// step's last 2R positions, from source rows src, src + 2, ...
__device__ __forceinline__ int ring_tokens(int n, long long p0, int first, int R, long long& q,
                                           long long& src) {
  q = 0;
  src = 0;
  if (n <= 0) return 0;
  long long lo = p0 + n - 2LL * R;
  if (lo < p0) lo = p0;
  lo += lo & 1;                                   // the first even position
  if (p0 + n <= lo) return 0;
  q = lo;
  src = (long long)first + (lo - p0);
  return (int)((p0 + n - lo + 1) >> 1);           // <= R
}

// A request whose ring update may rewrite the entry its first row reads
// (odd start, n >= 2R): the update follows that row.
__device__ __forceinline__ bool ring_follows_row(const StoreParams& p, int n, int p0) {
  return p.ring != nullptr && (p0 & 1) && n >= 2 * p.ring_size;
}

__device__ __forceinline__ bool ring_token_ok(const StoreParams& p, long long q, long long row) {
  return q >= 0 && row >= 0 && row < p.n_rows;
}

// Copies one request's ring tokens per lane through registers (the warp
// moves 2 KB kv | score rows from the input rows to ring entries, 3 at a
// time); a token at a negative position or past the rows is a fault.  Used
// where the update must follow a row in program order.
__device__ __forceinline__ void copy_ring_tokens(const StoreParams& p, long long q0, long long src0,
                                                 int r, int ntok, int lane) {
  constexpr int kCopies = 3;
  const int R = p.ring_size;
  const __nv_bfloat16* score_base = p.score ? p.score : p.rows + kDim;
  const long long sstride = p.score ? p.score_stride : p.row_stride;
  const int max_tok = __reduce_max_sync(kFullMask, (unsigned)ntok);
  for (int t = 0; t < max_tok; ++t) {
    const long long qt = q0 + 2LL * t, row = src0 + 2LL * t;
    const bool has = t < ntok;
    const bool bad = has && !ring_token_ok(p, qt, row);
    const unsigned n_bad = __popc(__ballot_sync(kFullMask, bad));
    if (lane == 0 && n_bad && p.err) atomicAdd(p.err, (int)n_bad);
    unsigned todo = __ballot_sync(kFullMask, has && !bad);
    const long long dst =
        has && !bad ? ((long long)r * R + (unsigned)(qt >> 1) % (unsigned)R) * (2 * kDim) : 0;
    while (todo) {
      long long rows_[kCopies], dsts_[kCopies];
      bool use[kCopies];
#pragma unroll
      for (int c = 0; c < kCopies; ++c) {
        use[c] = todo != 0;
        const int l = use[c] ? __ffs(todo) - 1 : 0;
        if (use[c]) todo &= todo - 1;
        rows_[c] = __shfl_sync(kFullMask, row, l);
        dsts_[c] = __shfl_sync(kFullMask, dst, l);
      }
      uint4 v[kCopies][4];
#pragma unroll
      for (int c = 0; c < kCopies; ++c) {
        if (!use[c]) continue;
        const uint8_t* kv = reinterpret_cast<const uint8_t*>(p.rows + rows_[c] * p.row_stride);
        const uint8_t* sc = reinterpret_cast<const uint8_t*>(score_base + rows_[c] * sstride);
        v[c][0] = ld_stream_v4(kv + 16 * lane);
        v[c][1] = ld_stream_v4(kv + 512 + 16 * lane);
        v[c][2] = ld_stream_v4(sc + 16 * lane);
        v[c][3] = ld_stream_v4(sc + 512 + 16 * lane);
      }
#pragma unroll
      for (int c = 0; c < kCopies; ++c) {
        if (!use[c]) continue;
        uint4* e = reinterpret_cast<uint4*>(p.ring + dsts_[c]);
        e[lane] = v[c][0];
        e[32 + lane] = v[c][1];
        e[64 + lane] = v[c][2];
        e[96 + lane] = v[c][3];
      }
    }
  }
}

// ---- ring tokens of the chunk through shared memory (the ring warp) -----
// Lane l holds slot S * b + l's tokens (none when its update follows its
// first row); the chunk's tokens are numbered lane by lane from g0 and move
// in batches of kDecStages: bulk loads into the stages, then bulk stores to
// the ring entries.
struct RingLane {
  long long q, src;
  int r, ntok, g0, total;
};

__device__ __forceinline__ RingLane ring_lane(const StoreParams& p, int r, bool in, int first,
                                              int n, int p0, int lane) {
  RingLane rl{0, 0, r, 0, 0, 0};
  if (in && !ring_follows_row(p, n, p0))
    rl.ntok = ring_tokens(n, p0, first, p.ring_size, rl.q, rl.src);
  int incl = rl.ntok;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(kFullMask, incl, o);
    if (lane >= o) incl += t;
  }
  rl.g0 = incl - rl.ntok;
  rl.total = __shfl_sync(kFullMask, incl, 31);
  int bad = 0;
  for (int t = 0; t < rl.ntok; ++t) bad += !ring_token_ok(p, rl.q + 2LL * t, rl.src + 2LL * t);
  bad = (int)__reduce_add_sync(kFullMask, (unsigned)bad);
  if (lane == 0 && bad && p.err) atomicAdd(p.err, bad);
  return rl;
}

// Issues batch m's bulk loads; false when the batch copies nothing.
__device__ __forceinline__ bool ring_issue(const StoreParams& p, DecodeShared& sh,
                                           const DecodeSmem& ds, const RingLane& rl, int m,
                                           int lane) {
  const int t0 = max(0, m * kDecStages - rl.g0), t1 = min(rl.ntok, (m + 1) * kDecStages - rl.g0);
  int good = 0;
  for (int t = t0; t < t1; ++t) good += ring_token_ok(p, rl.q + 2LL * t, rl.src + 2LL * t);
  const unsigned tot = __reduce_add_sync(kFullMask, (unsigned)good);
  if (tot == 0) return false;
  if (lane == 0) mbar_arrive_expect_tx(&sh.ring_bar, tot * kDecTokBytes);
  __syncwarp();
  const uint64_t pol = policy_evict_first();
  for (int t = t0; t < t1; ++t) {
    const long long row = rl.src + 2LL * t;
    if (!ring_token_ok(p, rl.q + 2LL * t, row)) continue;
    uint8_t* st = ds.stage + (size_t)(rl.g0 + t - m * kDecStages) * kDecTokBytes;
    const __nv_bfloat16* kv = p.rows + row * p.row_stride;
    if (p.score == nullptr) {
      bulk_g2s(st, kv, kDecTokBytes, &sh.ring_bar, pol);            // kv | score adjacent
    } else {
      bulk_g2s(st, kv, kDecTokBytes / 2, &sh.ring_bar, pol);
      bulk_g2s(st + kDecTokBytes / 2, p.score + row * p.score_stride, kDecTokBytes / 2,
               &sh.ring_bar, pol);
    }
  }
  return true;
}

// Waits for batch m's loads (the barrier's phase-th completed phase) and
// stores it to the ring entries.
__device__ __forceinline__ void ring_store(const StoreParams& p, DecodeShared& sh,
                                           const DecodeSmem& ds, const RingLane& rl, int m,
                                           int phase, int lane) {
  if (!mbar_wait(&sh.ring_bar, (uint32_t)(phase & 1), &sh.abort, p.err)) return;
  const int t0 = max(0, m * kDecStages - rl.g0), t1 = min(rl.ntok, (m + 1) * kDecStages - rl.g0);
  const int R = p.ring_size;
  for (int t = t0; t < t1; ++t) {
    const long long qt = rl.q + 2LL * t;
    if (!ring_token_ok(p, qt, rl.src + 2LL * t)) continue;
    const long long e = (long long)rl.r * R + (unsigned)(qt >> 1) % (unsigned)R;
    bulk_s2g(p.ring + e * (2 * kDim),
             ds.stage + (size_t)(rl.g0 + t - m * kDecStages) * kDecTokBytes, kDecTokBytes);
  }
  bulk_commit();
  bulk_wait_read();
  __syncwarp();
}

// ---- scan warps ----------------------------------------------------------
// The row warps store every slot's count, start position and rows (capped at
// n_out) in shared memory first; the scan warps then sum the rows of every
// chunk and take their prefix.  Scan warp 0 also does the ring updates that
// follow a first row at or past n_out.
__device__ __forceinline__ void scan_warps(const StoreParams& p, DecodeShared& sh,
                                           const DecodeSmem& ds, int at, int S, unsigned cap) {
  const int n = p.n_slots, G = (int)gridDim.x, b = (int)blockIdx.x;
  const int lane = at & 31, aw = at >> 5;
  bar_sync(kBarData, (kDecRows + kDecScanWarps) * 32);
  // rows per chunk: thread t sums chunks t, t + 96, ...
  for (int c = at; c < G; c += kDecScanThreads) {
    unsigned sum = 0;
    const int s0 = S * c, e = min(s0 + S, n);
#pragma unroll
    for (int u = 0; u < kDecodeMaxChunk; ++u)
      if (s0 + u < e) sum += ds.rows[s0 + u];
    sh.chunk_tot[c] = sum;
  }
  bar_sync(kBarAux, kDecScanThreads);
  // chunk c's first output row: the prefix of the chunk totals (each below
  // 4096 * n_out < 2^32), saturated at n_out; lane l: chunks [8l, 8l + 8)
  if (aw == 0) {
    unsigned v[kDecChunksPerLane], sum = 0;
#pragma unroll
    for (int i = 0; i < kDecChunksPerLane; ++i) {
      const int c = kDecChunksPerLane * lane + i;
      v[i] = c < G ? sh.chunk_tot[c] : 0u;
      sum += v[i];
    }
    unsigned incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned t = __shfl_up_sync(kFullMask, incl, o);
      if (lane >= o) incl += t;
    }
    unsigned run = incl - sum;
#pragma unroll
    for (int i = 0; i < kDecChunksPerLane; ++i) {
      const int c = kDecChunksPerLane * lane + i;
      if (c <= G) sh.chunk_base[c] = run < cap ? run : cap;
      run += v[i];
    }
    if (lane == 31 && G == kDecodeMaxGrid) sh.chunk_base[G] = run < cap ? run : cap;
  }
  bar_sync(kBarAux, kDecScanThreads);              // chunk_base complete for every scan warp
  if (at == 0) mbar_arrive(&sh.scan_bar);        // releases the row warps

  // the debug outputs' padding rows (output rows from the step's total up
  // to n_out), spread over the CTAs
  const unsigned total = sh.chunk_base[G];
  if (p.latent_out || p.prequant_out) {
    for (long long k = (long long)total + b + (long long)G * aw; k < p.n_out;
         k += (long long)G * kDecScanWarps)
      zero_row_outputs(p, k, lane);
  }
  if (aw == 0 && p.ring != nullptr && !*reinterpret_cast<volatile int*>(&sh.abort)) {
    // ring updates that follow a first row which falls at or past n_out: no
    // row reads their entry, so this chunk's CTA does them
    const int r = b * S + lane;
    const bool in = lane < S && r < n;
    const int nc = in ? ds.count[r] : 0, p0 = in ? ds.start[r] : 0;
    const unsigned rows = capped_rows(nc, p0, cap);
    unsigned incl = rows;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned t = __shfl_up_sync(kFullMask, incl, o);
      if (lane >= o) incl = sat_add(incl, t, cap);
    }
    const unsigned excl = __shfl_up_sync(kFullMask, incl, 1);
    const unsigned k0 = sat_add(sh.chunk_base[b], lane == 0 ? 0u : excl, cap);
    long long q = 0, src = 0;
    int ntok = 0;
    if (in && ring_follows_row(p, nc, p0) && k0 >= cap)
      ntok = ring_tokens(nc, p0, __ldg(p.ext + r), p.ring_size, q, src);
    copy_ring_tokens(p, q, src, r, ntok, lane);
  }
}

// ---- the ring warp: this chunk's ring tokens (lane l: slot S * b + l),
// batch by batch through the stages; it waits for nothing else in the CTA
__device__ __forceinline__ void ring_warp(const StoreParams& p, DecodeShared& sh,
                                         const DecodeSmem& ds, int S, int lane) {
  const int r = (int)blockIdx.x * S + lane;
  const bool in = lane < S && r < p.n_slots;
  int f = 0, c = 0, s = 0;
  if (in) {
    f = __ldg(p.ext + r);
    c = __ldg(p.ext + p.n_slots + r);
    s = p.start_pos ? __ldg(p.start_pos + r) : 0;
  }
  const RingLane rl = ring_lane(p, r, in, f, c, s, lane);
  int phase = 0;
  for (int m = 0; m * kDecStages < rl.total; ++m)
    if (ring_issue(p, sh, ds, rl, m, lane)) ring_store(p, sh, ds, rl, m, phase++, lane);
}

// ---- overflow rows ---------------------------------------------------------
// A chunk's local rows past the first 16 are its overflow rows; they are
// numbered chunk by chunk and taken, in that order, by the spare row warps
// (warps past their chunk's rows below n_out), numbered CTA by CTA.  With
// n_out <= 16 G there are always enough.

// The slot holding local row i_loc of chunk cs (lanes: its slots): fills r
// and the row's index j in its slot; false if none (not reached for a local
// row below the chunk's total).
__device__ __forceinline__ bool chunk_row_slot(const StoreParams& p, const DecodeSmem& ds, int cs,
                                               unsigned i_loc, int S, unsigned cap, int lane,
                                               int& r, long long& j) {
  const int rs = cs * S + lane;
  const bool in = lane < S && rs < p.n_slots;
  const unsigned nr = in ? ds.rows[rs] : 0u;
  unsigned incl = nr;
#pragma unroll
  for (int q = 1; q < 32; q <<= 1) {
    const unsigned t = __shfl_up_sync(kFullMask, incl, q);
    if (lane >= q) incl = sat_add(incl, t, cap);
  }
  const unsigned excl = __shfl_up_sync(kFullMask, incl, 1);
  const unsigned off = lane == 0 ? 0u : excl;
  const int l = __ffs(__ballot_sync(kFullMask, nr > 0 && off <= i_loc && i_loc < off + nr)) - 1;
  if (l < 0) return false;
  r = cs * S + l;
  j = (long long)i_loc - __shfl_sync(kFullMask, off, l);
  return true;
}

// After the scan: the overflow row that spare warp `spare` of this CTA
// takes, or false.  Lane l holds chunks [8l, 8l + 8).  Fills the row's slot,
// its index in the slot and its output row.
__device__ __forceinline__ bool overflow_row(const StoreParams& p, const DecodeShared& sh,
                                             const DecodeSmem& ds, int spare, int S, unsigned cap,
                                             int lane, int& r, long long& j, long long& k) {
  const int G = (int)gridDim.x, b = (int)blockIdx.x;
  unsigned ov_sum = 0, sp_sum = 0, sp_b = 0;
#pragma unroll
  for (int i = 0; i < kDecChunksPerLane; ++i) {
    const int c = kDecChunksPerLane * lane + i;
    const unsigned t = c < G ? sh.chunk_base[c + 1] - sh.chunk_base[c] : (unsigned)kDecRows;
    if (c == b) sp_b = sp_sum;
    ov_sum += t > (unsigned)kDecRows ? t - kDecRows : 0u;
    sp_sum += t < (unsigned)kDecRows ? kDecRows - t : 0u;
  }
  unsigned ov_incl = ov_sum, sp_incl = sp_sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned a = __shfl_up_sync(kFullMask, ov_incl, o);
    const unsigned c = __shfl_up_sync(kFullMask, sp_incl, o);
    if (lane >= o) { ov_incl += a; sp_incl += c; }
  }
  const unsigned ov_tot = __shfl_sync(kFullMask, ov_incl, 31);
  const unsigned o = __shfl_sync(kFullMask, sp_incl - sp_sum + sp_b, b / kDecChunksPerLane) +
                     (unsigned)spare;
  if (o >= ov_tot) return false;
  const unsigned ov_ex = ov_incl - ov_sum;
  const int owner = __ffs(__ballot_sync(kFullMask, ov_ex <= o && o < ov_incl)) - 1;
  int cs = 0;
  unsigned idx = 0;
  if (lane == owner) {
    unsigned acc = ov_ex;
#pragma unroll
    for (int i = 0; i < kDecChunksPerLane; ++i) {
      const int c = kDecChunksPerLane * lane + i;
      const unsigned t = c < G ? sh.chunk_base[c + 1] - sh.chunk_base[c] : 0u;
      const unsigned ovc = t > (unsigned)kDecRows ? t - kDecRows : 0u;
      if (o >= acc && o < acc + ovc) { cs = c; idx = o - acc; }
      acc += ovc;
    }
  }
  cs = __shfl_sync(kFullMask, cs, owner);
  const unsigned i_loc = kDecRows + __shfl_sync(kFullMask, idx, owner);
  k = (long long)sh.chunk_base[cs] + i_loc;
  return chunk_row_slot(p, ds, cs, i_loc, S, cap, lane, r, j);
}

template <int L, bool NORM, bool ROPE>
__global__ void __launch_bounds__(kDecThreads, 1)
compress_decode_kernel(const StoreParams p) {
  __shared__ DecodeShared sh;
  extern __shared__ __align__(128) uint8_t dsm[];
  const DecodeSmem ds{reinterpret_cast<int*>(dsm), reinterpret_cast<int*>(dsm) + kMaxSlots,
                      reinterpret_cast<uint16_t*>(dsm + 2 * kDecArrayBytes),
                      dsm + 2 * kDecArrayBytes + kDecRowsBytes};
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = (int)gridDim.x, b = (int)blockIdx.x, n = p.n_slots;
  const int S = (n + G - 1) / G;                  // slots per chunk, <= 32
  const unsigned cap = (unsigned)p.n_out;         // >= 1
  if (tid == 0) {
    mbar_init(&sh.scan_bar, 1);
    mbar_init(&sh.ring_bar, 1);
    sh.abort = 0;
    mbar_fence_init();
  }
  __syncthreads();
  grid_dependency_wait();
  if (warp == kDecRows + kDecScanWarps) {
    if (p.ring != nullptr) ring_warp(p, sh, ds, S, lane);
    allow_dependent_launch();
    return;
  }
  if (warp >= kDecRows) {
    scan_warps(p, sh, ds, tid - kDecRows * 32, S, cap);
    allow_dependent_launch();
    return;
  }

  // ---- row warps: every slot's count, start and rows into shared memory
  // (thread t: slots [8t, 8t + 8)); warp 0 also reads its chunk's slots
  // (lane l: slot S * b + l) and the RMSNorm weights
  {
    int f = 0, c = 0, st = 0;
    const int r = b * S + lane;
    const bool in = warp == 0 && lane < S && r < n;
    if (in) {
      f = __ldg(p.ext + r);
      c = __ldg(p.ext + n + r);
      st = p.start_pos ? __ldg(p.start_pos + r) : 0;
    }
    const int s0 = kDecSlotsPerRowThread * tid;
    int4 c4[2] = {make_int4(0, 0, 0, 0), make_int4(0, 0, 0, 0)}, t4[2] = {c4[0], c4[0]};
    if ((n & 3) == 0 && aligned16(p.ext) && (p.start_pos == nullptr || aligned16(p.start_pos)) &&
        s0 + kDecSlotsPerRowThread <= n) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        c4[h] = __ldg(reinterpret_cast<const int4*>(p.ext + n + s0) + h);
        if (p.start_pos) t4[h] = __ldg(reinterpret_cast<const int4*>(p.start_pos + s0) + h);
      }
    } else if (s0 < n) {
#pragma unroll
      for (int e = 0; e < kDecSlotsPerRowThread; ++e) {
        if (s0 + e < n) {
          (&c4[e >> 2].x)[e & 3] = __ldg(p.ext + n + s0 + e);
          if (p.start_pos) (&t4[e >> 2].x)[e & 3] = __ldg(p.start_pos + s0 + e);
        }
      }
    }
    if (NORM && warp == 0) {
      sh.norm_w[lane] = __ldg(reinterpret_cast<const uint4*>(p.norm_w) + lane);
      sh.norm_w[32 + lane] = __ldg(reinterpret_cast<const uint4*>(p.norm_w) + 32 + lane);
    }
    unsigned rw[kDecSlotsPerRowThread];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      reinterpret_cast<int4*>(ds.count + s0)[h] = c4[h];
      reinterpret_cast<int4*>(ds.start + s0)[h] = t4[h];
      rw[4 * h] = capped_rows(c4[h].x, t4[h].x, cap);
      rw[4 * h + 1] = capped_rows(c4[h].y, t4[h].y, cap);
      rw[4 * h + 2] = capped_rows(c4[h].z, t4[h].z, cap);
      rw[4 * h + 3] = capped_rows(c4[h].w, t4[h].w, cap);
    }
    *reinterpret_cast<uint4*>(ds.rows + s0) =
        make_uint4(rw[0] | rw[1] << 16, rw[2] | rw[3] << 16, rw[4] | rw[5] << 16, rw[6] | rw[7] << 16);
    bar_arrive(kBarData, (kDecRows + kDecScanWarps) * 32);
    if (warp == 0) {
      const unsigned nr = in ? capped_rows(c, st, cap) : 0u;
      unsigned incl = nr;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned t = __shfl_up_sync(kFullMask, incl, o);
        if (lane >= o) incl = sat_add(incl, t, cap);
      }
      const unsigned excl = __shfl_up_sync(kFullMask, incl, 1);
      sh.m_first[lane] = f;
      sh.m_count[lane] = c;
      sh.m_start[lane] = st;
      sh.m_off[lane] = lane == 0 ? 0u : excl;
      sh.m_n[lane] = nr;
      if (lane == 31) sh.t_loc = incl;
    }
  }
  bar_sync(kBarRows, kDecRows * 32);

  // ---- row warp w: local row w of the chunk.  Its loads and arithmetic run
  // before the scan is waited for (the arithmetic after it when the latent
  // is an output: that write needs the output row); a warp past the chunk's
  // rows below n_out may then take an overflow row.
  int r = -1, first = 0, p0 = 0, cnt = 0;
  long long j = 0, k = 0;
  if ((unsigned)warp < sh.t_loc) {
    const unsigned off = sh.m_off[lane], nr = sh.m_n[lane];
    const int l = __ffs(__ballot_sync(kFullMask, nr > 0 && off <= (unsigned)warp &&
                                                     (unsigned)warp < off + nr)) - 1;
    if (l >= 0) {                  // always: the offsets are exact below n_out
      r = b * S + l;
      j = warp - (long long)sh.m_off[l];
      first = sh.m_first[l];
      cnt = sh.m_count[l];
      p0 = sh.m_start[l];
    }
  }
  RowDesc d;
  d.state = kRowNone; d.pos = 0; d.r = 0; d.c = 0;
  RowIn<2, ROPE> in;
  RowMath m;
  int dest = -1;             // the page-table entry
  bool dest_ok = false, loaded = false, done_math = false, released = false;
  for (int it = 0; it < 2; ++it) {
    if (r >= 0 && !loaded) {
      loaded = true;
      long long src;
      d = decode_row_desc<ROPE>(p, r, j, first, p0, src);
      if (d.state == kRowOk || d.state == kRowOkRing) {
        const __nv_bfloat16* score_base = p.score ? p.score : p.rows + kDim;
        const long long sstride = p.score ? p.score_stride : p.row_stride;
        const long long t1 = src + 1;      // the pair's second token (a new row)
        if (d.state == kRowOkRing) {
          // token p0 - 1 from the ring: kv | score, 2 KB (plain loads: this
          // launch writes other entries of the ring)
          const uint4* e = reinterpret_cast<const uint4*>(
              p.ring + ((long long)d.r * p.ring_size + d.c % p.ring_size) * (2 * kDim));
          in.kv0[0] = e[lane];
          in.kv0[1] = e[32 + lane];
          in.s0[0] = e[64 + lane];
          in.s0[1] = e[96 + lane];
        } else {
          const uint8_t* kv = reinterpret_cast<const uint8_t*>(p.rows + src * p.row_stride);
          const uint8_t* sc = reinterpret_cast<const uint8_t*>(score_base + src * sstride);
          in.kv0[0] = ld_stream_v4(kv + 16 * lane);
          in.kv0[1] = ld_stream_v4(kv + 512 + 16 * lane);
          in.s0[0] = ld_stream_v4(sc + 16 * lane);
          in.s0[1] = ld_stream_v4(sc + 512 + 16 * lane);
        }
        const uint8_t* kv = reinterpret_cast<const uint8_t*>(p.rows + t1 * p.row_stride);
        const uint8_t* sc = reinterpret_cast<const uint8_t*>(score_base + t1 * sstride);
        in.kv1[0] = ld_stream_v4(kv + 16 * lane);
        in.kv1[1] = ld_stream_v4(kv + 512 + 16 * lane);
        in.s1[0] = ld_stream_v4(sc + 16 * lane);
        in.s1[1] = ld_stream_v4(sc + 512 + 16 * lane);
        if constexpr (ROPE) {
          if (lane >= 24) {
            const float4* f = reinterpret_cast<const float4*>(p.freqs + (long long)d.pos * kRopeDim);
            in.fr[0] = __ldg(f + 2 * (lane - 24));
            in.fr[1] = __ldg(f + 2 * (lane - 24) + 1);
          }
        }
        if (!p.out_loc) {
          const int lp = d.c >> p.page_bits;
          dest_ok = d.c >= 0 && lp < p.max_pages;
          if (dest_ok) dest = __ldg(p.page_table + (long long)d.r * p.max_pages + lp);
        }
      }
    }
    if (r >= 0 && (d.state == kRowOk || d.state == kRowOkRing) && !done_math &&
        (released || p.latent_out == nullptr)) {
      uint4 w[2] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
      if constexpr (NORM) {
        w[0] = sh.norm_w[lane];
        w[1] = sh.norm_w[32 + lane];
      }
      row_math<2, NORM, ROPE>(p, in, w, lane, m, released ? k : -1);
      done_math = true;
    }
    if (released) break;
    released = true;
    if (!mbar_wait(&sh.scan_bar, 0, &sh.abort, p.err)) { r = -1; break; }
    const unsigned cb = sh.chunk_base[b], tsat = sh.chunk_base[b + 1] - cb;
    if ((unsigned)warp < tsat) {               // a local row below n_out
      k = (long long)cb + warp;
      continue;
    }
    r = -1;
    d.state = kRowNone;
    loaded = done_math = dest_ok = false;
    const bool got = overflow_row(p, sh, ds, warp - (int)tsat, S, cap, lane, r, j, k);
    in = RowIn<2, ROPE>{};     // the dropped row's values: dead from here
    m = RowMath{};
    if (!got) break;
    first = __ldg(p.ext + r);
    cnt = ds.count[r];
    p0 = ds.start[r];
  }
  if (r >= 0) {
    if (p.out_loc && (d.state == kRowOk || d.state == kRowOkRing)) {
      dest = __ldg(p.out_loc + k);
      dest_ok = true;
    }
    if (row_computed(p, k, d.state, lane)) {
      const long long slot =
          p.out_loc ? (long long)dest
                    : (dest_ok ? ((long long)dest << p.page_bits) |
                                     (long long)(d.c & ((1 << p.page_bits) - 1))
                               : -1);
      row_store<L, NORM>(p, k, slot, m, lane);
    }
    // the update that may rewrite the entry this row read: program order in
    // this warp puts it after the row's loads
    if (j == 0 && ring_follows_row(p, cnt, p0)) {
      long long q = 0, src = 0;
      const int ntok = ring_tokens(cnt, p0, first, p.ring_size, q, src);
      copy_ring_tokens(p, q, src, r, lane == 0 ? ntok : 0, lane);
    }
  }
  allow_dependent_launch();
}

template <int L, bool NORM, bool ROPE>
static cudaError_t launch_decode_variant(const StoreParams& p, int grid, cudaStream_t s) {
  auto kern = compress_decode_kernel<L, NORM, ROPE>;
  // the slot arrays and ring stages, set once per device (published after
  // the attribute call succeeded)
  static std::atomic<int> attr_set[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 64 || !attr_set[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kDecSmemBytes);
    if (e != cudaSuccess) return e;
    if (dev < 64) attr_set[dev].store(1, std::memory_order_release);
  }
  return launch_dependent(kern, grid, kDecThreads, kDecSmemBytes, s, p);
}

template <int L>
static cudaError_t launch_decode_layout(const StoreParams& p, int grid, cudaStream_t s) {
  const bool norm = p.norm_w != nullptr, rope = p.freqs != nullptr;
  if (norm && rope) return launch_decode_variant<L, true, true>(p, grid, s);
  if (norm) return launch_decode_variant<L, true, false>(p, grid, s);
  if (rope) return launch_decode_variant<L, false, true>(p, grid, s);
  return launch_decode_variant<L, false, false>(p, grid, s);
}

int decode_grid(int n_slots, int n_out, int sms) {
  long long g = sms;
  const long long need = ((long long)n_out + kDecRows - 1) / kDecRows;
  if (g < need) g = need;
  if (g < 1 || g > kDecodeMaxGrid) return 0;
  if (((long long)n_slots + g - 1) / g > kDecodeMaxChunk) return 0;
  return (int)g;
}

cudaError_t launch_compress_decode(const StoreParams& p, int layout, int grid, cudaStream_t s) {
  if (layout == kV41) return launch_decode_layout<kV41>(p, grid, s);
  if (layout == kV41Fp4) return launch_decode_layout<kV41Fp4>(p, grid, s);
  return launch_decode_layout<kV4>(p, grid, s);
}

}  // namespace dsv4kv
