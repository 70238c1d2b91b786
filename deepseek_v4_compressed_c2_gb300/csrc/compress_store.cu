// Fused compressor: (ratio-2 pair pooling) -> RMSNorm -> RoPE -> store_row
// -> paged write, in one launch.
//
// sglang PR #39652 "dsv4.1: compression, KV I/O, and metadata kernels",
// Summary (c1/c2 bullet): the ratio-1 / ratio-2 compressors do pair-pooling
// (ratio 2), RMSNorm, RoPE and the main-KV write in one launch, returning the
// pre-RoPE latent; out_loc == 0 marks a padded graph row.  The review's
// cleanup of the c2 kernel issues the RoPE frequency load early so its
// latency overlaps the softmax and the RMSNorm reduction; here the
// frequencies arrive with the row's inputs.
// sglang PR #46230: the launch reads low_ratio_extend_offsets (int32 [2,
// request slots]: first row, row count) on the device, so it can sit inside
// a CUDA graph whose offsets are refreshed in place; ratio-2 input is the
// fused | kv | score | projection.
//
// Design (persistent, warp-specialised, two CTAs per SM):
//  * every CTA turns the per-slot row counts into an exclusive prefix in
//    shared memory (the plan), then walks tiles of kRows consecutive output
//    rows, tile = blockIdx.x + i * gridDim.x;
//  * one producer warp: one lane per row of the tile finds the row's request
//    (binary search over the prefix, shared memory only), writes a 16-byte
//    descriptor (state, position, request, row) and issues cp.async.bulk
//    copies of the row's source rows (one 4 KB copy for a ratio-2 pair in
//    the fused layout) and of its RoPE row into a 3-stage shared-memory
//    ring, an mbarrier per stage and consumer warp counting the bytes in
//    flight;
//  * eight consumer warps, each owning one row (ratio 2) or 2-4 (ratio 1) of
//    the stage: wait for the stage, pull the row into registers, release the
//    slot, look up the destination (out_loc or the page table), then pool,
//    normalise, rotate, quantize and store the row.  (The wide launch of
//    store-only rows, which has no arithmetic to hide that lookup behind,
//    has the producer look it up instead, after the row's copy is issued.)
//    Lane l
//    holds dims 8l..8l+7 and 256+8l..263+8l, so every shared-memory read is
//    conflict-free and every global store of a row half is one contiguous
//    warp access; the wide launch of store-only ratio-1 rows gives each
//    half-warp one row instead (consume_tiles_half), so the per-row work of
//    a warp's two rows is one instruction stream;
//  * with start positions or the pair-state ring (decode, verify, chunked
//    prefill) the consumers first run the per-request ring phase.
//  All waits are bounded (see tma.cuh).
#include <atomic>

#include "compress_row.cuh"
#include "internal.cuh"
#include "launchers.cuh"
#include "quant.cuh"
#include "tma.cuh"

namespace dsv4kv {

// Three launch shapes.  Streaming (large batches): 8 consumer warps, 3
// stages, two CTAs per SM, so each SM keeps 48 rows' inputs in flight.
// Streaming-3 (ratio-1 rows with RMSNorm or RoPE): 8 consumer warps of one
// row, 2 stages, three CTAs per SM (72 registers), for rows whose time is
// instruction issue rather than bytes.  Wide (ratio-1 rows that are only
// stored): 8 consumer warps of 2 rows, one per half-warp, 2 stages, three
// CTAs per SM (72 registers): the store-only quantizers are latency-bound
// at two CTAs per SM.  Decode and speculative verify steps (at most 16 rows
// per SM) take the kernel of compress_decode.cu instead.
enum StoreShapeId : int { kShapeStream = 0, kShapeStream3 = 1, kShapeWide = 2 };

template <int SHAPE>
struct StoreShape {
  static constexpr int kWarps = 8;                                   // consumer warps
  static constexpr int kStages = SHAPE == kShapeStream ? 3 : 2;
  static constexpr int kMinBlocks = SHAPE == kShapeStream ? 2 : 3;   // CTAs per SM
  static constexpr int kThreads = (kWarps + 1) * 32;
};

// The 16-byte descriptor of a planned row in a stage.  Streaming shapes: the
// plan's RowDesc, and each consumer looks the destination up itself (that
// global load overlaps the row's arithmetic; a producer waiting on it would
// hold back the copies of the next stage).  Wide shape (rows that are only
// stored): the state and the destination slot (out_loc[k] or the page-table
// entry, -1 past the table), looked up by the producer while the row's copy
// is in flight, so the consumer has no load to wait on.
struct __align__(16) SlotDesc {
  int state;
  int unused;
  long long slot;
};
static_assert(sizeof(SlotDesc) == sizeof(RowDesc), "one descriptor size");

template <int SHAPE>
struct StageDesc {
  using T = RowDesc;
  static constexpr bool kProducerSlot = false;
};
template <>
struct StageDesc<kShapeWide> {
  using T = SlotDesc;
  static constexpr bool kProducerSlot = true;
};

// Rows per consumer warp per stage: one ratio-2 pair (4 KB), four ratio-1
// rows when the row is only stored (32 KB stages either way), two ratio-1
// rows with RMSNorm or RoPE in the streaming shape or in the wide shape
// (four would spill), one in the streaming-3 shape (two spill at 72
// registers).
template <int RATIO, bool NORM, bool ROPE, int SHAPE>
struct StoreTile {
  static constexpr int kWarps = StoreShape<SHAPE>::kWarps;
  static constexpr int kStages = StoreShape<SHAPE>::kStages;
  static constexpr int kThreads = StoreShape<SHAPE>::kThreads;
  static constexpr int kRowsPerWarp =
      RATIO == 2 || SHAPE == kShapeStream3 ? 1 : (NORM || ROPE || SHAPE == kShapeWide ? 2 : 4);
  static constexpr int kRows = kWarps * kRowsPerWarp;              // rows per stage
  static constexpr int kInBytes = RATIO == 2 ? 4096 : 1024;        // kv0|s0|kv1|s1, or kv
  static constexpr int kRopeBytes = ROPE ? kRopeDim * 4 : 0;
  static constexpr int kSlotBytes = kInBytes + kRopeBytes;
  static constexpr int kStageBytes = kRows * kSlotBytes;
  // stages | descriptors | full barriers (one per stage and consumer warp),
  // empty barriers (one per stage), the plan barrier | abort flag (+pad)
  static constexpr int kBarriers = kStages * kWarps + kStages + 1;
  static constexpr int kFixedSmem = kStages * kStageBytes + kStages * kRows * (int)sizeof(RowDesc)
                                  + ((kBarriers * 8 + 8 + 15) & ~15);
  static_assert(kRows <= 32, "one producer lane per row");
  static_assert(kSlotBytes % 16 == 0 && kStageBytes % 128 == 0 && kFixedSmem % 16 == 0,
                "bulk-copy alignment");
};

// The in-CTA plan: first[i], start[i], count[i] and base[i] = sum_{r < i} rows_of_slot(r)
// for i in [0, n_slots] (base[n_slots] = total).
//  * The slot arrays come into shared memory as bulk copies (one per array,
//    completing on the plan barrier) when they are 16-byte aligned and
//    n_slots % 4 == 0; otherwise in one coalesced sweep of plain loads, all
//    issued before any is used (kPlanBatch slots per thread per sweep).
//  * Thread t then owns the PER consecutive slots [t * PER, (t + 1) * PER):
//    their row counts go to registers in one unrolled burst of
//    shared-memory loads, the thread scans them, a shuffle scan per warp and
//    a second one over the warps' totals add the offsets, and the exclusive
//    prefix is written to base.
constexpr int kPlanBatch = 16;

template <int RATIO, int PER>
__device__ __forceinline__ void plan_scan(int n_slots, long long* base, const int* start,
                                          const int* count, long long* s_warp) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
  const int beg = tid * PER, last = n_slots - 1;   // n_slots >= 1
  // loads at clamped (in-bounds) indices, issued together; slots past the
  // end count zero rows
  int cnt[PER], st[PER];
#pragma unroll
  for (int u = 0; u < PER; ++u) {
    const int i = min(beg + u, last);
    cnt[u] = ld_shared_s32(count + i);
    st[u] = ld_shared_s32(start + i);
  }
  long long v[PER];
  long long run = 0;
#pragma unroll
  for (int u = 0; u < PER; ++u) {
    const long long c = beg + u <= last ? rows_of_slot<RATIO>(cnt[u], st[u]) : 0;
    v[u] = run;
    run += c;
  }
  long long incl = run;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long t = __shfl_up_sync(kFullMask, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  // every warp scans the warps' totals across its lanes (nwarps <= 32)
  const long long wt = lane < nwarps ? s_warp[lane] : 0;
  long long wincl = wt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long t = __shfl_up_sync(kFullMask, wincl, o);
    if (lane >= o) wincl += t;
  }
  const long long total = __shfl_sync(kFullMask, wincl, 31);
  const long long off = incl - run + __shfl_sync(kFullMask, wincl - wt, warp);
#pragma unroll
  for (int u = 0; u < PER; ++u)
    if (beg + u <= last) st_shared_s64(base + beg + u, off + v[u]);
  if (tid == 0) st_shared_s64(base + n_slots, total);
}

// Returns false (the same on every thread) when the plan's copies timed out;
// the CTA then does nothing more.  The barrier inits by thread 0 precede the
// call.
template <int RATIO, int THREADS>
__device__ __noinline__ bool block_plan(const int* __restrict__ ext,
                                        const int* __restrict__ start_pos, int n_slots,
                                        long long* base, int* first, int* start, int* count,
                                        uint64_t* bar, volatile int* abort, int* err) {
  // chunk lengths are odd: thread t's slots start at word PER * t, and an odd
  // stride keeps a warp's 4-byte loads and 8-byte stores free of bank
  // conflicts
  constexpr int kPlanMaxPer = ((kMaxSlots + THREADS - 1) / THREADS) | 1;
  __shared__ long long s_warp[32];
  const int tid = threadIdx.x, nt = blockDim.x;
  const bool bulk = n_slots > 0 && (n_slots & 3) == 0 &&
                    (reinterpret_cast<uintptr_t>(ext) & 15) == 0 &&
                    (start_pos == nullptr || (reinterpret_cast<uintptr_t>(start_pos) & 15) == 0);
  if (bulk) {
    if (tid == 0) {
      const uint32_t b = 4u * (uint32_t)n_slots;
      const uint64_t pol = policy_evict_last();
      mbar_arrive_expect_tx(bar, start_pos ? 3 * b : 2 * b);
      bulk_g2s(first, ext, b, bar, pol);
      bulk_g2s(count, ext + n_slots, b, bar, pol);
      if (start_pos) bulk_g2s(start, start_pos, b, bar, pol);
    }
    if (start_pos == nullptr)
      for (int i = tid; i < n_slots; i += nt) start[i] = 0;
    __syncthreads();   // every thread sees the initialised barrier before polling it
    if (!mbar_wait(bar, 0, abort, err) && tid == 0) {
      // the copies still land in this CTA's shared memory: wait for them again
      for (uint32_t i = 0; i < kSpinLimit && !mbar_try_wait(bar, 0); ++i) {
      }
    }
  } else {
    for (int i0 = tid; i0 < n_slots; i0 += kPlanBatch * nt) {
      int f[kPlanBatch], n[kPlanBatch], p0[kPlanBatch];
#pragma unroll
      for (int u = 0; u < kPlanBatch; ++u) {
        const int i = i0 + u * nt;
        f[u] = 0; n[u] = 0; p0[u] = 0;
        if (i < n_slots) {
          f[u] = __ldg(ext + i);
          n[u] = __ldg(ext + n_slots + i);
          if (start_pos) p0[u] = __ldg(start_pos + i);
        }
      }
#pragma unroll
      for (int u = 0; u < kPlanBatch; ++u) {
        const int i = i0 + u * nt;
        if (i < n_slots) {
          first[i] = f[u];
          start[i] = p0[u];
          count[i] = n[u];
        }
      }
    }
  }
  __syncthreads();
  if (*abort) return false;
  if (n_slots == 0) {
    if (tid == 0) base[0] = 0;
    return true;
  }
  const int per = (n_slots + nt - 1) / nt;
  if (per <= 1)
    plan_scan<RATIO, 1>(n_slots, base, start, count, s_warp);
  else if (per <= 5)
    plan_scan<RATIO, 5>(n_slots, base, start, count, s_warp);
  else
    plan_scan<RATIO, kPlanMaxPer>(n_slots, base, start, count, s_warp);
  return true;
}

// The plan for output row k (shared memory only, no global loads): request
// slot r (last slot whose prefix <= k), row j = k - base[r] of the request,
// compressed index c = c_lo + j (c_lo = p0 for ratio 1, p0 / 2 for ratio 2),
// first token at position RATIO*c in source row first_r + RATIO*c - p0, or in
// the ring when that position precedes p0 (only with start positions at
// ratio 2, RING).
template <int RATIO, bool ROPE, bool RING>
__device__ __forceinline__ RowDesc plan_row(const StoreParams& p, long long k, long long total,
                                            const long long* s_base, const int* s_first,
                                            const int* s_start, const int* s_count,
                                            long long& src) {
  RowDesc d;
  d.state = kRowNone; d.pos = 0; d.r = 0; d.c = 0;
  src = 0;
  if (k >= p.n_out) return d;
  if (k >= total) { d.state = kRowPad; return d; }
  int lo = 0, hi = p.n_slots - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_base[mid] <= k) lo = mid; else hi = mid - 1;
  }
  const long long p0 = s_start[lo];
  const long long c = (RATIO == 2 ? (p0 >> 1) : p0) + (k - s_base[lo]);
  const long long pos = (long long)RATIO * c;
  d.r = lo;
  d.c = (int)c;
  d.pos = (int)pos;
  src = (long long)s_first[lo] + (pos - p0);
  if (RING && pos < p0) {                          // first token in the ring
    if (p.ring == nullptr) { d.state = kRowBad; return d; }
    if (s_count[lo] >= 2LL * p.ring_size) { d.state = kRowRing; return d; }
    const long long first = s_first[lo];
    const bool ok = first >= 0 && first + 1 <= p.n_rows && pos >= 0 && (!ROPE || pos < p.max_pos);
    d.state = ok ? kRowOkRing : kRowBad;
    return d;
  }
  const bool ok = src >= 0 && src + RATIO <= p.n_rows && pos >= 0 && (!ROPE || pos < p.max_pos);
  d.state = ok ? kRowOk : kRowBad;
  return d;
}

// Per-request ring work (ratio 2).  Each warp owns the request slots
// r = warp id + i * (warps in the grid) and makes two passes over them:
// (1) for a request whose step has n >= 2R new tokens, the pair whose first
// token precedes p0 -- token p0 - 1 from the ring entry ((p0 - 1) / 2) % R,
// token p0 from the first new row; (2) the ring update: each even-position
// new token among the last 2R positions of the step goes to entry
// (q / 2) % R.  A lane writes exactly the 16-byte words it read, and pass (1)
// ends before pass (2) starts, so every read of (1) precedes any write of the
// same entry.  With n < 2R the entries written are (p0+1)/2 .. (p0+n-1)/2,
// all different from the read entry (p0-1)/2 modulo R, so the tile path may
// read that entry at any time.  No other warp writes this request's ring,
// and no tile reads an entry that this phase writes, so the consumers run it
// before their tile loop, while the producer's first copies are in flight.
template <int L, bool NORM, bool ROPE, int WARPS>
__device__ __noinline__ void ring_phase(const StoreParams& p, const long long* s_base,
                                        const int* s_first, const int* s_start,
                                        const int* s_count, int warp, int lane) {
  const __nv_bfloat16* score_base = p.score ? p.score : p.rows + kDim;
  const long long sstride = p.score ? p.score_stride : p.row_stride;
  const long long stride = (long long)gridDim.x * WARPS;
  const int R = p.ring_size;
  // (1) ring rows of the requests with n >= 2R new tokens
  for (long long r = (long long)blockIdx.x * WARPS + warp; r < p.n_slots; r += stride) {
    const int n = ld_shared_s32(s_count + r);
    const long long p0 = ld_shared_s32(s_start + r);
    if (n <= 0 || !(p0 & 1) || p.ring == nullptr || n < 2LL * R) continue;
    const long long k = ld_shared_s64(s_base + r);
    if (k >= p.n_out) continue;
    const long long first = ld_shared_s32(s_first + r);
    float w[16];
    if constexpr (NORM) {
      const uint4* wp = reinterpret_cast<const uint4*>(p.norm_w);
      unpack_bf16x8(__ldg(wp + lane), w);
      unpack_bf16x8(__ldg(wp + 32 + lane), w + 8);
    }
    RowDesc d;
    d.r = (int)r; d.c = (int)(p0 >> 1); d.pos = (int)(p0 - 1);
    const bool ok = p0 >= 1 && first >= 0 && first + 1 <= p.n_rows && (!ROPE || d.pos < p.max_pos);
    d.state = ok ? kRowOk : kRowBad;
    RowIn<2, ROPE> in;
    long long slot = 0;
    if (ok) {
      const uint4* e = reinterpret_cast<const uint4*>(
          p.ring + ((r * R) + (d.c % R)) * (2 * kDim));
      const uint4* kv = reinterpret_cast<const uint4*>(p.rows + first * p.row_stride);
      const uint4* sc = reinterpret_cast<const uint4*>(score_base + first * sstride);
      in.kv0[0] = e[lane];       in.kv0[1] = e[32 + lane];
      in.s0[0] = e[64 + lane];   in.s0[1] = e[96 + lane];
      in.kv1[0] = kv[lane];      in.kv1[1] = kv[32 + lane];
      in.s1[0] = sc[lane];       in.s1[1] = sc[32 + lane];
      if constexpr (ROPE) {
        if (lane >= 24) {
          const float4* f = reinterpret_cast<const float4*>(p.freqs + (long long)d.pos * kRopeDim);
          in.fr[0] = f[2 * (lane - 24)];
          in.fr[1] = f[2 * (lane - 24) + 1];
        }
      }
      slot = dest_slot(p, k, d);
    }
    process_row<L, 2, NORM, ROPE>(p, k, d.state, slot, in, w, lane);
  }
  if (p.ring == nullptr) return;
  __syncwarp();
  // (2) the ring update.  The warp takes its requests kRingGroup at a time;
  // lane l stands for token tl = l % kRingLanes (+ multiples of kRingLanes)
  // of request l / kRingLanes and works out its source row and ring entry.
  // A ballot lists the lanes whose token is valid, and the warp copies those
  // tokens kRingCopies at a time (the 2 KB kv | score row, 16 bytes per lane
  // per load).  All the entries of a group are distinct.  A token at a
  // negative position, or whose source row is out of range, is a fault.
  constexpr int kRingGroup = 4, kRingLanes = 32 / kRingGroup, kRingCopies = 2;
  const int gj = lane / kRingLanes, tl = lane % kRingLanes;
  for (long long r0 = (long long)blockIdx.x * WARPS + warp; r0 < p.n_slots;
       r0 += kRingGroup * stride) {
    const long long r = r0 + gj * stride;
    long long qlo = 0, src = 0;
    int ntok = 0;
    if (r < p.n_slots) {
      const int n = ld_shared_s32(s_count + r);
      const long long p0 = ld_shared_s32(s_start + r);
      long long q = p0 + n - 2LL * R;
      if (q < p0) q = p0;
      q += q & 1;                                   // the first even position
      if (n > 0 && p0 + n > q) {
        qlo = q;
        ntok = (int)((p0 + n - q + 1) >> 1);        // <= R
        src = ld_shared_s32(s_first + r) + (q - p0);
      }
    }
    const int max_tok = __reduce_max_sync(kFullMask, (unsigned)ntok);
    for (int t0 = 0; t0 < max_tok; t0 += kRingLanes) {
      const int t = t0 + tl;
      const long long q = qlo + 2LL * t, row = src + 2LL * t;
      const bool has = t < ntok;
      const bool bad = has && (q < 0 || row < 0 || row >= p.n_rows);
      const unsigned n_bad = __popc(__ballot_sync(kFullMask, bad));
      if (lane == 0 && n_bad && p.err) atomicAdd(p.err, (int)n_bad);
      unsigned todo = __ballot_sync(kFullMask, has && !bad);
      const long long dst = has && !bad ? (r * R + (unsigned)(q >> 1) % (unsigned)R) * (2 * kDim) : 0;
      while (todo) {
        long long rows_[kRingCopies], dsts_[kRingCopies];
        bool use[kRingCopies];
#pragma unroll
        for (int c = 0; c < kRingCopies; ++c) {
          use[c] = todo != 0;
          const int l = use[c] ? __ffs(todo) - 1 : 0;
          if (use[c]) todo &= todo - 1;
          rows_[c] = __shfl_sync(kFullMask, row, l);
          dsts_[c] = __shfl_sync(kFullMask, dst, l);
        }
        uint4 v[kRingCopies][4];
#pragma unroll
        for (int c = 0; c < kRingCopies; ++c) {
          if (!use[c]) continue;
          const uint4* kv = reinterpret_cast<const uint4*>(p.rows + rows_[c] * p.row_stride);
          const uint4* sc = reinterpret_cast<const uint4*>(score_base + rows_[c] * sstride);
          v[c][0] = kv[lane]; v[c][1] = kv[32 + lane]; v[c][2] = sc[lane]; v[c][3] = sc[32 + lane];
        }
#pragma unroll
        for (int c = 0; c < kRingCopies; ++c) {
          if (!use[c]) continue;
          uint4* e = reinterpret_cast<uint4*>(p.ring + dsts_[c]);
          e[lane] = v[c][0]; e[32 + lane] = v[c][1]; e[64 + lane] = v[c][2]; e[96 + lane] = v[c][3];
        }
      }
    }
  }
}

// The consumer warps' tile loop: wait for a stage, pull the rows into
// registers, release the stage, then finish each row (process_row).
template <int L, int RATIO, bool NORM, bool ROPE, int SHAPE>
__device__ __forceinline__ void consume_tiles(const StoreParams& p, const uint8_t* s_stage,
                                              const RowDesc* s_desc, uint64_t* s_full,
                                              uint64_t* s_empty, volatile int* abort,
                                              int n_tiles, int warp, int lane) {
  using TL = StoreTile<RATIO, NORM, ROPE, SHAPE>;
  float w[16];
  if constexpr (NORM) {
    const uint4* wp = reinterpret_cast<const uint4*>(p.norm_w);
    unpack_bf16x8(__ldg(wp + lane), w);
    unpack_bf16x8(__ldg(wp + 32 + lane), w + 8);
  }
  // iteration it uses stage it % kStages for the (it / kStages)-th time (32-bit:
  // the producer's incremental form costs this loop registers and spills)
  int it = 0;
  for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, ++it) {
    const int s = it % TL::kStages;
    const uint32_t use = (uint32_t)(it / TL::kStages);
    if (!mbar_wait(&s_full[s * TL::kWarps + warp], use & 1u, abort, p.err)) break;
    RowDesc d[TL::kRowsPerWarp];
    RowIn<RATIO, ROPE> in[TL::kRowsPerWarp];
    long long slot[TL::kRowsPerWarp];
#pragma unroll
    for (int q = 0; q < TL::kRowsPerWarp; ++q) {
      const int t = warp * TL::kRowsPerWarp + q;
      d[q] = s_desc[s * TL::kRows + t];
      const bool ok = d[q].state == kRowOk || d[q].state == kRowOkRing;
      slot[q] = ok ? dest_slot(p, (long long)tile * TL::kRows + t, d[q]) : 0;
      const uint8_t* stage = s_stage + s * TL::kStageBytes;
      if (ok)
        load_row<RATIO, ROPE>(stage + t * TL::kInBytes,
                              stage + TL::kRows * TL::kInBytes + t * TL::kRopeBytes, lane, in[q]);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&s_empty[s]);
#pragma unroll
    for (int q = 0; q < TL::kRowsPerWarp; ++q) {
      const long long k = (long long)tile * TL::kRows + warp * TL::kRowsPerWarp + q;
      process_row<L, RATIO, NORM, ROPE>(p, k, d[q].state, slot[q], in[q], w, lane);
    }
  }
}

// The wide launch (ratio 1, rows only stored): each half-warp takes one of
// the warp's two rows in the half-warp layout of the chunk quantizers, so the
// per-row work (descriptor, row state, destination lookup, addressing) is
// one instruction stream for both rows instead of one per row.  Row states
// and outputs follow process_row: none -> nothing; pad / bad -> zeroed debug
// outputs (bad: one fault); ok -> a fault if the slot is past the pool, the
// debug outputs, and the stored row when 0 < slot < pool_rows.
template <int L>
__device__ __forceinline__ void consume_tiles_half(const StoreParams& p, const uint8_t* s_stage,
                                                   const SlotDesc* s_desc, uint64_t* s_full,
                                                   uint64_t* s_empty, volatile int* abort,
                                                   int n_tiles, int warp, int lane) {
  using TL = StoreTile<1, false, false, kShapeWide>;
  static_assert(TL::kRowsPerWarp == 2, "one row per half-warp");
  const int l = lane & 15;
  const int t = warp * 2 + (lane >> 4);     // this half's row in the tile
  // the 16-byte unit (8 dims) of the row that chunk c of sub-lane l holds:
  // dims 128c + 8l, or for FP4 the halves of groups l (c = 0, 1) and 16 + l
  // (c = 2, 3)
  int unit[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) unit[c] = L == kV41Fp4 ? 32 * (c >> 1) + 2 * l + (c & 1) : 16 * c + l;
  int it = 0;
  for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, ++it) {
    const int s = it % TL::kStages;
    const uint32_t use = (uint32_t)(it / TL::kStages);
    if (!mbar_wait(&s_full[s * TL::kWarps + warp], use & 1u, abort, p.err)) break;
    const SlotDesc d = s_desc[s * TL::kRows + t];
    const long long k = (long long)tile * TL::kRows + t;
    const bool ok = d.state == kRowOk;
    const long long slot = d.slot;
    const uint4* src = reinterpret_cast<const uint4*>(s_stage + s * TL::kStageBytes + t * TL::kInBytes);
    uint4 v[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) v[c] = ok ? src[unit[c]] : make_uint4(0u, 0u, 0u, 0u);
    __syncwarp();
    if (lane == 0) mbar_arrive(&s_empty[s]);
    if (!ok && d.state != kRowNone) {       // pad or bad (no shuffles on this branch)
      if (d.state == kRowBad && l == 0 && p.err) atomicAdd(p.err, 1);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        if (p.latent_out)
          reinterpret_cast<uint4*>(p.latent_out + k * kDim)[unit[c]] = make_uint4(0u, 0u, 0u, 0u);
        if (p.prequant_out) {
          float4* o = reinterpret_cast<float4*>(p.prequant_out + k * kDim) + 2 * unit[c];
          o[0] = make_float4(0.f, 0.f, 0.f, 0.f);
          o[1] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
    }
    const bool store = ok && slot > 0 && slot < p.pool_rows;
    if (ok && slot != 0 && !store && l == 0 && p.err) atomicAdd(p.err, 1);   // destination fault
    uint8_t* row = store ? PagedKV<L>{p.pool, p.page_bits}.row(slot) : nullptr;
    float xg[16];                             // FP4: the group being assembled
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      float x[8];
#pragma unroll
      for (int q = 0; q < 4; ++q)
        f2_split(f2_from_bf16x2(word_of(v[c], q)), x[2 * q], x[2 * q + 1]);
      if (ok && p.latent_out)   // no RMSNorm: the latent is the row itself
        reinterpret_cast<uint4*>(p.latent_out + k * kDim)[unit[c]] = pack_bf16x8(x);
      if (ok && p.prequant_out) {
        float4* o = reinterpret_cast<float4*>(p.prequant_out + k * kDim) + 2 * unit[c];
        o[0] = make_float4(x[0], x[1], x[2], x[3]);
        o[1] = make_float4(x[4], x[5], x[6], x[7]);
      }
      if constexpr (L == kV41Fp4) {
#pragma unroll
        for (int i = 0; i < 8; ++i) xg[8 * (c & 1) + i] = x[i];
        if (c & 1) store_group_fp4(xg, row, 16 * (c >> 1) + l, store);
      } else {
        store_chunk<L>(x, row, c, l, store);
      }
    }
  }
}

// RING: ratio 2 with start positions and/or the pair-state ring.  The
// launches without either take RING = false, whose kernel has no ring code.
template <int L, int RATIO, bool NORM, bool ROPE, bool RING, int SHAPE>
__global__ void __launch_bounds__(StoreShape<SHAPE>::kThreads, StoreShape<SHAPE>::kMinBlocks)
compress_store_kernel(const StoreParams p) {
  using TL = StoreTile<RATIO, NORM, ROPE, SHAPE>;
  using Desc = typename StageDesc<SHAPE>::T;
  constexpr bool kProducerSlot = StageDesc<SHAPE>::kProducerSlot;
  constexpr int kStages = TL::kStages;
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* s_stage = smem;
  Desc* s_desc = reinterpret_cast<Desc*>(smem + kStages * TL::kStageBytes);
  uint64_t* s_full = reinterpret_cast<uint64_t*>(s_desc + kStages * TL::kRows);
  uint64_t* s_empty = s_full + kStages * TL::kWarps;
  uint64_t* s_plan = s_empty + kStages;
  int* s_abort = reinterpret_cast<int*>(s_plan + 1);
  // the plan: base (an even count of 8-byte entries, >= n_slots + 1) | first
  // | start | count, each array 16-byte aligned when n_slots % 4 == 0
  long long* s_base = reinterpret_cast<long long*>(smem + TL::kFixedSmem);
  int* s_first = reinterpret_cast<int*>(s_base + ((p.n_slots + 2) & ~1));
  int* s_start = s_first + p.n_slots;
  int* s_count = s_start + p.n_slots;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      for (int w = 0; w < TL::kWarps; ++w)
        mbar_init(&s_full[s * TL::kWarps + w], kProducerSlot ? 2 : 1);
      mbar_init(&s_empty[s], TL::kWarps);
    }
    mbar_init(s_plan, 1);
    *s_abort = 0;
    mbar_fence_init();
  }
  grid_dependency_wait();
  volatile int* abort = s_abort;
  if (!block_plan<RATIO, TL::kThreads>(p.ext, p.start_pos, p.n_slots, s_base, s_first, s_start, s_count, s_plan,
                         abort, p.err))
    return;
  __syncthreads();
  const long long total = s_base[p.n_slots];
  const int n_tiles = (int)(((long long)p.n_out + TL::kRows - 1) / TL::kRows);

  if (warp == TL::kWarps) {
    // ------------------------------------------------------------ producer
    const uint64_t pol = policy_evict_first();
    const __nv_bfloat16* score_base = p.score ? p.score : p.rows + kDim;
    const long long sstride = p.score ? p.score_stride : p.row_stride;
    const bool fused_pair = p.score == nullptr && p.row_stride == 2 * kDim;
    int it = 0, s = 0;          // iterations; stage s, used `use` times before
    uint32_t use = 0;
    for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, ++it) {
      if (use > 0 && !mbar_wait(&s_empty[s], (use - 1) & 1u, abort, p.err)) break;
      RowDesc d;
      d.state = kRowNone;
      long long src = 0, slot = 0;
      if (lane < TL::kRows) {
        const long long k = (long long)tile * TL::kRows + lane;
        d = plan_row<RATIO, ROPE, RING>(p, k, total, s_base, s_first, s_start, s_count, src);
        if constexpr (kProducerSlot) {
          // the destination's global load stays in flight across the copies' issue
          if (d.state == kRowOk) slot = dest_slot(p, k, d);
        } else {
          s_desc[s * TL::kRows + lane] = d;
        }
      }
      // each consumer warp's rows complete on that warp's own barrier: the
      // first lane of the warp's rows (the group leader) arms it with their
      // bytes before the copies (and in the wide shape arrives a second time
      // once the group's descriptors, with their slots, are written).
      // Ratio 1: a group of consecutive packed source rows comes in one copy
      // issued by the leader.
      const bool copy = d.state == kRowOk || d.state == kRowOkRing;
      const int leader = lane & ~(TL::kRowsPerWarp - 1);
      bool merged = false;
      if constexpr (RATIO == 1 && TL::kRowsPerWarp > 1) {
        const long long src_l = __shfl_sync(kFullMask, src, leader);
        const bool next = lane < TL::kRows && d.state == kRowOk && src == src_l + (lane - leader);
        const unsigned all = __ballot_sync(kFullMask, next);
        const unsigned group = ((1u << TL::kRowsPerWarp) - 1u) << leader;
        merged = p.row_stride == kDim && (all & group) == group;
      }
      uint64_t* bar = &s_full[s * TL::kWarps + min(lane, TL::kRows - 1) / TL::kRowsPerWarp];
      uint32_t bytes = copy ? (uint32_t)TL::kSlotBytes : 0u;
#pragma unroll
      for (int o = 1; o < TL::kRowsPerWarp; o <<= 1) bytes += __shfl_xor_sync(kFullMask, bytes, o);
      __syncwarp();
      const bool group_leader = lane < TL::kRows && lane % TL::kRowsPerWarp == 0;
      if (group_leader) mbar_arrive_expect_tx(bar, bytes);
      __syncwarp();
      if (copy) {
        uint8_t* stage = s_stage + s * TL::kStageBytes;
        uint8_t* dst = stage + lane * TL::kInBytes;
        const __nv_bfloat16* r0 = p.rows + (d.state == kRowOkRing ? 0 : src) * p.row_stride;
        if constexpr (RATIO == 2) {
          if (d.state == kRowOkRing) {
            // token p0 - 1 from the ring (kv | score, 2 KB), token p0 = row src + 1
            const __nv_bfloat16* e =
                p.ring + ((long long)d.r * p.ring_size + (d.c % p.ring_size)) * (2 * kDim);
            const __nv_bfloat16* r1 = p.rows + (src + 1) * p.row_stride;
            bulk_g2s(dst, e, 2048, bar, pol);
            if (fused_pair) {
              bulk_g2s(dst + 2048, r1, 2048, bar, pol);
            } else {
              bulk_g2s(dst + 2048, r1, 1024, bar, pol);
              bulk_g2s(dst + 3072, score_base + (src + 1) * sstride, 1024, bar, pol);
            }
          } else if (fused_pair) {
            bulk_g2s(dst, r0, 4096, bar, pol);             // kv0|s0|kv1|s1
          } else {
            const __nv_bfloat16* c0 = score_base + src * sstride;
            bulk_g2s(dst, r0, 1024, bar, pol);
            bulk_g2s(dst + 1024, c0, 1024, bar, pol);
            bulk_g2s(dst + 2048, r0 + p.row_stride, 1024, bar, pol);
            bulk_g2s(dst + 3072, c0 + sstride, 1024, bar, pol);
          }
        } else if (!merged) {
          bulk_g2s(dst, r0, 1024, bar, pol);
        } else if (lane == leader) {
          bulk_g2s(dst, r0, 1024 * TL::kRowsPerWarp, bar, pol);
        }
        if constexpr (ROPE)
          bulk_g2s(stage + TL::kRows * TL::kInBytes + lane * TL::kRopeBytes,
                   p.freqs + (long long)d.pos * kRopeDim, kRopeDim * 4, bar, pol);
      }
      if constexpr (kProducerSlot) {
        if (lane < TL::kRows) s_desc[s * TL::kRows + lane] = SlotDesc{d.state, 0, slot};
        __syncwarp();
        if (group_leader) mbar_arrive(bar);
      }
      if (++s == kStages) { s = 0; ++use; }
    }
    // every issued copy has landed before the CTA may exit (bounded)
    if (lane < TL::kWarps) {
      for (int st = 0; st < kStages && st < it; ++st) {
        const uint32_t last_use = (uint32_t)((it - 1 - st) / kStages);
        uint64_t* bar = &s_full[st * TL::kWarps + lane];
        for (uint32_t i = 0; i < kSpinLimit && !mbar_try_wait(bar, last_use & 1u); ++i) {
        }
      }
    }
    allow_dependent_launch();
  } else {
    // ------------------------------------------------------------ consumers
    if constexpr (RATIO == 2 && RING)
      ring_phase<L, NORM, ROPE, TL::kWarps>(p, s_base, s_first, s_start, s_count, warp, lane);
    if constexpr (SHAPE == kShapeWide)
      consume_tiles_half<L>(p, s_stage, s_desc, s_full, s_empty, abort, n_tiles, warp, lane);
    else
      consume_tiles<L, RATIO, NORM, ROPE, SHAPE>(p, s_stage, s_desc, s_full, s_empty, abort,
                                                 n_tiles, warp, lane);
    allow_dependent_launch();
  }
}

template <int L, int RATIO, bool NORM, bool ROPE, bool RING, int SHAPE>
static cudaError_t launch_variant(const StoreParams& p, cudaStream_t stream) {
  using TL = StoreTile<RATIO, NORM, ROPE, SHAPE>;
  auto kern = compress_store_kernel<L, RATIO, NORM, ROPE, RING, SHAPE>;
  const size_t smem = (size_t)TL::kFixedSmem + sizeof(long long) * (size_t)((p.n_slots + 2) & ~1)
                    + 3 * sizeof(int) * (size_t)p.n_slots;
  // the largest size any call can need, set once per device; the flag is
  // published (release) only after the attribute call succeeded
  static std::atomic<int> attr_set_for_device[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 64 || !attr_set_for_device[dev].load(std::memory_order_acquire)) {
    const size_t max_smem = (size_t)TL::kFixedSmem + sizeof(long long) * ((kMaxSlots + 2) & ~1)
                          + 3 * sizeof(int) * kMaxSlots;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)max_smem);
    if (e != cudaSuccess) return e;
    if (dev < 64) attr_set_for_device[dev].store(1, std::memory_order_release);
  }
  // resident CTAs per SM at this shared-memory size, cached per device as
  // (smem << 8 | per_sm): the query costs more host time than the launch
  static std::atomic<unsigned long long> occupancy[64];
  int per_sm = 0;
  const unsigned long long seen = dev < 64 ? occupancy[dev].load(std::memory_order_relaxed) : 0ull;
  if (seen != 0 && (seen >> 8) == (unsigned long long)smem) {
    per_sm = (int)(seen & 0xFF);
  } else {
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, TL::kThreads, smem);
    if (e != cudaSuccess) return e;
    if (dev < 64 && per_sm > 0 && per_sm < 256)
      occupancy[dev].store(((unsigned long long)smem << 8) | (unsigned long long)per_sm,
                           std::memory_order_relaxed);
  }
  const long long tiles = ((long long)p.n_out + TL::kRows - 1) / TL::kRows;
  const long long cap = (long long)device_sm_count() * (per_sm > 0 ? per_sm : 1);
  const int grid = (int)(tiles < cap ? tiles : cap);
  return launch_dependent(kern, grid, TL::kThreads, smem, stream, p);
}

template <int L, int RATIO, bool RING, int SHAPE>
static cudaError_t launch_norm_rope(const StoreParams& p, cudaStream_t s) {
  const bool norm = p.norm_w != nullptr, rope = p.freqs != nullptr;
  if (norm && rope) return launch_variant<L, RATIO, true, true, RING, SHAPE>(p, s);
  if (norm) return launch_variant<L, RATIO, true, false, RING, SHAPE>(p, s);
  if (rope) return launch_variant<L, RATIO, false, true, RING, SHAPE>(p, s);
  return launch_variant<L, RATIO, false, false, RING, SHAPE>(p, s);
}

// The ring form (start positions and/or the pair-state ring) of steps of at
// most 16 output rows per SM -- decode, speculative-verify and short
// chunked-prefill steps -- runs the latency-shaped kernel of
// compress_decode.cu (one chunk of request slots per CTA, no wait for a
// plan of the whole step before a row's loads); longer steps (chunked
// prefill) stream.
template <int L>
static cudaError_t launch_ratio(const StoreParams& p, int ratio, cudaStream_t s) {
  if (ratio == 1) {
    const bool norm = p.norm_w != nullptr, rope = p.freqs != nullptr;
    if (norm && rope) return launch_variant<L, 1, true, true, false, kShapeStream3>(p, s);
    if (norm) return launch_variant<L, 1, true, false, false, kShapeStream3>(p, s);
    if (rope) return launch_variant<L, 1, false, true, false, kShapeStream3>(p, s);
    return launch_variant<L, 1, false, false, false, kShapeWide>(p, s);
  }
  if (p.start_pos == nullptr && p.ring == nullptr)
    return launch_norm_rope<L, 2, false, kShapeStream>(p, s);
  const long long sms = device_sm_count();
  if ((long long)p.n_out <= sms * kDecodeRowsPerCta) {
    const int grid = decode_grid(p.n_slots, p.n_out, (int)sms);
    if (grid > 0) return launch_compress_decode(p, L, grid, s);
  }
  return launch_norm_rope<L, 2, true, kShapeStream>(p, s);
}

cudaError_t launch_compress_store(const StoreParams& p, int layout, int ratio, cudaStream_t s) {
  if (layout == kV41) return launch_ratio<kV41>(p, ratio, s);
  if (layout == kV41Fp4) return launch_ratio<kV41Fp4>(p, ratio, s);
  return launch_ratio<kV4>(p, ratio, s);
}

}  // namespace dsv4kv
