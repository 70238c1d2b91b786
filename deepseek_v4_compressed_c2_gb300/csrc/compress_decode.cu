// Large decode / speculative-verify steps of the ratio-2 compressor: one
// launch for a step of a few new tokens per request that makes more than 8
// and at most 16 compressed rows per SM.
//
// sglang PR #39652 "dsv4.1: compression, KV I/O, and metadata kernels",
// Summary (c1/c2 bullet) and the review of the c2 kernel: the ratio-2 decode
// compressor keeps a pair-state ring, completes a pair at an odd position and
// rotates it with the RoPE frequencies of pos - 1; sglang PR #46230: the
// offsets are read on the device, so the launch can sit in a CUDA graph whose
// metadata is refreshed in place.
//
// Such a step is latency-bound (a few MB, L2-resident), so the launch is
// shaped for latency rather than bandwidth.  Every CTA owns exactly one tile
// of kDecRows consecutive output rows (grid = tiles) and has:
//  * a plan in shared memory: thread t reads the metadata of request slots
//    [8t, 8t + 8) with vector loads and stores it, and a saturating 32-bit
//    scan gives every slot's first output row (exact for every row below
//    n_out) -- no staged copy of the slot arrays;
//  * kDecRows row warps: warp w finds the slot of its row by binary search
//    over the slots' first rows, loads the row's inputs straight into
//    registers (the ring entry for a pair whose first token precedes the
//    step, the new token's kv | score, the RoPE row) and the destination
//    slot, then runs process_row;
//  * kDecRingWarps ring warps: the ring update (each even-position new token
//    among the last 2R positions of a request goes to entry (q / 2) % R).
// Every read of a ring entry precedes any write of it without a barrier: a
// request whose ring-reading row (its first row, at an odd start) is computed
// in this launch is updated by that row's CTA -- by the ring warps when its
// step has n < 2R tokens (the update then writes other entries than the one
// read), else by the row's own warp after the row (program order) -- and
// every other request by CTA r % grid, whose update no row of the launch
// reads.
#include <atomic>
#include <cstddef>

#include "compress_row.cuh"
#include "internal.cuh"
#include "launchers.cuh"
#include "tma.cuh"

namespace dsv4kv {

constexpr int kDecRows = kDecodeRowsPerCta;          // rows per CTA, one per row warp
constexpr int kDecRingWarps = 4;
constexpr int kDecWarps = kDecRows + kDecRingWarps;
constexpr int kDecThreads = kDecWarps * 32;
constexpr int kDecPer = 8;                            // plan: request slots per thread
constexpr int kDecPlanThreads = kMaxSlots / kDecPer;  // 512
constexpr int kDecPlanWarps = kDecPlanThreads / 32;
constexpr int kDecRingCopies = 3;                     // 2 KB tokens in flight per warp
static_assert(kDecPlanThreads <= kDecThreads && kDecPlanWarps <= 32, "plan fits the CTA");

// One ring-warp lane's request: its ring tokens (none when another CTA does
// its update).
struct RingWork {
  long long q, src;
  int r, ntok;
};

struct DecodeShared {
  uint4 norm_w[64];            // the RMSNorm weight row, bf16 [512]
  unsigned wsum[kDecPlanWarps];
  unsigned total;              // rows of the plan (saturated at n_out)
  int n_list;
  int list[kDecRows];          // ring-reading requests of this tile with ring tokens, n < 2R
};

// The plan's per-slot arrays (dynamic shared memory, after DecodeShared):
// first source row, new-token count, start position, first output row.
struct DecodePlan {
  int* first;
  int* count;
  int* start;
  unsigned* base;
};
constexpr size_t kDecPlanBytes = 4 * sizeof(int) * (size_t)kMaxSlots;

__device__ __forceinline__ unsigned sat_add(unsigned a, unsigned b, unsigned cap) {
  const unsigned s = a + b;    // a, b <= cap < 2^31: no wrap
  return s < cap ? s : cap;
}

// Slot metadata of slots [s0, s0 + kDecPer): first source row, new-token
// count, start position (0 without start positions); slots past n_slots get
// count 0.
__device__ __forceinline__ void load_slots(const StoreParams& p, int s0, int (&first)[kDecPer],
                                           int (&count)[kDecPer], int (&start)[kDecPer]) {
  const bool vec = (p.n_slots & 3) == 0 && s0 + kDecPer <= p.n_slots &&
                   (reinterpret_cast<uintptr_t>(p.ext) & 15) == 0 &&
                   (p.start_pos == nullptr || (reinterpret_cast<uintptr_t>(p.start_pos) & 15) == 0);
  if (vec) {
    const int4* f = reinterpret_cast<const int4*>(p.ext + s0);
    const int4* c = reinterpret_cast<const int4*>(p.ext + p.n_slots + s0);
    const int4 f0 = __ldg(f), f1 = __ldg(f + 1), c0 = __ldg(c), c1 = __ldg(c + 1);
    int4 t0 = make_int4(0, 0, 0, 0), t1 = t0;
    if (p.start_pos) {
      const int4* t = reinterpret_cast<const int4*>(p.start_pos + s0);
      t0 = __ldg(t);
      t1 = __ldg(t + 1);
    }
    first[0] = f0.x; first[1] = f0.y; first[2] = f0.z; first[3] = f0.w;
    first[4] = f1.x; first[5] = f1.y; first[6] = f1.z; first[7] = f1.w;
    count[0] = c0.x; count[1] = c0.y; count[2] = c0.z; count[3] = c0.w;
    count[4] = c1.x; count[5] = c1.y; count[6] = c1.z; count[7] = c1.w;
    start[0] = t0.x; start[1] = t0.y; start[2] = t0.z; start[3] = t0.w;
    start[4] = t1.x; start[5] = t1.y; start[6] = t1.z; start[7] = t1.w;
  } else {
#pragma unroll
    for (int u = 0; u < kDecPer; ++u) {
      const int r = s0 + u;
      const bool in = r < p.n_slots;
      first[u] = in ? __ldg(p.ext + r) : 0;
      count[u] = in ? __ldg(p.ext + p.n_slots + r) : 0;
      start[u] = in && p.start_pos ? __ldg(p.start_pos + r) : 0;
    }
  }
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

// The ring tokens of request slot r: the even positions q, q + 2, ... among
// the step's last 2R positions, from source rows src, src + 2, ...
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

// The ring tokens of request r, none when another CTA does its update (a
// round-robin candidate whose ring-reading row is computed is updated by
// that row's CTA: listed in sh.list, or by the row's warp when n >= 2R).
__device__ __forceinline__ RingWork ring_work(const StoreParams& p, const DecodePlan& pl, int r,
                                              bool candidate, unsigned cap) {
  RingWork w{0, 0, r, 0};
  if (r < 0) return w;
  const int n = pl.count[r], p0 = pl.start[r];
  if (candidate && (p0 & 1) && rows_of_slot<2>(n, p0) > 0 && pl.base[r] < cap) return w;
  w.ntok = ring_tokens(n, p0, pl.first[r], p.ring_size, w.q, w.src);
  return w;
}

// Copies ring tokens (the warp moves 2 KB kv | score rows from the input
// rows to ring entries, kDecRingCopies at a time): lane l's request has
// ntok tokens at positions q, q + 2, ... in source rows src, src + 2, ...;
// a token at a negative position or past the rows is a fault.
__device__ __forceinline__ void copy_ring_tokens(const StoreParams& p, const RingWork& rwk,
                                                 int lane) {
  const int R = p.ring_size;
  const __nv_bfloat16* score_base = p.score ? p.score : p.rows + kDim;
  const long long sstride = p.score ? p.score_stride : p.row_stride;
  const int max_tok = __reduce_max_sync(kFullMask, (unsigned)rwk.ntok);
  for (int t = 0; t < max_tok; ++t) {
    const long long qt = rwk.q + 2LL * t, row = rwk.src + 2LL * t;
    const bool has = t < rwk.ntok;
    const bool bad = has && (qt < 0 || row < 0 || row >= p.n_rows);
    const unsigned n_bad = __popc(__ballot_sync(kFullMask, bad));
    if (lane == 0 && n_bad && p.err) atomicAdd(p.err, (int)n_bad);
    unsigned todo = __ballot_sync(kFullMask, has && !bad);
    const long long dst =
        has && !bad ? ((long long)rwk.r * R + (unsigned)(qt >> 1) % (unsigned)R) * (2 * kDim) : 0;
    while (todo) {
      long long rows_[kDecRingCopies], dsts_[kDecRingCopies];
      bool use[kDecRingCopies];
#pragma unroll
      for (int c = 0; c < kDecRingCopies; ++c) {
        use[c] = todo != 0;
        const int l = use[c] ? __ffs(todo) - 1 : 0;
        if (use[c]) todo &= todo - 1;
        rows_[c] = __shfl_sync(kFullMask, row, l);
        dsts_[c] = __shfl_sync(kFullMask, dst, l);
      }
      uint4 v[kDecRingCopies][4];
#pragma unroll
      for (int c = 0; c < kDecRingCopies; ++c) {
        if (!use[c]) continue;
        const uint8_t* kv = reinterpret_cast<const uint8_t*>(p.rows + rows_[c] * p.row_stride);
        const uint8_t* sc = reinterpret_cast<const uint8_t*>(score_base + rows_[c] * sstride);
        v[c][0] = ld_stream_v4(kv + 16 * lane);
        v[c][1] = ld_stream_v4(kv + 512 + 16 * lane);
        v[c][2] = ld_stream_v4(sc + 16 * lane);
        v[c][3] = ld_stream_v4(sc + 512 + 16 * lane);
      }
#pragma unroll
      for (int c = 0; c < kDecRingCopies; ++c) {
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

// The ring warps' share of this CTA's ring items (warp rw takes items
// rw + kDecRingWarps * (lane + 32 m)): items below n_cand are the round-robin
// requests r = blockIdx.x + grid * i, the rest this tile's listed
// ring-reading requests of n < 2R.  No row of the launch reads an entry these
// updates write.
__device__ __forceinline__ void ring_copy(const StoreParams& p, const DecodePlan& pl,
                                          const int* list, int n_list, int n_cand, int rw,
                                          int lane, unsigned cap) {
  const int n_items = n_cand + n_list;
  for (int i0 = rw; i0 < n_items; i0 += kDecRingWarps * 32) {
    const int i = i0 + kDecRingWarps * lane;
    RingWork rwk{0, 0, -1, 0};
    if (i < n_cand) rwk = ring_work(p, pl, (int)blockIdx.x + (int)gridDim.x * i, true, cap);
    else if (i < n_items) rwk = ring_work(p, pl, list[i - n_cand], false, cap);
    copy_ring_tokens(p, rwk, lane);
  }
}

// The slot holding output row k: the last r with base[r] <= k (slots
// without rows share their successor's base and are passed over).
__device__ __forceinline__ int find_slot(const unsigned* base, int n_slots, unsigned k) {
  int lo = 0, hi = n_slots - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (base[mid] <= k) lo = mid; else hi = mid - 1;
  }
  return lo;
}

template <int L, bool NORM, bool ROPE>
__global__ void __launch_bounds__(kDecThreads, 1)
compress_decode_kernel(const StoreParams p) {
  __shared__ DecodeShared sh;
  extern __shared__ __align__(16) int s_plan[];
  const DecodePlan pl{s_plan, s_plan + kMaxSlots, s_plan + 2 * kMaxSlots,
                      reinterpret_cast<unsigned*>(s_plan + 3 * kMaxSlots)};
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const long long tile0 = (long long)blockIdx.x * kDecRows;
  const unsigned cap = (unsigned)p.n_out;         // >= 1: rows below it are exact
  if (tid == 0) sh.n_list = 0;
  grid_dependency_wait();
  if (NORM && tid >= kDecPlanThreads && tid < kDecPlanThreads + 64)
    sh.norm_w[tid - kDecPlanThreads] = __ldg(reinterpret_cast<const uint4*>(p.norm_w) + tid - kDecPlanThreads);

  // ---- plan: slot metadata into shared memory, rows per slot, a saturating scan
  const int s0 = tid * kDecPer;
  const bool whole = s0 + kDecPer <= p.n_slots;   // s0 % 8 == 0: 32-byte aligned in shared memory
  unsigned rows[kDecPer];
  unsigned tsum = 0;
  if (tid < kDecPlanThreads && s0 < p.n_slots) {
    int first[kDecPer], count[kDecPer], start[kDecPer];
    load_slots(p, s0, first, count, start);
#pragma unroll
    for (int u = 0; u < kDecPer; ++u) {
      const long long n = rows_of_slot<2>(count[u], start[u]);
      rows[u] = n < (long long)cap ? (unsigned)n : cap;
      tsum = sat_add(tsum, rows[u], cap);
    }
    if (whole) {
      int4* f = reinterpret_cast<int4*>(pl.first + s0);
      int4* c = reinterpret_cast<int4*>(pl.count + s0);
      int4* t = reinterpret_cast<int4*>(pl.start + s0);
      f[0] = make_int4(first[0], first[1], first[2], first[3]);
      f[1] = make_int4(first[4], first[5], first[6], first[7]);
      c[0] = make_int4(count[0], count[1], count[2], count[3]);
      c[1] = make_int4(count[4], count[5], count[6], count[7]);
      t[0] = make_int4(start[0], start[1], start[2], start[3]);
      t[1] = make_int4(start[4], start[5], start[6], start[7]);
    } else {
#pragma unroll
      for (int u = 0; u < kDecPer; ++u) {
        if (s0 + u < p.n_slots) {
          pl.first[s0 + u] = first[u];
          pl.count[s0 + u] = count[u];
          pl.start[s0 + u] = start[u];
        }
      }
    }
  } else {
#pragma unroll
    for (int u = 0; u < kDecPer; ++u) rows[u] = 0;
  }
  unsigned incl = tsum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned t = __shfl_up_sync(kFullMask, incl, o);
    if (lane >= o) incl = sat_add(incl, t, cap);
  }
  if (warp < kDecPlanWarps && lane == 31) sh.wsum[warp] = incl;
  __syncthreads();
  if (tid < kDecPlanThreads) {
    const unsigned wv = lane < kDecPlanWarps ? sh.wsum[lane] : 0u;
    unsigned wincl = wv;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned t = __shfl_up_sync(kFullMask, wincl, o);
      if (lane >= o) wincl = sat_add(wincl, t, cap);
    }
    const unsigned wexcl = __shfl_up_sync(kFullMask, wincl, 1);
    const unsigned woff = __shfl_sync(kFullMask, lane == 0 ? 0u : wexcl, warp);
    const unsigned texcl = __shfl_up_sync(kFullMask, incl, 1);
    unsigned b = sat_add(woff, lane == 0 ? 0u : texcl, cap);
    unsigned lo[kDecPer];
#pragma unroll
    for (int u = 0; u < kDecPer; ++u) {
      lo[u] = b;
      b = sat_add(b, rows[u], cap);
    }
    if (whole) {
      uint4* dst = reinterpret_cast<uint4*>(pl.base + s0);
      dst[0] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      dst[1] = make_uint4(lo[4], lo[5], lo[6], lo[7]);
    } else {
#pragma unroll
      for (int u = 0; u < kDecPer; ++u)
        if (s0 + u < p.n_slots) pl.base[s0 + u] = lo[u];
    }
    const unsigned total = __shfl_sync(kFullMask, wincl, 31);   // every plan warp
    if (tid == 0) sh.total = total;
    // this tile's ring-reading requests with ring tokens (a slot whose first
    // row lies in the tile and sits at an odd start) of n < 2R: the ring
    // warps update them at once (their updates miss the entry the row reads);
    // those of n >= 2R rewrite that entry, so the row's own warp updates them
    // after its row
    if (p.ring != nullptr) {
      unsigned m = 0;
#pragma unroll
      for (int u = 0; u < kDecPer; ++u)
        m |= (unsigned)(rows[u] > 0 && lo[u] < cap && (long long)lo[u] >= tile0 &&
                        (long long)lo[u] < tile0 + kDecRows) << u;
      while (m) {
        const int r = s0 + __ffs(m) - 1;
        m &= m - 1;
        const int n = pl.count[r], p0 = pl.start[r];
        long long q, tsrc;
        if ((p0 & 1) && n < 2 * p.ring_size &&
            ring_tokens(n, p0, pl.first[r], p.ring_size, q, tsrc) > 0)
          sh.list[atomicAdd(&sh.n_list, 1)] = r;
      }
    }
  }
  __syncthreads();

  // ---- row warp w: its row's slot by binary search, every load of the row
  // issued, then (after the barrier) the arithmetic that needs them
  const bool row_warp = warp < kDecRows;
  const long long k = tile0 + warp;
  RowDesc d;
  d.state = kRowNone; d.pos = 0; d.r = 0; d.c = 0;
  RowIn<2, ROPE> in;
  int dest = -1;             // out_loc[k], or the page-table entry
  bool dest_ok = false;
  int own_ring = -1;         // request whose ring update (n >= 2R) follows this row
  if (row_warp && k < p.n_out) {
    d.state = kRowPad;
    if ((unsigned)k < sh.total) {
      const int r = find_slot(pl.base, p.n_slots, (unsigned)k);
      const int first = pl.first[r], p0 = pl.start[r];
      long long src;
      d = decode_row_desc<ROPE>(p, r, k - pl.base[r], first, p0, src);
      if (p.ring != nullptr && (p0 & 1) && (unsigned)k == pl.base[r] &&
          pl.count[r] >= 2 * p.ring_size)
        own_ring = r;
      if (d.state == kRowOk || d.state == kRowOkRing) {
        const __nv_bfloat16* score_base = p.score ? p.score : p.rows + kDim;
        const long long sstride = p.score ? p.score_stride : p.row_stride;
        const long long t1 = src + 1;      // the pair's second token (a new row)
        if (d.state == kRowOkRing) {
          // token p0 - 1 from the ring: kv | score, 2 KB (plain loads: the
          // ring warps write the ring in this launch)
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
        if (p.out_loc) {
          dest = __ldg(p.out_loc + k);
          dest_ok = true;
        } else {
          const int lp = d.c >> p.page_bits;
          dest_ok = d.c >= 0 && lp < p.max_pages;
          if (dest_ok) dest = __ldg(p.page_table + (long long)d.r * p.max_pages + lp);
        }
      }
    }
  }
  // ring warps: every item whose update no row of this launch can observe
  // (the round-robin requests, this tile's requests of n < 2R) right away,
  // in parallel with the rows
  const int n_cand = (int)blockIdx.x < p.n_slots
                         ? (p.n_slots - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
  if (row_warp) {
    float w[16];
    if constexpr (NORM) {
      unpack_bf16x8(sh.norm_w[lane], w);
      unpack_bf16x8(sh.norm_w[32 + lane], w + 8);
    }
    long long slot = 0;
    if (d.state == kRowOk || d.state == kRowOkRing) {
      if (p.out_loc) slot = dest;
      else slot = dest_ok ? ((long long)dest << p.page_bits) | (long long)(d.c & ((1 << p.page_bits) - 1))
                          : -1;
    }
    process_row<L, 2, NORM, ROPE>(p, k, d, slot, in, w, lane);
    // the update of a request of n >= 2R rewrites the entry this row read:
    // program order in this warp puts it after the row's loads
    if (own_ring >= 0) {
      RingWork rwk{0, 0, own_ring, 0};
      if (lane == 0)
        rwk.ntok = ring_tokens(pl.count[own_ring], pl.start[own_ring], pl.first[own_ring],
                               p.ring_size, rwk.q, rwk.src);
      copy_ring_tokens(p, rwk, lane);
    }
  } else if (p.ring != nullptr) {
    ring_copy(p, pl, sh.list, sh.n_list, n_cand, warp - kDecRows, lane, cap);
  }
  allow_dependent_launch();
}

template <int L, bool NORM, bool ROPE>
static cudaError_t launch_decode_variant(const StoreParams& p, cudaStream_t s) {
  auto kern = compress_decode_kernel<L, NORM, ROPE>;
  // the plan's 64 KB of slot arrays, set once per device (published after
  // the attribute call succeeded)
  static std::atomic<int> attr_set[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 64 || !attr_set[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kDecPlanBytes);
    if (e != cudaSuccess) return e;
    if (dev < 64) attr_set[dev].store(1, std::memory_order_release);
  }
  const int tiles = (int)(((long long)p.n_out + kDecRows - 1) / kDecRows);
  return launch_dependent(kern, tiles, kDecThreads, kDecPlanBytes, s, p);
}

template <int L>
static cudaError_t launch_decode_layout(const StoreParams& p, cudaStream_t s) {
  const bool norm = p.norm_w != nullptr, rope = p.freqs != nullptr;
  if (norm && rope) return launch_decode_variant<L, true, true>(p, s);
  if (norm) return launch_decode_variant<L, true, false>(p, s);
  if (rope) return launch_decode_variant<L, false, true>(p, s);
  return launch_decode_variant<L, false, false>(p, s);
}

cudaError_t launch_compress_decode(const StoreParams& p, int layout, cudaStream_t s) {
  if (layout == kV41) return launch_decode_layout<kV41>(p, s);
  if (layout == kV41Fp4) return launch_decode_layout<kV41Fp4>(p, s);
  return launch_decode_layout<kV4>(p, s);
}

}  // namespace dsv4kv
