// Paged gather-dequant: a list of row ids -> bf16 rows (V41, V41_FP4, V4).
//
// sglang PR #39652 "dsv4.1: compression, KV I/O, and metadata kernels",
// Summary (dequantize_k_cache_paged gains the KVLayout parameter; V4.1
// dequantizers for fp8 and fp4); sglang PR #45909: this is the sparse-prefill
// KV dequant whose result the layers sharing a kv_source reuse.
//
// The fused variant (TOPK) reads the indexer's request-local top-k ids and
// maps them through the page table itself, so the sparse-prefill read needs
// no separate slot pass or slot buffer.
//
// One warp per gathered row, kRowsPerWarp rows in flight per warp: the id
// list is read once per group of rows (one lane per id, then shuffled), all
// code/scale loads of the group are issued before any conversion, and each
// output row is written as two fully coalesced 512-byte warp stores.  Lane l
// owns the 8-dim chunks l and l + 32, i.e. output bytes [16l, 16l+16) and
// [512 + 16l, ...), so every store instruction covers one contiguous half row.
#include <atomic>

#include "internal.cuh"
#include "launchers.cuh"
#include "quant.cuh"
#include "tma.cuh"

namespace dsv4kv {

// Streaming (evict-first) 16-byte store for the gathered rows: an output of
// about the L2's size that later kernels read at most once per layer, so it
// should not displace the pool rows and inputs still to be read.
__device__ __forceinline__ void st_stream_v4(void* p, uint4 v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};"
               :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}

constexpr int kGatherWarps = 8;
constexpr int kGatherThreads = kGatherWarps * 32;
constexpr int kRowsPerWarp = 4;

// Where a gathered row's pool slot comes from: an id list, or (TOPK) the
// request-local top-k ids mapped through the request's page table exactly as
// topk_to_slots does (flashinfer_sparse.py, _compressed_topk_to_slots).
struct GatherSrc {
  const int* ids;                  // [n] slots (plain gather)
  const int* topk;                 // [n_tok, k] request-local compressed ids, or nullptr:
  const int* fill_len;             //   short-context form, ids j < fill_len[t] ([n_tok])
  const int* token_to_req;         // [n_tok]
  const unsigned char* is_valid;   // [n_tok] or nullptr
  const int* page_table;           // [n_req, max_pages]
  int n_req, max_pages, page_bits, k;
  int* lens;                       // [n_tok], caller-zeroed, or nullptr
};

// Slot of request-local id `id` in page-table entry `phys` (64-bit, no wrap):
// -1 with one fault when the entry is negative or the slot does not fit int32.
__device__ __forceinline__ int page_slot(int phys, int id, int page_bits, int* err) {
  const long long slot =
      phys < 0 ? -1LL : ((long long)phys << page_bits) | (id & ((1 << page_bits) - 1));
  if (slot < 0 || slot > 2147483647LL) {
    if (err) atomicAdd(err, 1);
    return -1;
  }
  return (int)slot;
}

// Slot of gathered row i under TOPK; -1 = zero row.  Faults: a token whose
// request index is outside the table (counted once, at column 0), a page
// index past the table or a page entry that is no page (per entry).
__device__ __forceinline__ int topk_row_slot(const GatherSrc& g, long long i, int* err) {
  const long long t = i / g.k;
  const int c = (int)(i - t * g.k);
  const int r = __ldg(g.token_to_req + t);
  const int id = g.topk ? __ldg(g.topk + i) : (c < __ldg(g.fill_len + t) ? c : -1);
  if (r < 0 || r >= g.n_req) {
    if (c == 0 && err) atomicAdd(err, 1);
    return -1;
  }
  if ((g.is_valid && g.is_valid[t] == 0) || id < 0) return -1;
  const int lp = id >> g.page_bits;
  if (lp >= g.max_pages) {
    if (err) atomicAdd(err, 1);
    return -1;
  }
  return page_slot(__ldg(g.page_table + (long long)r * g.max_pages + lp), id, g.page_bits, err);
}

template <int L, bool TOPK>
__global__ void __launch_bounds__(kGatherThreads)
dequant_gather_kernel(const uint8_t* __restrict__ pool, long long pool_rows, const GatherSrc g,
                      long long n, __nv_bfloat16* __restrict__ out, int* err) {
  constexpr int RB = LayoutTraits<L>::kRowBytes;
  const int lane = threadIdx.x & 31;
  const long long gw = (long long)blockIdx.x * kGatherWarps + (threadIdx.x >> 5);
  const long long stride = (long long)gridDim.x * kGatherWarps * kRowsPerWarp;

  for (long long i0 = gw * kRowsPerWarp; i0 < n; i0 += stride) {
    int my_id = -1;
    if constexpr (!TOPK) {
      if (lane < kRowsPerWarp && i0 + lane < n) my_id = __ldg(g.ids + i0 + lane);
    } else {
      const bool mine = lane < kRowsPerWarp && i0 + lane < n;
      if (mine) my_id = topk_row_slot(g, i0 + lane, err);
      if (g.lens) {
        // count valid slots per token, one atomic per token present in the group
        const long long t = mine ? (i0 + lane) / g.k : -1;
        const long long t0 = __shfl_sync(kFullMask, t, 0);
        const unsigned same = __ballot_sync(kFullMask, mine && t == t0);
        const unsigned valid = __ballot_sync(kFullMask, mine && my_id >= 0);
        if (lane == 0 && (same & valid)) atomicAdd(g.lens + t0, __popc(same & valid));
        if (mine && t != t0 && my_id >= 0) atomicAdd(g.lens + t, 1);
      }
    }

    int id[kRowsPerWarp];
    bool valid[kRowsPerWarp];
#pragma unroll
    for (int t = 0; t < kRowsPerWarp; ++t) {
      id[t] = __shfl_sync(kFullMask, my_id, t);
      valid[t] = id[t] >= 0 && id[t] < pool_rows;
    }

    if constexpr (L == kV41) {
      uint2 c0[kRowsPerWarp], c1[kRowsPerWarp];
      uint4 sc[kRowsPerWarp];
#pragma unroll
      for (int t = 0; t < kRowsPerWarp; ++t) {
        if (valid[t]) {
          const uint8_t* row = pool + (long long)id[t] * RB;
          c0[t] = ld_stream_v2(row + 8 * lane);
          c1[t] = ld_stream_v2(row + 256 + 8 * lane);
          sc[t] = ld_stream_v4(row + LayoutTraits<kV41>::kCodeBytes);  // same 16 B for all lanes
        }
      }
#pragma unroll
      for (int t = 0; t < kRowsPerWarp; ++t) {
        const long long i = i0 + t;
        if (i >= n) break;
        uint4* o = reinterpret_cast<uint4*>(out + i * kDim);
        if (!valid[t]) {
          if (id[t] >= pool_rows && lane == 0 && err) atomicAdd(err, 1);
          st_stream_v4(o + lane, make_uint4(0, 0, 0, 0));
          st_stream_v4(o + 32 + lane, make_uint4(0, 0, 0, 0));
          continue;
        }
        // chunk l: dims 8l..8l+7, group l/4; chunk l+32: group 8 + l/4
        const int sh = 8 * ((lane >> 2) & 3);
        const uint32_t e0 = ((lane < 16 ? sc[t].x : sc[t].y) >> sh) & 0xFFu;
        const uint32_t e1 = ((lane < 16 ? sc[t].z : sc[t].w) >> sh) & 0xFFu;
        st_stream_v4(o + lane, dequant8_v41(c0[t], ue8m0_scale(e0)));
        st_stream_v4(o + 32 + lane, dequant8_v41(c1[t], ue8m0_scale(e1)));
      }
    } else if constexpr (L == kV4) {
      // half 0: codes of dims 8l.., group l/8; half 1: lanes 0..23 codes of
      // dims 256+8l.., group 4 + l/8; lanes 24..31 the stored bf16 rope dims
      uint2 c0[kRowsPerWarp], c1[kRowsPerWarp], c2[kRowsPerWarp], sc[kRowsPerWarp];
#pragma unroll
      for (int t = 0; t < kRowsPerWarp; ++t) {
        if (valid[t]) {
          const uint8_t* row = pool + (long long)id[t] * RB;
          c0[t] = ld_stream_v2(row + 8 * lane);
          if (lane < 24) {
            c1[t] = ld_stream_v2(row + 256 + 8 * lane);
          } else {
            c1[t] = ld_stream_v2(row + kNopeDim + 16 * (lane - 24));
            c2[t] = ld_stream_v2(row + kNopeDim + 16 * (lane - 24) + 8);
          }
          sc[t] = ld_stream_v2(row + LayoutTraits<kV4>::kCodeBytes);   // same 8 B for all lanes
        }
      }
#pragma unroll
      for (int t = 0; t < kRowsPerWarp; ++t) {
        const long long i = i0 + t;
        if (i >= n) break;
        uint4* o = reinterpret_cast<uint4*>(out + i * kDim);
        if (!valid[t]) {
          if (id[t] >= pool_rows && lane == 0 && err) atomicAdd(err, 1);
          st_stream_v4(o + lane, make_uint4(0, 0, 0, 0));
          st_stream_v4(o + 32 + lane, make_uint4(0, 0, 0, 0));
          continue;
        }
        const int g0 = lane >> 3, g1 = 4 + (lane >> 3);
        const uint32_t e0 = ((g0 < 4 ? sc[t].x : sc[t].y) >> (8 * (g0 & 3))) & 0xFFu;
        st_stream_v4(o + lane, dequant8_v41(c0[t], ue8m0_scale(e0)));
        if (lane < 24) {
          const uint32_t e1 = (sc[t].y >> (8 * (g1 & 3))) & 0xFFu;
          st_stream_v4(o + 32 + lane, dequant8_v41(c1[t], ue8m0_scale(e1)));
        } else {
          st_stream_v4(o + 32 + lane, make_uint4(c1[t].x, c1[t].y, c2[t].x, c2[t].y));
        }
      }
    } else {
      uint32_t c0[kRowsPerWarp], c1[kRowsPerWarp], s0[kRowsPerWarp], s1[kRowsPerWarp];
#pragma unroll
      for (int t = 0; t < kRowsPerWarp; ++t) {
        if (valid[t]) {
          const uint8_t* row = pool + (long long)id[t] * RB;
          c0[t] = ld_stream_u32(row + 4 * lane);
          c1[t] = ld_stream_u32(row + 128 + 4 * lane);
          // chunk l: group l/2; chunk l+32: group 16 + l/2
          s0[t] = __ldg(row + LayoutTraits<kV41Fp4>::kCodeBytes + (lane >> 1));
          s1[t] = __ldg(row + LayoutTraits<kV41Fp4>::kCodeBytes + 16 + (lane >> 1));
        }
      }
#pragma unroll
      for (int t = 0; t < kRowsPerWarp; ++t) {
        const long long i = i0 + t;
        if (i >= n) break;
        uint4* o = reinterpret_cast<uint4*>(out + i * kDim);
        if (!valid[t]) {
          if (id[t] >= pool_rows && lane == 0 && err) atomicAdd(err, 1);
          st_stream_v4(o + lane, make_uint4(0, 0, 0, 0));
          st_stream_v4(o + 32 + lane, make_uint4(0, 0, 0, 0));
          continue;
        }
        st_stream_v4(o + lane, dequant8_fp4(c0[t], e4m3_to_f32(s0[t])));
        st_stream_v4(o + 32 + lane, dequant8_fp4(c1[t], e4m3_to_f32(s1[t])));
      }
    }
  }
}

// ------------------------------------------------------------------ TMA form
// V41 and V41_FP4 rows are whole multiples of 16 bytes, so each gathered row
// can arrive by one cp.async.bulk copy.  Persistent CTAs of one producer warp
// and kTmaWarps consumer warps walk tiles of kTmaRows rows
// (tile = blockIdx.x + i * gridDim.x):
//  * the producer's lane l owns row l of a tile: it resolves the row's slot
//    (TOPK: the request-local id and the token's request are loaded two tiles
//    ahead, the page-table entry one tile ahead, so each tile waits on one
//    dependent load), counts faults and lens, publishes the slot in shared
//    memory and issues the row's copy into a kTmaStages-deep stage ring; each
//    consumer warp's rows complete on that warp's own mbarrier;
//  * consumer warp w owns rows 4w..4w+3 of every tile: it waits for them,
//    pulls codes and scales from shared memory into registers, releases the
//    stage and writes each bf16 row as two contiguous 512-byte warp stores.
// The rows in flight (two CTAs x 4 stages x 32 rows per SM) do not depend on
// registers, unlike the load-to-register form, whose warps wait on each
// group's loads before converting it.
constexpr int kTmaWarps = 8;
constexpr int kTmaThreads = (kTmaWarps + 1) * 32;
constexpr int kTmaRows = 32;                            // one per producer lane
constexpr int kTmaRowsPerWarp = kTmaRows / kTmaWarps;   // 4
constexpr int kTmaStages = 4;

template <int L>
struct GatherTile {
  static constexpr int kRB = LayoutTraits<L>::kRowBytes;
  static constexpr int kStageBytes = kTmaRows * kRB;
  static constexpr int kSlotOff = kTmaStages * kStageBytes;            // int slot per staged row
  static constexpr int kBarOff = kSlotOff + kTmaStages * kTmaRows * 4;
  static constexpr int kBarriers = kTmaStages * kTmaWarps + kTmaStages;  // full (stage x warp), empty
  static constexpr int kSmem = kBarOff + kBarriers * 8 + 16;             // + abort flag
  static_assert(kRB % 16 == 0 && kStageBytes % 16 == 0 && kBarOff % 8 == 0, "bulk-copy alignment");
};

// A TOPK row's inputs to the page-table step: its request-local id, the
// token's request, and whether the token is valid.
struct TopkRaw {
  int id;
  int r;
  bool live;   // row exists, token valid
};

__device__ __forceinline__ TopkRaw topk_raw(const GatherSrc& g, long long i, long long n) {
  TopkRaw a{-1, -1, false};
  if (i >= n) return a;
  const long long t = i / g.k;
  a.r = __ldg(g.token_to_req + t);
  if (g.topk) {
    a.id = __ldg(g.topk + i);
  } else {
    const int c = (int)(i - t * g.k);
    a.id = c < __ldg(g.fill_len + t) ? c : -1;
  }
  a.live = !g.is_valid || g.is_valid[t] != 0;
  return a;
}

// Lane l resolves row base + l (-1: zero row), with topk_row_slot's faults;
// TOPK also counts lens.  Called by the whole producer warp.
template <bool TOPK>
__device__ __forceinline__ int tma_row_slot(const GatherSrc& g, long long base, long long n,
                                            const TopkRaw& a, int lane, int* err) {
  const long long i = base + lane;
  int slot = -1;
  if constexpr (!TOPK) {
    if (i < n) slot = __ldg(g.ids + i);
  } else {
    const bool mine = i < n;
    if (mine) {
      if (a.r < 0 || a.r >= g.n_req) {
        if (i % g.k == 0 && err) atomicAdd(err, 1);
      } else if (a.live && a.id >= 0) {
        const int lp = a.id >> g.page_bits;
        if (lp >= g.max_pages) {
          if (err) atomicAdd(err, 1);
        } else {
          slot = page_slot(__ldg(g.page_table + (long long)a.r * g.max_pages + lp), a.id,
                           g.page_bits, err);
        }
      }
    }
    if (g.lens) {
      // count valid slots per token, one atomic per token present in the tile
      const long long t = mine ? i / g.k : -1;
      const long long t0 = __shfl_sync(kFullMask, t, 0);
      const unsigned same = __ballot_sync(kFullMask, mine && t == t0);
      const unsigned valid = __ballot_sync(kFullMask, mine && slot >= 0);
      if (lane == 0 && (same & valid)) atomicAdd(g.lens + t0, __popc(same & valid));
      if (mine && t != t0 && slot >= 0) atomicAdd(g.lens + t, 1);
    }
  }
  return slot;
}

template <int L, bool TOPK>
__global__ void __launch_bounds__(kTmaThreads, 2)
dequant_gather_tma_kernel(const uint8_t* __restrict__ pool, long long pool_rows, const GatherSrc g,
                          long long n, __nv_bfloat16* __restrict__ out, int* err) {
  using GT = GatherTile<L>;
  extern __shared__ __align__(128) uint8_t smem[];
  int* s_slot = reinterpret_cast<int*>(smem + GT::kSlotOff);
  uint64_t* s_full = reinterpret_cast<uint64_t*>(smem + GT::kBarOff);
  uint64_t* s_empty = s_full + kTmaStages * kTmaWarps;
  int* s_abort = reinterpret_cast<int*>(s_empty + kTmaStages);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kTmaStages * kTmaWarps; ++i) mbar_init(&s_full[i], 1);
    for (int s = 0; s < kTmaStages; ++s) mbar_init(&s_empty[s], kTmaWarps);
    *s_abort = 0;
    mbar_fence_init();
  }
  __syncthreads();
  grid_dependency_wait();
  volatile int* abort = s_abort;
  const long long n_tiles = (n + kTmaRows - 1) / kTmaRows;
  const long long step = gridDim.x;

  if (warp == kTmaWarps) {
    // ------------------------------------------------------------ producer
    const uint64_t pol = policy_evict_first();
    long long tile = blockIdx.x;
    TopkRaw raw_next{-1, -1, false};
    int slot = -1;
    if constexpr (TOPK) {
      slot = tma_row_slot<TOPK>(g, tile * kTmaRows, n,
                                topk_raw(g, tile * kTmaRows + lane, n), lane, err);
      raw_next = topk_raw(g, (tile + step) * kTmaRows + lane, n);
    } else {
      slot = tma_row_slot<TOPK>(g, tile * kTmaRows, n, raw_next, lane, err);
    }
    long long it = 0;
    for (; tile < n_tiles; tile += step, ++it) {
      TopkRaw raw_after{-1, -1, false};
      if constexpr (TOPK) raw_after = topk_raw(g, (tile + 2 * step) * kTmaRows + lane, n);
      const int s = (int)(it % kTmaStages);
      const uint32_t use = (uint32_t)(it / kTmaStages);
      if (use > 0 && !mbar_wait(&s_empty[s], (use - 1) & 1u, abort, err)) break;
      const bool valid = slot >= 0 && slot < pool_rows;
      if (slot >= pool_rows && err) atomicAdd(err, 1);
      s_slot[s * kTmaRows + lane] = valid ? slot : -1;
      uint64_t* bar = &s_full[s * kTmaWarps + lane / kTmaRowsPerWarp];
      uint32_t bytes = valid ? (uint32_t)GT::kRB : 0u;
#pragma unroll
      for (int o = 1; o < kTmaRowsPerWarp; o <<= 1) bytes += __shfl_xor_sync(kFullMask, bytes, o);
      __syncwarp();
      if (lane % kTmaRowsPerWarp == 0) mbar_arrive_expect_tx(bar, bytes);
      __syncwarp();
      if (valid)
        bulk_g2s(smem + s * GT::kStageBytes + lane * GT::kRB, pool + (long long)slot * GT::kRB,
                 GT::kRB, bar, pol);
      // the next tile's slots, while this tile's copies are in flight
      slot = tma_row_slot<TOPK>(g, (tile + step) * kTmaRows, n, raw_next, lane, err);
      raw_next = raw_after;
    }
    // every issued copy has landed before the CTA may exit (bounded)
    if (lane < kTmaWarps) {
      for (int s = 0; s < kTmaStages && s < it; ++s) {
        const uint32_t last_use = (uint32_t)((it - 1 - s) / kTmaStages);
        uint64_t* bar = &s_full[s * kTmaWarps + lane];
        for (uint32_t i = 0; i < kSpinLimit && !mbar_try_wait(bar, last_use & 1u); ++i) {
        }
      }
    }
    allow_dependent_launch();
    return;
  }

  // ------------------------------------------------------------ consumers
  long long it = 0;
  for (long long tile = blockIdx.x; tile < n_tiles; tile += step, ++it) {
    const int s = (int)(it % kTmaStages);
    const uint32_t use = (uint32_t)(it / kTmaStages);
    if (!mbar_wait(&s_full[s * kTmaWarps + warp], use & 1u, abort, err)) break;
    const uint8_t* stage = smem + s * GT::kStageBytes;
    int sl[kTmaRowsPerWarp];
    if constexpr (L == kV41) {
      uint2 c0[kTmaRowsPerWarp], c1[kTmaRowsPerWarp];
      uint4 sc[kTmaRowsPerWarp];
#pragma unroll
      for (int q = 0; q < kTmaRowsPerWarp; ++q) {
        const int r = warp * kTmaRowsPerWarp + q;
        sl[q] = s_slot[s * kTmaRows + r];
        if (sl[q] >= 0) {
          const uint8_t* row = stage + r * GT::kRB;
          c0[q] = *reinterpret_cast<const uint2*>(row + 8 * lane);
          c1[q] = *reinterpret_cast<const uint2*>(row + 256 + 8 * lane);
          sc[q] = *reinterpret_cast<const uint4*>(row + LayoutTraits<kV41>::kCodeBytes);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_empty[s]);
#pragma unroll
      for (int q = 0; q < kTmaRowsPerWarp; ++q) {
        const long long i = tile * kTmaRows + warp * kTmaRowsPerWarp + q;
        if (i >= n) break;
        uint4* o = reinterpret_cast<uint4*>(out + i * kDim);
        if (sl[q] < 0) {
          st_stream_v4(o + lane, make_uint4(0, 0, 0, 0));
          st_stream_v4(o + 32 + lane, make_uint4(0, 0, 0, 0));
          continue;
        }
        // chunk l: dims 8l..8l+7, group l/4; chunk l+32: group 8 + l/4
        const int sh = 8 * ((lane >> 2) & 3);
        const uint32_t e0 = ((lane < 16 ? sc[q].x : sc[q].y) >> sh) & 0xFFu;
        const uint32_t e1 = ((lane < 16 ? sc[q].z : sc[q].w) >> sh) & 0xFFu;
        st_stream_v4(o + lane, dequant8_v41(c0[q], ue8m0_scale(e0)));
        st_stream_v4(o + 32 + lane, dequant8_v41(c1[q], ue8m0_scale(e1)));
      }
    } else {
      uint32_t c0[kTmaRowsPerWarp], c1[kTmaRowsPerWarp], s0[kTmaRowsPerWarp], s1[kTmaRowsPerWarp];
#pragma unroll
      for (int q = 0; q < kTmaRowsPerWarp; ++q) {
        const int r = warp * kTmaRowsPerWarp + q;
        sl[q] = s_slot[s * kTmaRows + r];
        if (sl[q] >= 0) {
          const uint8_t* row = stage + r * GT::kRB;
          c0[q] = *reinterpret_cast<const uint32_t*>(row + 4 * lane);
          c1[q] = *reinterpret_cast<const uint32_t*>(row + 128 + 4 * lane);
          // chunk l: group l/2; chunk l+32: group 16 + l/2
          s0[q] = row[LayoutTraits<kV41Fp4>::kCodeBytes + (lane >> 1)];
          s1[q] = row[LayoutTraits<kV41Fp4>::kCodeBytes + 16 + (lane >> 1)];
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_empty[s]);
#pragma unroll
      for (int q = 0; q < kTmaRowsPerWarp; ++q) {
        const long long i = tile * kTmaRows + warp * kTmaRowsPerWarp + q;
        if (i >= n) break;
        uint4* o = reinterpret_cast<uint4*>(out + i * kDim);
        if (sl[q] < 0) {
          st_stream_v4(o + lane, make_uint4(0, 0, 0, 0));
          st_stream_v4(o + 32 + lane, make_uint4(0, 0, 0, 0));
          continue;
        }
        st_stream_v4(o + lane, dequant8_fp4(c0[q], e4m3_to_f32(s0[q])));
        st_stream_v4(o + 32 + lane, dequant8_fp4(c1[q], e4m3_to_f32(s1[q])));
      }
    }
  }
  allow_dependent_launch();
}

template <int L, bool TOPK>
static cudaError_t launch_tma(const uint8_t* pool, long long pool_rows, const GatherSrc& g,
                              long long n, __nv_bfloat16* out, int* err, cudaStream_t s) {
  using GT = GatherTile<L>;
  auto kern = dequant_gather_tma_kernel<L, TOPK>;
  static std::atomic<int> occupancy[64];   // resident CTAs per SM, per device (attribute set then)
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int per_sm = dev < 64 ? occupancy[dev].load(std::memory_order_relaxed) : 0;
  if (per_sm <= 0) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, GT::kSmem);
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kTmaThreads, GT::kSmem);
    if (e != cudaSuccess) return e;
    if (dev < 64 && per_sm > 0) occupancy[dev].store(per_sm, std::memory_order_relaxed);
  }
  const long long tiles = (n + kTmaRows - 1) / kTmaRows;
  const long long cap = (long long)device_sm_count() * (per_sm > 0 ? per_sm : 1);
  const int grid = (int)(tiles < cap ? tiles : cap);
  return launch_dependent(kern, grid, kTmaThreads, GT::kSmem, s, pool, pool_rows, g, n, out, err);
}

template <int L, bool TOPK>
static cudaError_t launch_layout(const uint8_t* pool, long long pool_rows, const GatherSrc& g,
                                 long long n, __nv_bfloat16* out, int* err, cudaStream_t s) {
  auto kern = dequant_gather_kernel<L, TOPK>;
  // resident CTAs per SM, queried once per device (no dynamic shared memory)
  static std::atomic<int> occupancy[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int per_sm = dev < 64 ? occupancy[dev].load(std::memory_order_relaxed) : 0;
  if (per_sm <= 0) {
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kGatherThreads, 0);
    if (e != cudaSuccess) return e;
    if (dev < 64) occupancy[dev].store(per_sm, std::memory_order_relaxed);
  }
  const long long rows_per_block = (long long)kGatherWarps * kRowsPerWarp;
  const long long want = (n + rows_per_block - 1) / rows_per_block;
  const long long cap = (long long)device_sm_count() * (per_sm > 0 ? per_sm : 1);
  const int grid = (int)(want < cap ? want : cap);
  kern<<<grid, kGatherThreads, 0, s>>>(pool, pool_rows, g, n, out, err);
  return cudaGetLastError();
}

cudaError_t launch_dequant_gather(int layout, const uint8_t* pool, long long pool_rows,
                                  const int* ids, long long n, __nv_bfloat16* out, int* err,
                                  cudaStream_t s) {
  GatherSrc g{};
  g.ids = ids;
  if (layout == kV41) return launch_tma<kV41, false>(pool, pool_rows, g, n, out, err, s);
  if (layout == kV4) return launch_layout<kV4, false>(pool, pool_rows, g, n, out, err, s);
  return launch_tma<kV41Fp4, false>(pool, pool_rows, g, n, out, err, s);
}

cudaError_t launch_dequant_gather_topk(int layout, const uint8_t* pool, long long pool_rows,
                                       const int* topk, const int* fill_len, int n_tok, int k,
                                       const int* token_to_req, const unsigned char* is_valid,
                                       const int* page_table, int n_req, int max_pages,
                                       int page_bits, __nv_bfloat16* out, int* lens, int* err,
                                       cudaStream_t s) {
  GatherSrc g{};
  g.topk = topk;
  g.fill_len = fill_len;
  g.token_to_req = token_to_req;
  g.is_valid = is_valid;
  g.page_table = page_table;
  g.n_req = n_req;
  g.max_pages = max_pages;
  g.page_bits = page_bits;
  g.k = k;
  g.lens = lens;
  const long long n = (long long)n_tok * k;
  if (layout == kV41) return launch_tma<kV41, true>(pool, pool_rows, g, n, out, err, s);
  if (layout == kV4) return launch_layout<kV4, true>(pool, pool_rows, g, n, out, err, s);
  return launch_tma<kV41Fp4, true>(pool, pool_rows, g, n, out, err, s);
}

}  // namespace dsv4kv
