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
#include "quant.cuh"

namespace dsv4kv {

constexpr int kGatherWarps = 8;
constexpr int kGatherThreads = kGatherWarps * 32;
constexpr int kRowsPerWarp = 4;

// Where a gathered row's pool slot comes from: an id list, or (TOPK) the
// request-local top-k ids mapped through the request's page table exactly as
// topk_to_slots does (flashinfer_sparse.py, _compressed_topk_to_slots).
struct GatherSrc {
  const int* ids;                  // [n] slots (plain gather)
  const int* topk;                 // [n_tok, k] request-local compressed ids
  const int* token_to_req;         // [n_tok]
  const unsigned char* is_valid;   // [n_tok] or nullptr
  const int* page_table;           // [n_req, max_pages]
  int n_req, max_pages, page_bits, k;
  int* lens;                       // [n_tok], caller-zeroed, or nullptr
};

// Slot of gathered row i under TOPK; -1 = zero row.  Faults: a token whose
// request index is outside the table (counted once, at column 0), a page
// index past the table (per entry).
__device__ __forceinline__ int topk_row_slot(const GatherSrc& g, long long i, int* err) {
  const long long t = i / g.k;
  const int c = (int)(i - t * g.k);
  const int r = __ldg(g.token_to_req + t);
  const int id = __ldg(g.topk + i);
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
  const unsigned phys = (unsigned)__ldg(g.page_table + (long long)r * g.max_pages + lp);
  return (int)((phys << g.page_bits) | ((unsigned)id & ((1u << g.page_bits) - 1u)));
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
          o[lane] = make_uint4(0, 0, 0, 0);
          o[32 + lane] = make_uint4(0, 0, 0, 0);
          continue;
        }
        // chunk l: dims 8l..8l+7, group l/4; chunk l+32: group 8 + l/4
        const int sh = 8 * ((lane >> 2) & 3);
        const uint32_t e0 = ((lane < 16 ? sc[t].x : sc[t].y) >> sh) & 0xFFu;
        const uint32_t e1 = ((lane < 16 ? sc[t].z : sc[t].w) >> sh) & 0xFFu;
        o[lane] = dequant8_v41(c0[t], ue8m0_scale(e0));
        o[32 + lane] = dequant8_v41(c1[t], ue8m0_scale(e1));
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
          o[lane] = make_uint4(0, 0, 0, 0);
          o[32 + lane] = make_uint4(0, 0, 0, 0);
          continue;
        }
        const int g0 = lane >> 3, g1 = 4 + (lane >> 3);
        const uint32_t e0 = ((g0 < 4 ? sc[t].x : sc[t].y) >> (8 * (g0 & 3))) & 0xFFu;
        o[lane] = dequant8_v41(c0[t], ue8m0_scale(e0));
        if (lane < 24) {
          const uint32_t e1 = (sc[t].y >> (8 * (g1 & 3))) & 0xFFu;
          o[32 + lane] = dequant8_v41(c1[t], ue8m0_scale(e1));
        } else {
          o[32 + lane] = make_uint4(c1[t].x, c1[t].y, c2[t].x, c2[t].y);
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
          o[lane] = make_uint4(0, 0, 0, 0);
          o[32 + lane] = make_uint4(0, 0, 0, 0);
          continue;
        }
        o[lane] = dequant8_fp4(c0[t], e4m3_to_f32(s0[t]));
        o[32 + lane] = dequant8_fp4(c1[t], e4m3_to_f32(s1[t]));
      }
    }
  }
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
  if (layout == kV41) return launch_layout<kV41, false>(pool, pool_rows, g, n, out, err, s);
  if (layout == kV4) return launch_layout<kV4, false>(pool, pool_rows, g, n, out, err, s);
  return launch_layout<kV41Fp4, false>(pool, pool_rows, g, n, out, err, s);
}

cudaError_t launch_dequant_gather_topk(int layout, const uint8_t* pool, long long pool_rows,
                                       const int* topk, int n_tok, int k, const int* token_to_req,
                                       const unsigned char* is_valid, const int* page_table,
                                       int n_req, int max_pages, int page_bits,
                                       __nv_bfloat16* out, int* lens, int* err, cudaStream_t s) {
  GatherSrc g{};
  g.topk = topk;
  g.token_to_req = token_to_req;
  g.is_valid = is_valid;
  g.page_table = page_table;
  g.n_req = n_req;
  g.max_pages = max_pages;
  g.page_bits = page_bits;
  g.k = k;
  g.lens = lens;
  const long long n = (long long)n_tok * k;
  if (layout == kV41) return launch_layout<kV41, true>(pool, pool_rows, g, n, out, err, s);
  if (layout == kV4) return launch_layout<kV4, true>(pool, pool_rows, g, n, out, err, s);
  return launch_layout<kV41Fp4, true>(pool, pool_rows, g, n, out, err, s);
}

}  // namespace dsv4kv
