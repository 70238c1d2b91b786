// Paged gather-dequant: a list of row ids -> bf16 rows.
//
// sglang PR #39652 "dsv4.1: compression, KV I/O, and metadata kernels",
// Summary (dequantize_k_cache_paged gains the KVLayout parameter; V4.1
// dequantizers for fp8 and fp4); sglang PR #45909: this is the sparse-prefill
// KV dequant whose result the layers sharing a kv_source reuse.
//
// One warp per gathered row, kRowsPerWarp rows in flight per warp: the id
// list is read once per group of rows (one lane per id, then shuffled), all
// code/scale loads of the group are issued before any conversion, and each
// output row is written as two fully coalesced 512-byte warp stores.  Lane l
// owns the 8-dim chunks l and l + 32, i.e. output bytes [16l, 16l+16) and
// [512 + 16l, ...), so every store instruction covers one contiguous half row.
#include "internal.cuh"
#include "quant.cuh"

namespace dsv4kv {

constexpr int kGatherWarps = 8;
constexpr int kGatherThreads = kGatherWarps * 32;
constexpr int kRowsPerWarp = 4;

template <int L>
__global__ void __launch_bounds__(kGatherThreads)
dequant_gather_kernel(const uint8_t* __restrict__ pool, long long pool_rows,
                      const int* __restrict__ ids, long long n,
                      __nv_bfloat16* __restrict__ out, int* err) {
  constexpr int RB = LayoutTraits<L>::kRowBytes;
  const int lane = threadIdx.x & 31;
  const long long gw = (long long)blockIdx.x * kGatherWarps + (threadIdx.x >> 5);
  const long long stride = (long long)gridDim.x * kGatherWarps * kRowsPerWarp;

  for (long long i0 = gw * kRowsPerWarp; i0 < n; i0 += stride) {
    int my_id = -1;
    if (lane < kRowsPerWarp && i0 + lane < n) my_id = __ldg(ids + i0 + lane);

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

template <int L>
static cudaError_t launch_layout(const uint8_t* pool, long long pool_rows, const int* ids,
                                 long long n, __nv_bfloat16* out, int* err, cudaStream_t s) {
  auto kern = dequant_gather_kernel<L>;
  int per_sm = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kGatherThreads, 0);
  if (e != cudaSuccess) return e;
  const long long rows_per_block = (long long)kGatherWarps * kRowsPerWarp;
  const long long want = (n + rows_per_block - 1) / rows_per_block;
  const long long cap = (long long)device_sm_count() * (per_sm > 0 ? per_sm : 1);
  const int grid = (int)(want < cap ? want : cap);
  kern<<<grid, kGatherThreads, 0, s>>>(pool, pool_rows, ids, n, out, err);
  return cudaGetLastError();
}

cudaError_t launch_dequant_gather(int layout, const uint8_t* pool, long long pool_rows,
                                  const int* ids, long long n, __nv_bfloat16* out, int* err,
                                  cudaStream_t s) {
  if (layout == kV41) return launch_layout<kV41>(pool, pool_rows, ids, n, out, err, s);
  return launch_layout<kV41Fp4>(pool, pool_rows, ids, n, out, err, s);
}

}  // namespace dsv4kv
