// Fused compressor: (ratio-2 pair pooling) -> RMSNorm -> RoPE -> store_row
// -> paged write, one warp per output row, in one launch.
//
// sglang PR #39652 "dsv4.1: compression, KV I/O, and metadata kernels",
// Summary (c1/c2 bullet): the ratio-1 / ratio-2 compressors do pair-pooling
// (ratio 2), RMSNorm, RoPE and the main-KV write in one launch, returning the
// pre-RoPE latent; out_loc == 0 marks a padded graph row.  The review's
// cleanup of the c2 kernel issues the RoPE frequency load before the softmax
// and the RMSNorm reduction so its latency overlaps them; this kernel does
// the same.
// sglang PR #46230: the launch reads low_ratio_extend_offsets (int32 [2,
// request slots]: first row, row count) on the device, so it can sit inside
// a CUDA graph whose offsets are refreshed in place; ratio-2 input is the
// fused | kv | score | projection.
//
// Work decomposition.  Each CTA first turns the per-slot row counts into an
// exclusive prefix (shared memory), then its warps walk output rows k in a
// grid-stride loop: binary search k -> request slot r, row j = k - base[r].
// Lane l holds dims [16l, 16l+16) of the row in registers; every global
// access is a 16-byte vector access, and a warp instruction touches 512
// contiguous bytes.  All loads of a row (kv, score, RoPE frequencies) are
// issued before any arithmetic.
#include "internal.cuh"
#include "quant.cuh"

namespace dsv4kv {

constexpr int kStoreWarps = 8;
constexpr int kStoreThreads = kStoreWarps * 32;

// base[i] = sum_{r < i} max(count_r, 0) / RATIO for i in [0, n_slots]
template <int RATIO>
__device__ void block_scan_counts(const int* __restrict__ ext, int n_slots, long long* base) {
  __shared__ long long s_warp[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nt = blockDim.x, nwarps = nt >> 5;
  const int per = (n_slots + nt - 1) / nt;
  const int beg = min(tid * per, n_slots), end = min(beg + per, n_slots);
  long long local = 0;
  for (int i = beg; i < end; ++i) local += max(ext[n_slots + i], 0) / RATIO;
  long long v = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long t = __shfl_up_sync(kFullMask, v, o);
    if (lane >= o) v += t;
  }
  if (lane == 31) s_warp[warp] = v;
  __syncthreads();
  if (warp == 0) {
    long long wv = lane < nwarps ? s_warp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long t = __shfl_up_sync(kFullMask, wv, o);
      if (lane >= o) wv += t;
    }
    s_warp[lane] = wv;
  }
  __syncthreads();
  long long excl = v - local + (warp > 0 ? s_warp[warp - 1] : 0);
  for (int i = beg; i < end; ++i) {
    base[i] = excl;
    excl += max(ext[n_slots + i], 0) / RATIO;
  }
  if (tid == nt - 1) base[n_slots] = excl;
}

// fast exp2 / reciprocal: relative error ~2^-22, far inside the 1e-5
// tolerance on the pre-quant row; exact at 0 and for powers of two
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void zero_row_outputs(const StoreParams& p, long long k, int lane) {
  if (p.latent_out) {
    uint4* d = reinterpret_cast<uint4*>(p.latent_out + k * kDim + 16 * lane);
    d[0] = make_uint4(0, 0, 0, 0);
    d[1] = make_uint4(0, 0, 0, 0);
  }
  if (p.prequant_out) {
    float4* d = reinterpret_cast<float4*>(p.prequant_out + k * kDim + 16 * lane);
#pragma unroll
    for (int i = 0; i < 4; ++i) d[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

template <int L, int RATIO, bool NORM, bool ROPE>
__global__ void __launch_bounds__(kStoreThreads)
compress_store_kernel(const StoreParams p) {
  extern __shared__ long long s_base[];  // n_slots + 1
  block_scan_counts<RATIO>(p.ext, p.n_slots, s_base);
  __syncthreads();
  const long long total = s_base[p.n_slots];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;

  float w[16];
  if constexpr (NORM) {
    const uint4* wp = reinterpret_cast<const uint4*>(p.norm_w + 16 * lane);
    unpack_bf16x8(__ldg(wp), w);
    unpack_bf16x8(__ldg(wp + 1), w + 8);
  }
  const __nv_bfloat16* score_base = p.score ? p.score : p.rows + kDim;
  const long long sstride = p.score ? p.score_stride : p.row_stride;
  const long long page_mask = (1LL << p.page_bits) - 1;

  for (long long k = (long long)blockIdx.x * kStoreWarps + warp; k < p.n_out;
       k += (long long)gridDim.x * kStoreWarps) {
    if (k >= total) {  // padding row: no source, nothing stored
      zero_row_outputs(p, k, lane);
      continue;
    }
    int lo = 0, hi = p.n_slots - 1;
    while (lo < hi) {  // last slot whose base <= k (empty slots share a base)
      const int mid = (lo + hi + 1) >> 1;
      if (s_base[mid] <= k) lo = mid; else hi = mid - 1;
    }
    const int r = lo;
    const long long j = k - s_base[r];
    const long long first = p.ext[r];
    const long long src = first + (long long)RATIO * j;
    const long long pos = (long long)RATIO * j;
    bool ok = src >= 0 && src + RATIO <= p.n_rows;
    if (ROPE) ok = ok && pos < p.max_pos;
    if (!ok) {
      if (lane == 0 && p.err) atomicAdd(p.err, 1);
      zero_row_outputs(p, k, lane);
      continue;
    }
    // destination (independent of the arithmetic; fetched early)
    long long slot;
    if (p.out_loc) {
      slot = p.out_loc[k];
    } else {
      const long long lp = j >> p.page_bits;
      slot = lp < p.max_pages
                 ? ((long long)p.page_table[(long long)r * p.max_pages + lp] << p.page_bits) | (j & page_mask)
                 : -1;
    }

    // ---- loads: everything this row needs, issued together
    const __nv_bfloat16* kv0 = p.rows + src * p.row_stride + 16 * lane;
    uint4 a0 = ld_stream_v4(kv0), a1 = ld_stream_v4(kv0 + 8);
    uint4 b0, b1, c0, c1, d0, d1;
    if constexpr (RATIO == 2) {
      const __nv_bfloat16* kv1 = kv0 + p.row_stride;
      const __nv_bfloat16* s0 = score_base + src * sstride + 16 * lane;
      const __nv_bfloat16* s1 = s0 + sstride;
      b0 = ld_stream_v4(kv1); b1 = ld_stream_v4(kv1 + 8);
      c0 = ld_stream_v4(s0);  c1 = ld_stream_v4(s0 + 8);
      d0 = ld_stream_v4(s1);  d1 = ld_stream_v4(s1 + 8);
    }
    float4 fr[4];
    if (ROPE && lane >= 28) {
      const float4* fp = reinterpret_cast<const float4*>(p.freqs + pos * kRopeDim + 16 * (lane - 28));
#pragma unroll
      for (int i = 0; i < 4; ++i) fr[i] = __ldg(fp + i);
    }

    // ---- pool
    float x[16];
    unpack_bf16x8(a0, x);
    unpack_bf16x8(a1, x + 8);
    if constexpr (RATIO == 2) {
      float k1[16], s0[16], s1[16];
      unpack_bf16x8(b0, k1); unpack_bf16x8(b1, k1 + 8);
      unpack_bf16x8(c0, s0); unpack_bf16x8(c1, s0 + 8);
      unpack_bf16x8(d0, s1); unpack_bf16x8(d1, s1 + 8);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        // softmax over the pair: the larger score gets 1/(1+e), the other
        // e/(1+e), e = exp(-|s0 - s1|)
        const float d = s0[i] - s1[i];
        const float e = ex2_approx(-fabsf(d) * 1.4426950408889634f);
        const float wb = rcp_approx(1.f + e);
        const float ws = e * wb;
        x[i] = d >= 0.f ? fmaf(wb, x[i], ws * k1[i]) : fmaf(ws, x[i], wb * k1[i]);
      }
    }
    // ---- RMSNorm over all 512 dims
    if constexpr (NORM) {
      float ss = 0.f;
#pragma unroll
      for (int i = 0; i < 16; ++i) ss = fmaf(x[i], x[i], ss);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(kFullMask, ss, o);
      const float inv = rsqrtf(fmaf(ss, 1.f / kDim, p.eps));
#pragma unroll
      for (int i = 0; i < 16; ++i) x[i] = (x[i] * inv) * w[i];
    }
    if (p.latent_out) {  // post-norm, pre-RoPE
      uint4* d = reinterpret_cast<uint4*>(p.latent_out + k * kDim + 16 * lane);
      d[0] = pack_bf16x8(x);
      d[1] = pack_bf16x8(x + 8);
    }
    // ---- RoPE on dims 448..511: interleaved pairs rotated by (cos, sin)
    if (ROPE && lane >= 28) {
      const float* f = reinterpret_cast<const float*>(fr);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float c = f[2 * i], s = f[2 * i + 1];
        const float a = x[2 * i], b = x[2 * i + 1];
        x[2 * i] = fmaf(a, c, -b * s);
        x[2 * i + 1] = fmaf(a, s, b * c);
      }
    }
    if (p.prequant_out) {
      float4* d = reinterpret_cast<float4*>(p.prequant_out + k * kDim + 16 * lane);
#pragma unroll
      for (int i = 0; i < 4; ++i) d[i] = make_float4(x[4 * i], x[4 * i + 1], x[4 * i + 2], x[4 * i + 3]);
    }
    // ---- quantize + paged store
    if (slot == 0) continue;  // padded graph row
    if (slot < 0 || slot >= p.pool_rows) {
      if (lane == 0 && p.err) atomicAdd(p.err, 1);
      continue;
    }
    const PagedKV<L> kv{p.pool, p.page_bits};
    store_row_lane<L>(x, kv.row(slot), lane);
  }
}

template <int L, int RATIO, bool NORM, bool ROPE>
static cudaError_t launch_variant(const StoreParams& p, cudaStream_t stream) {
  auto kern = compress_store_kernel<L, RATIO, NORM, ROPE>;
  const size_t smem = sizeof(long long) * (size_t)(p.n_slots + 1);
  int per_sm = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kStoreThreads, smem);
  if (e != cudaSuccess) return e;
  const long long want = ((long long)p.n_out + kStoreWarps - 1) / kStoreWarps;
  const long long cap = (long long)device_sm_count() * (per_sm > 0 ? per_sm : 1);
  const int grid = (int)(want < cap ? want : cap);
  kern<<<grid, kStoreThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

template <int L, int RATIO>
static cudaError_t launch_norm_rope(const StoreParams& p, cudaStream_t s) {
  const bool norm = p.norm_w != nullptr, rope = p.freqs != nullptr;
  if (norm && rope) return launch_variant<L, RATIO, true, true>(p, s);
  if (norm) return launch_variant<L, RATIO, true, false>(p, s);
  if (rope) return launch_variant<L, RATIO, false, true>(p, s);
  return launch_variant<L, RATIO, false, false>(p, s);
}

cudaError_t launch_compress_store(const StoreParams& p, int layout, int ratio, cudaStream_t s) {
  if (layout == kV41) return ratio == 1 ? launch_norm_rope<kV41, 1>(p, s) : launch_norm_rope<kV41, 2>(p, s);
  return ratio == 1 ? launch_norm_rope<kV41Fp4, 1>(p, s) : launch_norm_rope<kV41Fp4, 2>(p, s);
}

}  // namespace dsv4kv
