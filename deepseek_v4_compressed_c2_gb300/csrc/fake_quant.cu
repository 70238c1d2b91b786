// Fake quantization of latent rows: bf16 -> store_row -> dequant -> bf16, no
// pool in between.
//
// sglang PR #39652 "dsv4.1: compression, KV I/O, and metadata kernels",
// Summary / test table (fake_quant_compressed_kv, fake_quant_fp4): the
// quantize-then-dequantize of compressed-KV rows in one pass, the values the
// attention would read back from the cache.
//
// One warp per row.  The row goes through the very store_row_split the
// compressor uses, into a 16-byte aligned row buffer in shared memory, and
// comes back through the same per-layout decode as the gather, so the result
// equals a store followed by a gather of that row bit for bit.  A lane reads
// and writes only its own 16-byte chunks (dims 8l..8l+7 and 256+8l..), so
// in == out is allowed.
#include <atomic>

#include "internal.cuh"
#include "launchers.cuh"
#include "quant.cuh"

namespace dsv4kv {

constexpr int kFqWarps = 8;
constexpr int kFqRowBuf = 592;   // the largest row (584 B) rounded up to 16

template <int L>
__global__ void __launch_bounds__(kFqWarps * 32)
fake_quant_kernel(const __nv_bfloat16* in, long long n, long long in_stride, __nv_bfloat16* out) {
  __shared__ __align__(16) uint8_t s_row[kFqWarps][kFqRowBuf];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* row = s_row[warp];
  for (long long i = (long long)blockIdx.x * kFqWarps + warp; i < n;
       i += (long long)gridDim.x * kFqWarps) {
    const uint4* src = reinterpret_cast<const uint4*>(in + i * in_stride);
    float x[16];
    unpack_bf16x8(src[lane], x);
    unpack_bf16x8(src[32 + lane], x + 8);
    store_row_split<L>(x, row, lane);
    __syncwarp();
    uint4 lo, hi;
    if constexpr (L == kV41) {
      const uint2 c0 = *reinterpret_cast<const uint2*>(row + 8 * lane);
      const uint2 c1 = *reinterpret_cast<const uint2*>(row + 256 + 8 * lane);
      const uint4 sc = *reinterpret_cast<const uint4*>(row + LayoutTraits<kV41>::kCodeBytes);
      // chunk l: dims 8l..8l+7, group l/4; chunk l+32: group 8 + l/4
      const int sh = 8 * ((lane >> 2) & 3);
      lo = dequant8_v41(c0, ue8m0_scale(((lane < 16 ? sc.x : sc.y) >> sh) & 0xFFu));
      hi = dequant8_v41(c1, ue8m0_scale(((lane < 16 ? sc.z : sc.w) >> sh) & 0xFFu));
    } else if constexpr (L == kV41Fp4) {
      const uint32_t c0 = *reinterpret_cast<const uint32_t*>(row + 4 * lane);
      const uint32_t c1 = *reinterpret_cast<const uint32_t*>(row + 128 + 4 * lane);
      // chunk l: group l/2; chunk l+32: group 16 + l/2
      const uint32_t s0 = row[LayoutTraits<kV41Fp4>::kCodeBytes + (lane >> 1)];
      const uint32_t s1 = row[LayoutTraits<kV41Fp4>::kCodeBytes + 16 + (lane >> 1)];
      lo = dequant8_fp4(c0, e4m3_to_f32(s0));
      hi = dequant8_fp4(c1, e4m3_to_f32(s1));
    } else {
      // half 0: dims 8l.., group l/8; half 1: lanes 0..23 dims 256+8l..,
      // group 4 + l/8; lanes 24..31 the stored bf16 rope dims
      const uint2 c0 = *reinterpret_cast<const uint2*>(row + 8 * lane);
      const uint2 sc = *reinterpret_cast<const uint2*>(row + LayoutTraits<kV4>::kCodeBytes);
      const int g0 = lane >> 3, g1 = 4 + (lane >> 3);
      lo = dequant8_v41(c0, ue8m0_scale(((g0 < 4 ? sc.x : sc.y) >> (8 * (g0 & 3))) & 0xFFu));
      if (lane < 24) {
        const uint2 c1 = *reinterpret_cast<const uint2*>(row + 256 + 8 * lane);
        hi = dequant8_v41(c1, ue8m0_scale((sc.y >> (8 * (g1 & 3))) & 0xFFu));
      } else {
        hi = *reinterpret_cast<const uint4*>(row + kNopeDim + 16 * (lane - 24));
      }
    }
    __syncwarp();   // the row buffer is rewritten by the next row
    uint4* dst = reinterpret_cast<uint4*>(out + i * kDim);
    dst[lane] = lo;
    dst[32 + lane] = hi;
  }
}

// One wave: the grid is the resident CTAs (SMs x CTAs per SM at the kernel's
// register count), so no CTA starts after another has finished its rows.
template <int L>
static cudaError_t launch_fq(const __nv_bfloat16* in, long long n, long long in_stride,
                             __nv_bfloat16* out, cudaStream_t stream) {
  static std::atomic<int> per_sm_of_device[64];   // 0: not queried yet
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int per_sm = dev < 64 ? per_sm_of_device[dev].load(std::memory_order_relaxed) : 0;
  if (per_sm == 0) {
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fake_quant_kernel<L>, kFqWarps * 32, 0);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    if (dev < 64) per_sm_of_device[dev].store(per_sm, std::memory_order_relaxed);
  }
  const long long want = (n + kFqWarps - 1) / kFqWarps;
  const long long cap = (long long)device_sm_count() * per_sm;
  const int grid = (int)(want < cap ? want : cap);
  fake_quant_kernel<L><<<grid, kFqWarps * 32, 0, stream>>>(in, n, in_stride, out);
  return cudaGetLastError();
}

cudaError_t launch_fake_quant(int layout, const __nv_bfloat16* in, long long n,
                              long long in_stride, __nv_bfloat16* out, cudaStream_t stream) {
  if (layout == kV41) return launch_fq<kV41>(in, n, in_stride, out, stream);
  if (layout == kV41Fp4) return launch_fq<kV41Fp4>(in, n, in_stride, out, stream);
  return launch_fq<kV4>(in, n, in_stride, out, stream);
}

}  // namespace dsv4kv
