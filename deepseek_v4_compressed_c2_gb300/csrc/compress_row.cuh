// Per-row work of the fused compressor, shared by its launch forms (the
// streaming / wide persistent kernel in compress_store.cu and the decode /
// verify kernel in compress_decode.cu): the row states and descriptor of the
// write plan, the destination lookup, and process_row -- pair pooling
// (ratio 2), RMSNorm, RoPE, store_row and the paged write of one 512-dim row
// by one warp.
//
// sglang PR #39652 "dsv4.1: compression, KV I/O, and metadata kernels",
// Summary (c1/c2 bullet: pair-pooling, RMSNorm, RoPE and the main-KV write in
// one launch, returning the pre-RoPE latent; out_loc == 0 marks a padded
// graph row); PagedKV<layout, page_bits>::row for the destination address.
#pragma once
#include <cstdint>

#include "internal.cuh"
#include "layout.cuh"
#include "quant.cuh"

namespace dsv4kv {

// kRowOkRing: the pair's first token is in the ring and the producer copies
// the ring entry into the stage like any row.  kRowRing: the same, but the
// request's step is long enough (n >= 2R) for its ring update to reuse that
// entry, so the per-request ring phase computes the row (read before write,
// in one warp) and the tiles skip it.
enum RowState : int { kRowNone = 0, kRowPad = 1, kRowBad = 2, kRowOk = 3, kRowRing = 4,
                      kRowOkRing = 5 };

struct __align__(16) RowDesc {
  int state;
  int pos;   // RATIO * c, the position of the row's first token
  int r;     // request slot
  int c;     // compressed index inside the request (the page-table index)
};


// Compressed rows a request slot produces: RATIO 1: its n new tokens;
// RATIO 2: the pairs whose second token is new, (p0 + n) / 2 - p0 / 2.
template <int RATIO>
__device__ __forceinline__ long long rows_of_slot(int n, int p0) {
  if (n <= 0) return 0;
  if (RATIO == 1) return n;
  return (((long long)p0 + n) >> 1) - ((long long)p0 >> 1);
}


// Destination slot of a planned row: out_loc[k], or the page table at the
// compressed index c (-1 when the page index is past the table).
__device__ __forceinline__ long long dest_slot(const StoreParams& p, long long k, const RowDesc& d) {
  if (p.out_loc) return p.out_loc[k];
  const int lp = d.c >> p.page_bits;     // page_bits <= 16
  if (d.c < 0 || lp >= p.max_pages) return -1;
  return ((long long)p.page_table[(long long)d.r * p.max_pages + lp] << p.page_bits)
         | (long long)(d.c & ((1 << p.page_bits) - 1));
}

__device__ __forceinline__ void zero_row_outputs(const StoreParams& p, long long k, int lane) {
  if (p.latent_out) {
    uint4* d = reinterpret_cast<uint4*>(p.latent_out + k * kDim);
    d[lane] = make_uint4(0, 0, 0, 0);
    d[32 + lane] = make_uint4(0, 0, 0, 0);
  }
  if (p.prequant_out) {
    float4* d = reinterpret_cast<float4*>(p.prequant_out + k * kDim);
    d[2 * lane] = make_float4(0.f, 0.f, 0.f, 0.f);
    d[2 * lane + 1] = make_float4(0.f, 0.f, 0.f, 0.f);
    d[64 + 2 * lane] = make_float4(0.f, 0.f, 0.f, 0.f);
    d[64 + 2 * lane + 1] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

// fast exp2 / reciprocal: relative error ~2^-22, far inside the 1e-5
// tolerance on the pre-quant row; exact at 0 and at powers of two
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

// One row's inputs, pulled out of the stage into registers.
template <int RATIO, bool ROPE>
struct RowIn {
  uint4 kv0[2], kv1[2], s0[2], s1[2];
  float4 fr[2];
};

// Stage layout: the rows' inputs back to back (kInBytes each), then their
// RoPE rows (kRopeBytes each), so consecutive source rows can arrive in one
// copy.
template <int RATIO, bool ROPE>
__device__ __forceinline__ void load_row(const uint8_t* in_row, const uint8_t* rope_row, int lane,
                                         RowIn<RATIO, ROPE>& in) {
  const uint4* b = reinterpret_cast<const uint4*>(in_row);   // 64 uint4 per 1 KB block
  in.kv0[0] = b[lane];
  in.kv0[1] = b[32 + lane];
  if constexpr (RATIO == 2) {
    in.s0[0] = b[64 + lane];
    in.s0[1] = b[96 + lane];
    in.kv1[0] = b[128 + lane];
    in.kv1[1] = b[160 + lane];
    in.s1[0] = b[192 + lane];
    in.s1[1] = b[224 + lane];
  }
  if constexpr (ROPE) {
    if (lane >= 24) {
      const float4* f = reinterpret_cast<const float4*>(rope_row);
      in.fr[0] = f[2 * (lane - 24)];
      in.fr[1] = f[2 * (lane - 24) + 1];
    }
  }
}

// A row between its arithmetic and its store: the lane's 16 values of x * w
// (pooled, RMSNorm weight applied, RoPE'd) as 8 fp32 pairs and the norm's
// deferred 1 / rms.  row_math needs only the row's inputs (and, for the
// post-norm pre-RoPE latent it writes on the way, the output row latent_k;
// latent_k < 0 writes none);
// row_store also needs the output row k and the destination slot, so a
// launch without the latent output can do the arithmetic before it knows
// them.
struct RowMath {
  uint64_t x2[8];
  float inv;
};

// The RMSNorm weights of a lane's pair q (dims 2q, 2q + 1 of its 16): from
// 16 floats, or from the packed bf16 row (two uint4), with the same bits.
__device__ __forceinline__ uint64_t norm_w_pair(const float (&w)[16], int q) {
  return f2(w[2 * q], w[2 * q + 1]);
}
__device__ __forceinline__ uint64_t norm_w_pair(const uint4 (&w)[2], int q) {
  const uint32_t v = word_of(w[q >> 2], q & 3);
  return f2(bf16_lo(v), bf16_hi(v));
}

template <int RATIO, bool NORM, bool ROPE, typename NormW>
__device__ __forceinline__ void row_math(const StoreParams& p, const RowIn<RATIO, ROPE>& in,
                                         const NormW& w, int lane, RowMath& m,
                                         long long latent_k) {
  // the lane's 16 values as 8 fp32 pairs: pairs 0..3 = dims 8l.., 4..7 =
  // dims 256+8l..; every pair comes from one bf16 word
  uint64_t (&x2)[8] = m.x2;
#pragma unroll
  for (int q = 0; q < 8; ++q) x2[q] = f2_from_bf16x2(word_of(in.kv0[q >> 2], q & 3));
  if constexpr (RATIO == 2) {
    // softmax over the pair, anchored on the member with the larger score:
    // with t = (s1 - s0) log2(e), the other member's weight is
    // w = 1 / (1 + 2^|t|) <= 1/2 and x = anchor + (other - anchor) * w.
    // The approximate exp / reciprocal then only perturb the small
    // correction term, so a saturated pair (w below the anchor's half ulp)
    // pools to the anchor exactly, as in exact arithmetic (an ex2 overflow
    // gives w = 0).  The sign of t picks the anchor (negative: k0) and the
    // sign of the weight together: x = anchor + (k0 - k1) * (+-w).
    const uint64_t log2e = f2(1.4426950408889634f, 1.4426950408889634f), one = f2(1.f, 1.f);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const uint64_t k1 = f2_from_bf16x2(word_of(in.kv1[q >> 2], q & 3));
      const uint64_t a = f2_from_bf16x2(word_of(in.s0[q >> 2], q & 3));
      const uint64_t b = f2_from_bf16x2(word_of(in.s1[q >> 2], q & 3));
      float t0, t1, d0, d1, ka0, ka1, kb0, kb1;
      f2_split(f2_mul(f2_sub(b, a), log2e), t0, t1);
      f2_split(f2_add(f2(ex2_approx(fabsf(t0)), ex2_approx(fabsf(t1))), one), d0, d1);
      f2_split(x2[q], ka0, ka1);
      f2_split(k1, kb0, kb1);
      const uint32_t u0 = __float_as_uint(t0), u1 = __float_as_uint(t1);
      const uint32_t m0 = (uint32_t)((int32_t)u0 >> 31), m1 = (uint32_t)((int32_t)u1 >> 31);
      const uint64_t anchor =
          f2(__uint_as_float((__float_as_uint(ka0) & m0) | (__float_as_uint(kb0) & ~m0)),
             __uint_as_float((__float_as_uint(ka1) & m1) | (__float_as_uint(kb1) & ~m1)));
      const uint64_t wt = f2(__uint_as_float(__float_as_uint(rcp_approx(d0)) ^ (u0 & 0x80000000u)),
                             __uint_as_float(__float_as_uint(rcp_approx(d1)) ^ (u1 & 0x80000000u)));
      x2[q] = f2_fma(f2_sub(x2[q], k1), wt, anchor);
    }
  }
  // RMSNorm: x_n = (x * w) * inv with inv = rsqrt(mean(x^2) + eps).  The
  // product by inv is deferred: RoPE rotates x * w, and the V41 quantizer
  // folds inv into its power-of-two multiplier, which rounds exactly like
  // quantizing the explicit x_n (see store_row_v41_scaled).
  m.inv = 1.f;
  if constexpr (NORM) {
    uint64_t acc[2] = {0ull, 0ull};     // partial sums of dims = 0,1 and 2,3 (mod 4)
#pragma unroll
    for (int q = 0; q < 8; ++q) acc[q & 1] = f2_fma(x2[q], x2[q], acc[q & 1]);
    float s0, s1, s2, s3;
    f2_split(acc[0], s0, s1);
    f2_split(acc[1], s2, s3);
    float t = (s0 + s1) + (s2 + s3);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(kFullMask, t, o);
    m.inv = rsqrtf(fmaf(t, 1.f / kDim, p.eps));
#pragma unroll
    for (int q = 0; q < 8; ++q) x2[q] = f2_mul(x2[q], norm_w_pair(w, q));
  }
  if (p.latent_out && latent_k >= 0) {  // post-norm, pre-RoPE
    const uint64_t inv2 = f2(m.inv, m.inv);
    float xn[16];
#pragma unroll
    for (int q = 0; q < 8; ++q) f2_split(f2_mul(x2[q], inv2), xn[2 * q], xn[2 * q + 1]);
    uint4* o = reinterpret_cast<uint4*>(p.latent_out + latent_k * kDim);
    o[lane] = pack_bf16x8(xn);
    o[32 + lane] = pack_bf16x8(xn + 8);
  }
  if constexpr (ROPE) {
    // lanes 24..31 hold dims 448+8(l-24) .. +7 in pairs 4..7: 4 complex
    // pairs (a, b) rotated by (c, s): (a c - b s, a s + b c)
    if (lane >= 24) {
      const float f[8] = {in.fr[0].x, in.fr[0].y, in.fr[0].z, in.fr[0].w,
                          in.fr[1].x, in.fr[1].y, in.fr[1].z, in.fr[1].w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float c = f[2 * q], sn = f[2 * q + 1];
        float a, b;
        f2_split(x2[4 + q], a, b);
        x2[4 + q] = f2(fmaf(a, c, b * -sn), fmaf(a, sn, b * c));   // (a c - b s, a s + b c)
      }
    }
  }
}

// The pre-quant output and the quantized row k at `slot` of a computed row.
template <int L, bool NORM>
__device__ __forceinline__ void row_store(const StoreParams& p, long long k, long long slot,
                                          RowMath& m, int lane) {
  uint64_t (&x2)[8] = m.x2;
  const uint64_t inv2 = f2(m.inv, m.inv);
  float x[16];
  const bool store = slot > 0 && slot < p.pool_rows;
  if (slot != 0 && !store && lane == 0 && p.err) atomicAdd(p.err, 1);   // destination fault
  if (p.prequant_out || L != kV41 || !NORM) {
    // explicit pre-quant row (debug output, FP4, V4, or no norm: inv == 1)
    if constexpr (NORM) {
#pragma unroll
      for (int q = 0; q < 8; ++q) x2[q] = f2_mul(x2[q], inv2);
    }
    f2_unpack16(x2, x);
    if (p.prequant_out) {
      float4* o = reinterpret_cast<float4*>(p.prequant_out + k * kDim);
      o[2 * lane] = make_float4(x[0], x[1], x[2], x[3]);
      o[2 * lane + 1] = make_float4(x[4], x[5], x[6], x[7]);
      o[64 + 2 * lane] = make_float4(x[8], x[9], x[10], x[11]);
      o[64 + 2 * lane + 1] = make_float4(x[12], x[13], x[14], x[15]);
    }
    if (store) store_row_split<L>(x, PagedKV<L>{p.pool, p.page_bits}.row(slot), lane);
  } else if (store) {
    store_row_v41_scaled(x2, m.inv, PagedKV<kV41>{p.pool, p.page_bits}.row(slot), lane);
  }
}

// A row that is not computed: nothing for a row another phase computes, else
// zero debug outputs, and a fault for a bad row.  True when it is computed.
__device__ __forceinline__ bool row_computed(const StoreParams& p, long long k, int state,
                                             int lane) {
  if (state == kRowOk || state == kRowOkRing) return true;
  if (state == kRowNone || state == kRowRing) return false;
  if (state == kRowBad && lane == 0 && p.err) atomicAdd(p.err, 1);
  zero_row_outputs(p, k, lane);
  return false;
}

template <int L, int RATIO, bool NORM, bool ROPE>
__device__ __forceinline__ void process_row(const StoreParams& p, long long k, int state,
                                            long long slot, const RowIn<RATIO, ROPE>& in,
                                            const float (&w)[16], int lane) {
  if (!row_computed(p, k, state, lane)) return;
  RowMath m;
  row_math<RATIO, NORM, ROPE>(p, in, w, lane, m, k);
  row_store<L, NORM>(p, k, slot, m, lane);
}


}  // namespace dsv4kv
